"""fp64 CPU oracle for the KDA intra-chunk backward (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline /
reference arm import this package.  The library and its CUDA kernels never do,
and this package imports nothing from the library.

``kda_ref.c`` holds the arithmetic (plain loops in fp64, see its header for the
definitions it follows).  This module compiles it with the host C compiler into
``libkda_oracle.so`` next to the source, and exposes numpy/torch-friendly wrappers
that widen the (already quantised) inputs to fp64.
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "kda_ref.c")
LIB = os.path.join(_HERE, "libkda_oracle.so")

# -ffp-contract=off: no fused multiply-add contraction, so x86 and Arm hosts give
# bit-identical fp64 results; no fast-math of any kind.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off"]

_lib = None


def build(src: str = SRC, out: str = LIB, extra_flags=()) -> str:
    """Compile an oracle source file into a shared library and return its path."""
    cmd = ["gcc", *CFLAGS, *extra_flags, "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def _bind(lib):
    dp = ctypes.POINTER(ctypes.c_double)
    i = ctypes.c_int
    lib.kda_intra_fwd_ref_f64.argtypes = [dp] * 6 + [i] * 6
    lib.kda_intra_fwd_ref_f64.restype = i
    lib.kda_intra_bwd_ref_f64.argtypes = [dp] * 10 + [i] * 6
    lib.kda_intra_bwd_ref_f64.restype = i
    lib.kda_oracle_max_threads.argtypes = []
    lib.kda_oracle_max_threads.restype = i
    return lib


def load(path: str | None = None):
    """Load (building if needed) the oracle library.  ``path`` loads another build."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        if (not os.path.exists(LIB)
                or os.path.getmtime(LIB) < os.path.getmtime(SRC)):
            build()
        _lib = _bind(ctypes.CDLL(LIB))
    return _lib


def _f64(x) -> np.ndarray:
    """Widen a torch tensor or array to a contiguous fp64 numpy array (exact)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def max_threads(lib=None) -> int:
    return (lib or load()).kda_oracle_max_threads()


def intra_fwd(q, k, g, beta, *, bt: int = 64, nthreads: int = 0, lib=None):
    """Aqk, Akk as fp64 arrays of shape [B, T, H, bt]."""
    lib = lib or load()
    q, k, g, beta = _f64(q), _f64(k), _f64(g), _f64(beta)
    B, T, H, K = q.shape
    Aqk = np.empty((B, T, H, bt))
    Akk = np.empty((B, T, H, bt))
    rc = lib.kda_intra_fwd_ref_f64(_ptr(q), _ptr(k), _ptr(g), _ptr(beta),
                                   _ptr(Aqk), _ptr(Akk), B, T, H, K, bt, nthreads)
    if rc:
        raise ValueError("oracle forward rejected its arguments")
    return Aqk, Akk


def intra_bwd(q, k, g, beta, dAqk, dAkk, *, bt: int = 64, nthreads: int = 0, lib=None):
    """dq, dk, db, dg as fp64 arrays ([B,T,H,K] x3 and [B,T,H])."""
    lib = lib or load()
    q, k, g, beta = _f64(q), _f64(k), _f64(g), _f64(beta)
    dAqk, dAkk = _f64(dAqk), _f64(dAkk)
    B, T, H, K = q.shape
    dq = np.empty((B, T, H, K))
    dk = np.empty((B, T, H, K))
    dg = np.empty((B, T, H, K))
    db = np.empty((B, T, H))
    rc = lib.kda_intra_bwd_ref_f64(_ptr(q), _ptr(k), _ptr(g), _ptr(beta),
                                   _ptr(dAqk), _ptr(dAkk), _ptr(dq), _ptr(dk),
                                   _ptr(db), _ptr(dg), B, T, H, K, bt, nthreads)
    if rc:
        raise ValueError("oracle backward rejected its arguments")
    return dq, dk, db, dg
