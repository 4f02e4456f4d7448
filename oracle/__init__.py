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


def chunk_reverse_cumsum(x, bt: int = 64) -> np.ndarray:
    """Inclusive reverse cumsum along tokens inside each chunk of bt tokens:
    out[t] = sum of x[t'] over t' >= t in t's chunk (axis 1 of a [B, T, ...] array)."""
    x = _f64(x)
    B, T = x.shape[:2]
    y = x.reshape(B, T // bt, bt, *x.shape[2:])
    y = np.flip(np.cumsum(np.flip(y, axis=2), axis=2), axis=2)
    return np.ascontiguousarray(y.reshape(x.shape))


def intra_bwd_ex(q, k, g, beta, dAqk, dAkk, *, dq_in=None, dk_in=None, dg_in=None,
                 db_in=None, fold_dg=False, bt: int = 64, nthreads: int = 0, lib=None):
    """The extended contract, composed from intra_bwd:

    * grouped value heads: q, k have H heads, the rest HV = g.shape[2]; value head hv
      uses q/k head hv // (HV // H), so the per-value-head problem is intra_bwd on q/k
      with every head repeated HV // H times;
    * incoming gradients are added to the outputs;
    * fold_dg replaces dg (incoming part included) by its chunk-local reverse cumsum.
    """
    q, k = _f64(q), _f64(k)
    HV, H = _f64(g).shape[2], q.shape[2]
    if HV % H:
        raise ValueError("HV must be a multiple of H")
    G = HV // H
    if G > 1:
        q = np.repeat(q, G, axis=2)
        k = np.repeat(k, G, axis=2)
    dq, dk, db, dg = intra_bwd(q, k, g, beta, dAqk, dAkk, bt=bt, nthreads=nthreads, lib=lib)
    if dq_in is not None:
        dq = dq + _f64(dq_in)
    if dk_in is not None:
        dk = dk + _f64(dk_in)
    if db_in is not None:
        db = db + _f64(db_in)
    if dg_in is not None:
        dg = dg + _f64(dg_in)
    if fold_dg:
        dg = chunk_reverse_cumsum(dg, bt)
    return dq, dk, db, dg


def intra_bwd_varlen(q, k, g, beta, dAqk, dAkk, cu_seqlens, *, dq_in=None, dk_in=None,
                     dg_in=None, db_in=None, fold_dg=False, bt: int = 64, nthreads: int = 0,
                     lib=None):
    """Variable-length sequences packed along T (B == 1), composed from intra_bwd_ex.

    Reading (the bwd_intra page's host wrapper takes cu_seqlens / chunk_indices and
    sends them to its fallback): chunks restart at every sequence start, so a
    sequence's last chunk may be short, and every per-chunk definition holds over the
    chunk's valid rows only.  Each sequence is padded to whole chunks with rows that
    take no part in any sum (q = k = 0, beta = 0, zero dA rows, zero incoming
    gradients; the gate held at the last valid row's value), solved as one
    fixed-length problem and cut back to its own rows.  Rows of tokens outside every
    sequence come back as NaN.
    """
    cu = [int(v) for v in np.asarray(cu_seqlens).reshape(-1)]
    arrs = {n: _f64(v) for n, v in (("q", q), ("k", k), ("g", g), ("beta", beta),
                                     ("dAqk", dAqk), ("dAkk", dAkk))}
    ins = {n: (None if v is None else _f64(v)) for n, v in (("dq_in", dq_in), ("dk_in", dk_in),
                                                            ("dg_in", dg_in), ("db_in", db_in))}
    if arrs["q"].shape[0] != 1:
        raise ValueError("variable-length inputs have B == 1")
    T, HV = arrs["g"].shape[1], arrs["g"].shape[2]
    K = arrs["q"].shape[3]
    dq = np.full((1, T, HV, K), np.nan)
    dk = np.full((1, T, HV, K), np.nan)
    dg = np.full((1, T, HV, K), np.nan)
    db = np.full((1, T, HV), np.nan)
    for a, b in zip(cu[:-1], cu[1:]):
        L = b - a
        if L <= 0:
            continue
        Lp = -(-L // bt) * bt

        def pad(x, edge=False):
            if x is None:
                return None
            y = x[:, a:b]
            fill = np.repeat(y[:, -1:], Lp - L, axis=1) if edge else \
                np.zeros((1, Lp - L) + y.shape[2:])
            return np.concatenate([y, fill], axis=1)

        part = intra_bwd_ex(pad(arrs["q"]), pad(arrs["k"]), pad(arrs["g"], edge=True),
                            pad(arrs["beta"]), pad(arrs["dAqk"]), pad(arrs["dAkk"]),
                            dq_in=pad(ins["dq_in"]), dk_in=pad(ins["dk_in"]),
                            dg_in=pad(ins["dg_in"]), db_in=pad(ins["db_in"]),
                            fold_dg=fold_dg, bt=bt, nthreads=nthreads, lib=lib)
        for out, x in zip((dq, dk, db, dg), part):
            out[:, a:b] = x[:, :L]
    return dq, dk, db, dg


def intra_fwd_ex(q, k, g, beta, *, cu_seqlens=None, bt: int = 64, nthreads: int = 0, lib=None):
    """The forward with grouped value heads and variable-length sequences, composed
    from intra_fwd the same way intra_bwd_ex / intra_bwd_varlen compose the backward
    (q/k heads repeated; each sequence padded to whole chunks, solved, cut back; rows of
    tokens outside every sequence come back as NaN)."""
    q, k, g, beta = _f64(q), _f64(k), _f64(g), _f64(beta)
    HV, H = g.shape[2], q.shape[2]
    if HV % H:
        raise ValueError("HV must be a multiple of H")
    if HV > H:
        q = np.repeat(q, HV // H, axis=2)
        k = np.repeat(k, HV // H, axis=2)
    if cu_seqlens is None:
        return intra_fwd(q, k, g, beta, bt=bt, nthreads=nthreads, lib=lib)
    cu = [int(v) for v in np.asarray(cu_seqlens).reshape(-1)]
    T = g.shape[1]
    Aqk = np.full((1, T, HV, bt), np.nan)
    Akk = np.full((1, T, HV, bt), np.nan)
    for a, b in zip(cu[:-1], cu[1:]):
        L = b - a
        if L <= 0:
            continue
        Lp = -(-L // bt) * bt

        def pad(x, edge=False):
            y = x[:, a:b]
            fill = np.repeat(y[:, -1:], Lp - L, axis=1) if edge else \
                np.zeros((1, Lp - L) + y.shape[2:])
            return np.concatenate([y, fill], axis=1)

        fa, fk = intra_fwd(pad(q), pad(k), pad(g, edge=True), pad(beta), bt=bt,
                           nthreads=nthreads, lib=lib)
        Aqk[:, a:b] = fa[:, :L]
        Akk[:, a:b] = fk[:, :L]
    return Aqk, Akk
