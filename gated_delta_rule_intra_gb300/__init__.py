"""Python binding of libkda, the sm_103a KDA intra-chunk backward.

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libkda.so`` (built in-tree by ``build.build_library()``).  There is
no CPU or framework fallback; if the library is missing every call raises.

The functions carry the C names of ``include/kda.h``:

* ``kda_intra_bwd``       -- fast path (TF32 tensor-core cross terms)
* ``kda_intra_bwd_fp32``  -- all-FP32 path
* ``kda_intra_bwd_ex``    -- fast path with options: grouped value heads, incoming
  gradients added in-kernel, dg folded to its chunk-local reverse cumsum, dq/dk in
  the q/k dtype, variable-length sequences (``cu_seqlens``), the diagonal quadrant
  factorized (``factor_diag``), the cross sums in split TF32 for FP32-level accuracy
  (``split_tf32``)
* ``prepare_chunk_indices`` -- the (sequence, chunk) table of a ``cu_seqlens``
* ``kda_intra_bwd_host``  -- host buffers in and out, copies on the stream
* ``kda_intra_bwd_host_static`` -- the same without a workspace, staged in the library's
  fixed device array (``HOST_STATIC_MAX_BYTES``) for callers that cannot allocate
* ``kda_intra_fwd``       -- the forward score matrices Aqk, Akk (grouped value heads
  and variable-length sequences through ``kda_intra_fwd_ex``)
* ``kda_status_str``, ``kda_abi_version``
* ``use_library``, ``kda_debug_checks``, ``kda_debug_set_flags`` -- run the same calls
  through the bounds-checked debug build ``libkda_debug.so`` (tests)
"""

from __future__ import annotations

import contextlib
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkda.so")
DEBUG_LIB_PATH = os.path.join(_HERE, "libkda_debug.so")

# KDA_ABI_VERSION of the include/kda.h these ctypes mirrors follow (option structs,
# signatures); a library of any other version is refused at load.
ABI_VERSION = 9
KDA_OK = 0
KDA_BF16 = 0
KDA_FP16 = 1
BT = 64
K = 128
KDA_ERR_TOO_LARGE = 10
HOST_STATIC_MAX_BYTES = 32 << 20  # KDA_HOST_STATIC_MAX_BYTES of include/kda.h

_DTYPES = {torch.bfloat16: KDA_BF16, torch.float16: KDA_FP16}
_lib = None


class KdaOpts(ctypes.Structure):
    """Mirror of kda_intra_bwd_opts_t."""
    _fields_ = [("HV", ctypes.c_int), ("dq_in", ctypes.c_void_p), ("dk_in", ctypes.c_void_p),
                ("dg_in", ctypes.c_void_p), ("db_in", ctypes.c_void_p),
                ("fold_dg", ctypes.c_int), ("dqdk_io_dtype", ctypes.c_int),
                ("cu_seqlens", ctypes.c_void_p), ("chunk_indices", ctypes.c_void_p),
                ("num_seqs", ctypes.c_int), ("num_chunks", ctypes.c_int),
                ("factor_diag", ctypes.c_int), ("split_tf32", ctypes.c_int)]


class KdaFwdOpts(ctypes.Structure):
    """Mirror of kda_intra_fwd_opts_t."""
    _fields_ = [("HV", ctypes.c_int), ("cu_seqlens", ctypes.c_void_p),
                ("chunk_indices", ctypes.c_void_p), ("num_seqs", ctypes.c_int),
                ("num_chunks", ctypes.c_int)]


class KdaError(RuntimeError):
    def __init__(self, code: int, fn: str):
        self.code = code
        super().__init__(f"{fn} failed: {kda_status_str(code)} (status {code})")


def load_library(path: str | None = None):
    """Load libkda.so (raises if it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(
            f"{p} is missing: build it with gated_delta_rule_intra_gb300.build."
            "build_library() (or __graft_entry__.build()); there is no fallback")
    lib = ctypes.CDLL(p)
    vp, fp, i, st = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int
    sig = [vp, vp, fp, fp, fp, fp, fp, fp, fp, fp, i, i, i, i, vp]
    for name in ("kda_intra_bwd", "kda_intra_bwd_fp32"):
        f = getattr(lib, name)
        f.argtypes = sig
        f.restype = st
    lib.kda_intra_bwd_ex.argtypes = sig[:-1] + [ctypes.POINTER(KdaOpts), vp]
    lib.kda_intra_bwd_ex.restype = st
    lib.kda_intra_bwd_host.argtypes = sig[:-1] + [vp, ctypes.c_size_t, vp]
    lib.kda_intra_bwd_host.restype = st
    lib.kda_intra_bwd_host_static.argtypes = sig
    lib.kda_intra_bwd_host_static.restype = st
    lib.kda_intra_fwd.argtypes = [vp, vp, fp, fp, fp, fp, i, i, i, i, vp]
    lib.kda_intra_fwd.restype = st
    lib.kda_intra_fwd_ex.argtypes = [vp, vp, fp, fp, fp, fp, i, i, i, i,
                                     ctypes.POINTER(KdaFwdOpts), vp]
    lib.kda_intra_fwd_ex.restype = st
    lib.kda_intra_bwd_host_workspace_bytes.argtypes = [i, i, i, i]
    lib.kda_intra_bwd_host_workspace_bytes.restype = ctypes.c_size_t
    lib.kda_status_str.argtypes = [i]
    lib.kda_status_str.restype = ctypes.c_char_p
    lib.kda_abi_version.argtypes = []
    lib.kda_abi_version.restype = i
    lib.kda_debug_checks.argtypes = []
    lib.kda_debug_checks.restype = i
    lib.kda_debug_set_flags.argtypes = [vp]
    lib.kda_debug_set_flags.restype = st
    if lib.kda_abi_version() != ABI_VERSION:
        raise RuntimeError(
            f"{p} has ABI version {lib.kda_abi_version()}, this binding needs {ABI_VERSION}: "
            "rebuild it with gated_delta_rule_intra_gb300.build.build_library()")
    if path is None:
        _lib = lib
    return lib


@contextlib.contextmanager
def use_library(path: str):
    """Route every call of this module through another build of libkda (for instance
    the bounds-checked ``libkda_debug.so``) inside the ``with`` block."""
    global _lib
    saved = _lib
    _lib = load_library(path)
    try:
        yield _lib
    finally:
        _lib = saved


def kda_debug_checks() -> bool:
    """True when the library in use is the bounds-checked debug build."""
    return bool(load_library().kda_debug_checks())


def kda_debug_set_flags(word) -> None:
    """Debug build only: later launches report index or wait failures into ``word``
    (a CUDA int32 tensor of one element, caller-owned; None stops reporting)."""
    if word is not None and (word.device.type != "cuda" or word.numel() != 1
                             or word.dtype != torch.int32):
        raise ValueError("the flag word must be a one-element int32 CUDA tensor")
    rc = load_library().kda_debug_set_flags(
        ctypes.c_void_p(None if word is None else word.data_ptr()))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_debug_set_flags")


def kda_status_str(code: int) -> str:
    return load_library().kda_status_str(int(code)).decode()


def kda_abi_version() -> int:
    return load_library().kda_abi_version()


def _shape(q):
    if q.dim() != 4 or q.shape[-1] != K:
        raise ValueError(f"q must be [B, T, H, {K}], got {tuple(q.shape)}")
    return q.shape[0], q.shape[1], q.shape[2]


def _check(name, t, shape, dtype, device):
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.dtype != dtype:
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _outputs(q, dq, dk, db, dg):
    B, T, H = _shape(q)
    f32 = torch.float32
    dq = torch.empty(B, T, H, K, device=q.device, dtype=f32) if dq is None else dq
    dk = torch.empty(B, T, H, K, device=q.device, dtype=f32) if dk is None else dk
    dg = torch.empty(B, T, H, K, device=q.device, dtype=f32) if dg is None else dg
    db = torch.empty(B, T, H, device=q.device, dtype=f32) if db is None else db
    return dq, dk, db, dg


def _validate(q, k, g, beta, dAqk, dAkk, dq, dk, db, dg, device):
    B, T, H = _shape(q)
    if q.dtype not in _DTYPES:
        raise ValueError(f"q/k dtype must be bf16 or fp16, got {q.dtype}")
    f32 = torch.float32
    _check("q", q, (B, T, H, K), q.dtype, device)
    _check("k", k, (B, T, H, K), q.dtype, device)
    _check("g", g, (B, T, H, K), f32, device)
    _check("beta", beta, (B, T, H), f32, device)
    _check("dAqk", dAqk, (B, T, H, BT), f32, device)
    _check("dAkk", dAkk, (B, T, H, BT), f32, device)
    for n, t in (("dq", dq), ("dk", dk), ("dg", dg)):
        _check(n, t, (B, T, H, K), f32, device)
    _check("db", db, (B, T, H), f32, device)
    return B, T, H


def _stream_handle(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else stream)


def _device_call(fn_name, q, k, g, beta, dAqk, dAkk, dq, dk, db, dg, stream):
    if q.device.type != "cuda":
        raise ValueError(f"{fn_name} needs CUDA tensors (no CPU path exists)")
    dq, dk, db, dg = _outputs(q, dq, dk, db, dg)
    B, T, H = _validate(q, k, g, beta, dAqk, dAkk, dq, dk, db, dg, q.device)
    lib = load_library()
    ptr = ctypes.c_void_p
    with torch.cuda.device(q.device):
        rc = getattr(lib, fn_name)(
            ptr(q.data_ptr()), ptr(k.data_ptr()), ptr(g.data_ptr()), ptr(beta.data_ptr()),
            ptr(dAqk.data_ptr()), ptr(dAkk.data_ptr()), ptr(dq.data_ptr()),
            ptr(dk.data_ptr()), ptr(db.data_ptr()), ptr(dg.data_ptr()),
            B, T, H, _DTYPES[q.dtype], _stream_handle(stream, q.device))
    if rc != KDA_OK:
        raise KdaError(rc, fn_name)
    return dq, dk, db, dg


def kda_intra_bwd(q, k, g, beta, dAqk, dAkk, dq=None, dk=None, db=None, dg=None,
                  stream=None):
    """Intra-chunk backward (fast path).  Returns (dq, dk, db, dg), all fp32.

    Tensors: q, k [B,T,H,128] bf16/fp16; g [B,T,H,128] fp32 chunk-local cumulative
    log2 gate; beta [B,T,H] fp32; dAqk, dAkk [B,T,H,64] fp32.  Outputs may be passed
    in (contiguous fp32) or are allocated.  Runs on ``stream`` (default: current).
    """
    return _device_call("kda_intra_bwd", q, k, g, beta, dAqk, dAkk, dq, dk, db, dg, stream)


def kda_intra_bwd_fp32(q, k, g, beta, dAqk, dAkk, dq=None, dk=None, db=None, dg=None,
                       stream=None):
    """Same contract as ``kda_intra_bwd``; every product and sum in FP32."""
    return _device_call("kda_intra_bwd_fp32", q, k, g, beta, dAqk, dAkk, dq, dk, db, dg,
                        stream)


def prepare_chunk_indices(cu_seqlens, bt: int = BT):
    """The chunk table of packed variable-length sequences: an int32 [num_chunks, 2]
    tensor on cu_seqlens' device whose row c is (n, j) = chunk j of sequence n, in
    sequence order (sequence n covers tokens [cu_seqlens[n], cu_seqlens[n+1]) and has
    ceil(len / bt) chunks; empty sequences have none).  Reads cu_seqlens on the host."""
    cu = torch.as_tensor(cu_seqlens).to("cpu", torch.int64)
    if cu.dim() != 1 or cu.numel() < 2:
        raise ValueError("cu_seqlens must be 1-d with at least two entries")
    lens = cu[1:] - cu[:-1]
    if cu[0].item() != 0 or bool((lens < 0).any()):
        raise ValueError("cu_seqlens must start at 0 and be non-decreasing")
    nch = (lens + bt - 1) // bt
    seq = torch.repeat_interleave(torch.arange(len(nch)), nch)
    first = torch.cumsum(nch, 0) - nch
    idx = torch.arange(int(nch.sum())) - torch.repeat_interleave(first, nch)
    out = torch.stack([seq, idx], dim=1).to(torch.int32)
    dev = cu_seqlens.device if isinstance(cu_seqlens, torch.Tensor) else "cpu"
    return out.to(dev).contiguous()


def kda_intra_bwd_ex(q, k, g, beta, dAqk, dAkk, dq=None, dk=None, db=None, dg=None, *,
                     dq_in=None, dk_in=None, dg_in=None, db_in=None, fold_dg=False,
                     dqdk_io_dtype=False, cu_seqlens=None, chunk_indices=None,
                     factor_diag=False, split_tf32=False, stream=None):
    """Intra-chunk backward with the extended options of ``kda_intra_bwd_ex``.

    q, k have H heads; g, beta, dAqk, dAkk, the outputs and the optional incoming
    gradients have HV = g.shape[2] heads (value head hv reads q/k head hv // (HV // H)).
    ``dq_in``.. ``db_in`` are added in-kernel (they may be the output tensors
    themselves); ``fold_dg`` returns dg as its inclusive reverse cumsum inside each
    64-token chunk; ``dqdk_io_dtype`` writes dq and dk in q's dtype.
    ``cu_seqlens`` (int32 [N + 1] on the device, B must be 1) packs N sequences of any
    length along T; ``chunk_indices`` (int32 [num_chunks, 2] on the device) defaults to
    ``prepare_chunk_indices(cu_seqlens)``, which reads cu_seqlens on the host.
    ``factor_diag`` factorizes the lower-left 8x8 quadrant of each diagonal 16x16 block
    through the block's row 8 (every exponent stays <= 0) instead of one exp2 per
    (r, s, d); faster, equal up to rounding.  ``split_tf32`` takes the cross-sub-block
    sums in split TF32 (three tensor-core products per term) for FP32-level accuracy
    (1e-4), with no other option but grouped value heads.
    Returns (dq, dk, db, dg).
    """
    if q.device.type != "cuda":
        raise ValueError("kda_intra_bwd_ex needs CUDA tensors (no CPU path exists)")
    B, T, H = _shape(q)
    if q.dtype not in _DTYPES:
        raise ValueError(f"q/k dtype must be bf16 or fp16, got {q.dtype}")
    if g.dim() != 4:
        raise ValueError("g must be [B, T, HV, 128]")
    HV = g.shape[2]
    dev, f32 = q.device, torch.float32
    odt = q.dtype if dqdk_io_dtype else f32
    dq = torch.empty(B, T, HV, K, device=dev, dtype=odt) if dq is None else dq
    dk = torch.empty(B, T, HV, K, device=dev, dtype=odt) if dk is None else dk
    dg = torch.empty(B, T, HV, K, device=dev, dtype=f32) if dg is None else dg
    db = torch.empty(B, T, HV, device=dev, dtype=f32) if db is None else db
    _check("q", q, (B, T, H, K), q.dtype, dev)
    _check("k", k, (B, T, H, K), q.dtype, dev)
    _check("g", g, (B, T, HV, K), f32, dev)
    _check("beta", beta, (B, T, HV), f32, dev)
    _check("dAqk", dAqk, (B, T, HV, BT), f32, dev)
    _check("dAkk", dAkk, (B, T, HV, BT), f32, dev)
    _check("dq", dq, (B, T, HV, K), odt, dev)
    _check("dk", dk, (B, T, HV, K), odt, dev)
    _check("dg", dg, (B, T, HV, K), f32, dev)
    _check("db", db, (B, T, HV), f32, dev)
    opts = KdaOpts()
    opts.HV = HV
    for name, t, shape in (("dq_in", dq_in, (B, T, HV, K)), ("dk_in", dk_in, (B, T, HV, K)),
                           ("dg_in", dg_in, (B, T, HV, K)), ("db_in", db_in, (B, T, HV))):
        if t is not None:
            _check(name, t, shape, f32, dev)
            setattr(opts, name, t.data_ptr())
    opts.fold_dg = int(bool(fold_dg))
    opts.dqdk_io_dtype = int(bool(dqdk_io_dtype))
    opts.factor_diag = int(bool(factor_diag))
    opts.split_tf32 = int(bool(split_tf32))
    _varlen_opts(opts, cu_seqlens, chunk_indices, dev)
    lib = load_library()
    ptr = ctypes.c_void_p
    with torch.cuda.device(dev):
        rc = lib.kda_intra_bwd_ex(
            ptr(q.data_ptr()), ptr(k.data_ptr()), ptr(g.data_ptr()), ptr(beta.data_ptr()),
            ptr(dAqk.data_ptr()), ptr(dAkk.data_ptr()), ptr(dq.data_ptr()),
            ptr(dk.data_ptr()), ptr(db.data_ptr()), ptr(dg.data_ptr()),
            B, T, H, _DTYPES[q.dtype], ctypes.byref(opts), _stream_handle(stream, dev))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_intra_bwd_ex")
    return dq, dk, db, dg


def _varlen_opts(opts, cu_seqlens, chunk_indices, dev):
    if cu_seqlens is not None:
        if chunk_indices is None:
            chunk_indices = prepare_chunk_indices(cu_seqlens)
        _check("cu_seqlens", cu_seqlens, (cu_seqlens.numel(),), torch.int32, dev)
        _check("chunk_indices", chunk_indices, (chunk_indices.shape[0], 2), torch.int32, dev)
        opts.cu_seqlens = cu_seqlens.data_ptr()
        opts.chunk_indices = chunk_indices.data_ptr() if chunk_indices.numel() else 0
        opts.num_seqs = cu_seqlens.numel() - 1
        opts.num_chunks = chunk_indices.shape[0]
    elif chunk_indices is not None:
        raise ValueError("chunk_indices needs cu_seqlens")


def kda_intra_fwd(q, k, g, beta, Aqk=None, Akk=None, *, cu_seqlens=None, chunk_indices=None,
                  stream=None):
    """Aqk, Akk ([B, T, HV, 64] fp32, zeros outside the support) of the intra-chunk
    forward on the CUDA tensors q, k ([B, T, H, 128] bf16/fp16), g ([B, T, HV, 128]
    fp32) and beta ([B, T, HV] fp32); HV = g.shape[2] is a multiple of H (value head
    hv reads q/k head hv // (HV // H)).  ``cu_seqlens`` / ``chunk_indices`` as for
    ``kda_intra_bwd_ex``."""
    if q.device.type != "cuda":
        raise ValueError("kda_intra_fwd needs CUDA tensors (no CPU path exists)")
    B, T, H = _shape(q)
    if q.dtype not in _DTYPES:
        raise ValueError(f"q/k dtype must be bf16 or fp16, got {q.dtype}")
    if g.dim() != 4:
        raise ValueError("g must be [B, T, HV, 128]")
    HV = g.shape[2]
    dev, f32 = q.device, torch.float32
    Aqk = torch.empty(B, T, HV, BT, device=dev, dtype=f32) if Aqk is None else Aqk
    Akk = torch.empty(B, T, HV, BT, device=dev, dtype=f32) if Akk is None else Akk
    _check("q", q, (B, T, H, K), q.dtype, dev)
    _check("k", k, (B, T, H, K), q.dtype, dev)
    _check("g", g, (B, T, HV, K), f32, dev)
    _check("beta", beta, (B, T, HV), f32, dev)
    _check("Aqk", Aqk, (B, T, HV, BT), f32, dev)
    _check("Akk", Akk, (B, T, HV, BT), f32, dev)
    opts = KdaFwdOpts()
    opts.HV = HV
    _varlen_opts(opts, cu_seqlens, chunk_indices, dev)
    lib = load_library()
    ptr = ctypes.c_void_p
    with torch.cuda.device(dev):
        rc = lib.kda_intra_fwd_ex(ptr(q.data_ptr()), ptr(k.data_ptr()), ptr(g.data_ptr()),
                                  ptr(beta.data_ptr()), ptr(Aqk.data_ptr()),
                                  ptr(Akk.data_ptr()), B, T, H, _DTYPES[q.dtype],
                                  ctypes.byref(opts), _stream_handle(stream, dev))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_intra_fwd_ex")
    return Aqk, Akk


def kda_intra_bwd_host_workspace_bytes(B: int, T: int, H: int, qk_dtype=torch.bfloat16):
    return load_library().kda_intra_bwd_host_workspace_bytes(B, T, H, _DTYPES[qk_dtype])


def kda_intra_bwd_host(q, k, g, beta, dAqk, dAkk, dq, dk, db, dg, workspace, stream=None):
    """Host tensors in and out (pin them for asynchronous copies).

    ``workspace`` is a CUDA uint8 tensor of at least
    ``kda_intra_bwd_host_workspace_bytes(B, T, H, q.dtype)`` bytes.  The call queues
    the copies and the kernel on ``stream`` and returns; synchronise the stream
    before reading dq/dk/db/dg.
    """
    for n, t in (("q", q), ("k", k), ("g", g), ("beta", beta), ("dAqk", dAqk),
                 ("dAkk", dAkk), ("dq", dq), ("dk", dk), ("db", db), ("dg", dg)):
        if t.device.type != "cpu":
            raise ValueError(f"{n} must be a host tensor")
    B, T, H = _validate(q, k, g, beta, dAqk, dAkk, dq, dk, db, dg, torch.device("cpu"))
    if workspace.device.type != "cuda":
        raise ValueError("workspace must be device memory")
    lib = load_library()
    ptr = ctypes.c_void_p
    nbytes = workspace.numel() * workspace.element_size()
    with torch.cuda.device(workspace.device):
        rc = lib.kda_intra_bwd_host(
            ptr(q.data_ptr()), ptr(k.data_ptr()), ptr(g.data_ptr()), ptr(beta.data_ptr()),
            ptr(dAqk.data_ptr()), ptr(dAkk.data_ptr()), ptr(dq.data_ptr()),
            ptr(dk.data_ptr()), ptr(db.data_ptr()), ptr(dg.data_ptr()),
            B, T, H, _DTYPES[q.dtype], ptr(workspace.data_ptr()), nbytes,
            _stream_handle(stream, workspace.device))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_intra_bwd_host")
    return dq, dk, db, dg


def kda_intra_bwd_host_static(q, k, g, beta, dAqk, dAkk, dq, dk, db, dg, device=None,
                              stream=None):
    """``kda_intra_bwd_host`` without a workspace: for callers holding host tensors
    that may not allocate device memory.  The device staging is the library's own
    fixed array of ``HOST_STATIC_MAX_BYTES`` per GPU, so the problem must fit it
    (``kda_intra_bwd_host_workspace_bytes(B, T, H) <= HOST_STATIC_MAX_BYTES``, else
    ``KdaError`` with ``KDA_ERR_TOO_LARGE``).  Runs on ``device`` (default: the current
    CUDA device) and ``stream``; every call shares the one array, so calls must not
    overlap on the GPU.  Synchronise the stream before reading dq/dk/db/dg.
    """
    for n, t in (("q", q), ("k", k), ("g", g), ("beta", beta), ("dAqk", dAqk),
                 ("dAkk", dAkk), ("dq", dq), ("dk", dk), ("db", db), ("dg", dg)):
        if t.device.type != "cpu":
            raise ValueError(f"{n} must be a host tensor")
    B, T, H = _validate(q, k, g, beta, dAqk, dAkk, dq, dk, db, dg, torch.device("cpu"))
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None \
        else torch.device(device)
    lib = load_library()
    ptr = ctypes.c_void_p
    with torch.cuda.device(dev):
        rc = lib.kda_intra_bwd_host_static(
            ptr(q.data_ptr()), ptr(k.data_ptr()), ptr(g.data_ptr()), ptr(beta.data_ptr()),
            ptr(dAqk.data_ptr()), ptr(dAkk.data_ptr()), ptr(dq.data_ptr()),
            ptr(dk.data_ptr()), ptr(db.data_ptr()), ptr(dg.data_ptr()),
            B, T, H, _DTYPES[q.dtype], _stream_handle(stream, dev))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_intra_bwd_host_static")
    return dq, dk, db, dg
