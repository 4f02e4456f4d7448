"""libkda loads, exports what include/kda.h declares, and rejects bad arguments
before touching the GPU (these tests never reach a CUDA call)."""

import ctypes
import os
import re

import pytest

import gated_delta_rule_intra_gb300 as kda

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")

(OK, ERR_NULL, ERR_SHAPE, ERR_DTYPE, ERR_ALIGN, ERR_CUDA, ERR_DEVICE, ERR_OVERLAP,
 ERR_WORKSPACE) = range(9)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    return kda.load_library()


def test_header_declares_the_entry_points():
    names = declared_functions()
    for want in ("kda_intra_bwd", "kda_intra_bwd_fp32", "kda_intra_bwd_host",
                 "kda_intra_bwd_host_workspace_bytes", "kda_status_str",
                 "kda_abi_version", "kda_intra_bwd_ex", "kda_intra_fwd"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"libkda.so does not export {name}"


def test_abi_version(lib):
    text = open(HEADER).read()
    want = int(re.search(r"#define KDA_ABI_VERSION (\d+)", text).group(1))
    assert kda.kda_abi_version() == want
    assert kda.ABI_VERSION == want  # the binding's struct mirrors follow this header


def test_status_strings(lib):
    for code in range(10):
        s = kda.kda_status_str(code)
        assert s.startswith("KDA_")
    assert kda.kda_status_str(99) == "KDA_ERR_UNKNOWN"


# Fake, never-dereferenced device addresses: validation must fail first.
BASE = 1 << 40
SPAN = 1 << 34


def fake_args(B=1, T=64, H=1, dtype=0, **override):
    ptrs = {n: BASE + i * SPAN for i, n in enumerate(
        ("q", "k", "g", "beta", "dAqk", "dAkk", "dq", "dk", "db", "dg"))}
    ptrs.update(override)
    vp = ctypes.c_void_p
    return [vp(ptrs[n]) for n in ("q", "k", "g", "beta", "dAqk", "dAkk", "dq", "dk", "db",
                                  "dg")] + [B, T, H, dtype, vp(0)]


@pytest.mark.parametrize("fn", ["kda_intra_bwd", "kda_intra_bwd_fp32"])
@pytest.mark.parametrize("case,want", [
    (dict(q=0), ERR_NULL),
    (dict(dg=0), ERR_NULL),
    (dict(beta=0), ERR_NULL),
    (dict(T=63), ERR_SHAPE),
    (dict(T=100), ERR_SHAPE),
    (dict(T=0), ERR_SHAPE),
    (dict(B=0), ERR_SHAPE),
    (dict(H=-1), ERR_SHAPE),
    (dict(H=65537), ERR_SHAPE),
    (dict(B=1 << 16, T=1 << 16), ERR_SHAPE),
    (dict(B=1 << 20, T=1 << 20, H=64), ERR_SHAPE),
    (dict(dtype=2), ERR_DTYPE),
    (dict(dtype=-1), ERR_DTYPE),
    (dict(q=BASE + 8), ERR_ALIGN),
    (dict(dAkk=BASE + 5 * SPAN + 4), ERR_ALIGN),
    (dict(dq=BASE + 6 * SPAN + 2), ERR_ALIGN),
    (dict(beta=BASE + 3 * SPAN + 2), ERR_ALIGN),
    (dict(dq=BASE), ERR_OVERLAP),                 # output aliases q
    (dict(dk=BASE + 6 * SPAN + 1024), ERR_OVERLAP),  # dk inside dq
    (dict(db=BASE + 9 * SPAN + 16), ERR_OVERLAP),    # db inside dg
])
def test_rejected_before_launch(lib, fn, case, want):
    case = dict(case)
    shape = {k: case.pop(k) for k in ("B", "T", "H", "dtype") if k in case}
    rc = getattr(lib, fn)(*fake_args(**shape, **case))
    assert rc == want, kda.kda_status_str(rc)


def test_inputs_may_alias_each_other(lib):
    # q == k is a legal call (read-only inputs); it must get past validation.  With
    # no GPU in this process the call then stops at the device query, never earlier.
    import torch
    if torch.cuda.is_available():
        pytest.skip("would launch on a real device")
    rc = lib.kda_intra_bwd(*fake_args(k=BASE))
    assert rc in (ERR_CUDA, ERR_DEVICE)


def test_host_entry_point_validation(lib):
    vp = ctypes.c_void_p
    args = fake_args()[:-1]
    need = lib.kda_intra_bwd_host_workspace_bytes(1, 64, 1, 0)
    assert need > 0
    assert lib.kda_intra_bwd_host(*args, vp(0), need, vp(0)) == ERR_WORKSPACE
    assert lib.kda_intra_bwd_host(*args, vp(BASE + 20 * SPAN), need - 1, vp(0)) == ERR_WORKSPACE
    assert lib.kda_intra_bwd_host(*args, vp(BASE + 20 * SPAN + 16), need, vp(0)) == ERR_ALIGN
    bad = fake_args(T=65)[:-1]
    assert lib.kda_intra_bwd_host(*bad, vp(BASE + 20 * SPAN), need, vp(0)) == ERR_SHAPE
    assert lib.kda_intra_bwd_host_workspace_bytes(1, 65, 1, 0) == 0
    assert lib.kda_intra_bwd_host_workspace_bytes(1, 64, 1, 7) == 0


def test_workspace_size_formula(lib):
    B, T, H = 2, 128, 3
    rows = B * T * H
    al = lambda x: (x + 255) // 256 * 256  # noqa: E731
    want = 2 * al(rows * 256) + 4 * al(rows * 512) + 2 * al(rows * 4) + 2 * al(rows * 256)
    assert lib.kda_intra_bwd_host_workspace_bytes(B, T, H, 0) == want


def test_python_binding_refuses_cpu_tensors():
    import torch
    q = torch.zeros(1, 64, 1, 128, dtype=torch.bfloat16)
    f = torch.zeros(1, 64, 1, 128)
    b = torch.zeros(1, 64, 1)
    a = torch.zeros(1, 64, 1, 64)
    with pytest.raises(ValueError, match="CUDA"):
        kda.kda_intra_bwd(q, q, f, b, a, a)


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="no fallback"):
        kda.load_library(str(tmp_path / "libkda.so"))


# ---------------------------------------------------------------- kda_intra_bwd_ex

def ex_call(lib, B=1, T=64, H=1, dtype=0, HV=0, fold=0, emit=0, ins=None, **override):
    args = fake_args(B, T, H, dtype, **override)[:-1]
    opts = kda.KdaOpts()
    opts.HV = HV
    opts.fold_dg = fold
    opts.dqdk_io_dtype = emit
    for name, val in (ins or {}).items():
        setattr(opts, name, val)
    return lib.kda_intra_bwd_ex(*args, ctypes.byref(opts), ctypes.c_void_p(0))


def test_ex_rejections(lib):
    assert ex_call(lib, H=2, HV=3) == ERR_SHAPE              # HV not a multiple of H
    assert ex_call(lib, H=2, HV=-2) == ERR_SHAPE
    assert ex_call(lib, H=1, HV=2, emit=1) == 9               # io-dtype outputs with GVA
    assert ex_call(lib, fold=2) == 9
    assert ex_call(lib, emit=3) == 9
    assert ex_call(lib, ins={"factor_diag": 2}) == 9
    assert ex_call(lib, ins={"factor_diag": -1}) == 9
    assert ex_call(lib, ins={"dq_in": BASE + 11 * SPAN + 2}) == ERR_ALIGN
    # an incoming gradient overlapping an output other than its own
    assert ex_call(lib, ins={"dk_in": BASE + 6 * SPAN}) == ERR_OVERLAP
    # partial overlap with its own output
    assert ex_call(lib, ins={"dq_in": BASE + 6 * SPAN + 64}) == ERR_OVERLAP
    assert ex_call(lib, q=0) == ERR_NULL


def test_ex_split_tf32_rejections(lib):
    """split_tf32 takes no other option but HV (and only the values 0 and 1)."""
    assert ex_call(lib, ins={"split_tf32": 2}) == 9
    assert ex_call(lib, ins={"split_tf32": -1}) == 9
    assert ex_call(lib, fold=1, ins={"split_tf32": 1}) == 9
    assert ex_call(lib, emit=1, ins={"split_tf32": 1}) == 9
    assert ex_call(lib, ins={"split_tf32": 1, "factor_diag": 1}) == 9
    assert ex_call(lib, ins={"split_tf32": 1, "db_in": BASE + 8 * SPAN}) == 9
    assert ex_call(lib, ins={"split_tf32": 1, **varlen_ins()}) == 9


def test_ex_accepts_in_place_and_reaches_the_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("would launch on a real device")
    ins = {"dq_in": BASE + 6 * SPAN, "dk_in": BASE + 7 * SPAN, "db_in": BASE + 8 * SPAN,
           "dg_in": BASE + 9 * SPAN}
    assert ex_call(lib, H=2, HV=4, fold=1, ins=ins) in (ERR_CUDA, ERR_DEVICE)
    assert ex_call(lib, emit=1) in (ERR_CUDA, ERR_DEVICE)
    assert ex_call(lib, ins={"factor_diag": 1}) in (ERR_CUDA, ERR_DEVICE)
    assert ex_call(lib, H=2, HV=4, ins={"split_tf32": 1}) in (ERR_CUDA, ERR_DEVICE)
    # NULL options behave like kda_intra_bwd
    args = fake_args()[:-1]
    assert lib.kda_intra_bwd_ex(*args, None, ctypes.c_void_p(0)) in (ERR_CUDA, ERR_DEVICE)


def varlen_ins(num_seqs=2, num_chunks=3, cu=BASE + 10 * SPAN, ci=BASE + 11 * SPAN):
    return {"cu_seqlens": cu, "chunk_indices": ci, "num_seqs": num_seqs,
            "num_chunks": num_chunks}


def test_ex_varlen_rejections(lib):
    assert ex_call(lib, B=2, T=128, ins=varlen_ins()) == ERR_SHAPE        # varlen needs B == 1
    assert ex_call(lib, ins=varlen_ins(num_seqs=0)) == ERR_SHAPE
    assert ex_call(lib, ins=varlen_ins(num_chunks=-1)) == ERR_SHAPE
    assert ex_call(lib, T=0, ins=varlen_ins()) == ERR_SHAPE
    assert ex_call(lib, H=1, HV=1 << 16, ins=varlen_ins(num_chunks=1 << 16)) == ERR_SHAPE
    assert ex_call(lib, ins=varlen_ins(cu=0)) == ERR_NULL                  # table without offsets
    assert ex_call(lib, ins=varlen_ins(ci=0)) == ERR_NULL                  # offsets, chunks, no table
    assert ex_call(lib, ins=varlen_ins(cu=BASE + 10 * SPAN + 2)) == ERR_ALIGN
    assert ex_call(lib, ins=varlen_ins(ci=BASE + 11 * SPAN + 1)) == ERR_ALIGN
    # the offsets inside an output buffer
    assert ex_call(lib, ins=varlen_ins(cu=BASE + 8 * SPAN + 16)) == ERR_OVERLAP
    # a chunk table running into db
    assert ex_call(lib, ins=varlen_ins(ci=BASE + 8 * SPAN - 8, num_chunks=2)) == ERR_OVERLAP
    # and without varlen, T % 64 is still required
    assert ex_call(lib, T=100) == ERR_SHAPE


def test_ex_varlen_accepts_any_token_count(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("would launch on a real device")
    for T in (1, 63, 100, 64 * 7 + 5):
        assert ex_call(lib, T=T, ins=varlen_ins()) in (ERR_CUDA, ERR_DEVICE)
    # an empty chunk table may be NULL
    assert ex_call(lib, T=5, ins=varlen_ins(ci=0, num_chunks=0)) in (ERR_CUDA, ERR_DEVICE, 0)


def test_prepare_chunk_indices():
    import torch
    cu = torch.tensor([0, 1, 64, 64, 193, 200], dtype=torch.int32)
    ci = kda.prepare_chunk_indices(cu)
    assert ci.dtype == torch.int32 and ci.shape == (6, 2)
    assert ci.tolist() == [[0, 0], [1, 0], [3, 0], [3, 1], [3, 2], [4, 0]]
    assert kda.prepare_chunk_indices(torch.tensor([0, 0])).shape == (0, 2)
    with pytest.raises(ValueError):
        kda.prepare_chunk_indices(torch.tensor([1, 5]))
    with pytest.raises(ValueError):
        kda.prepare_chunk_indices(torch.tensor([0, 5, 3]))


# ---------------------------------------------------------------- kda_intra_fwd

def fwd_call(lib, B=1, T=64, H=1, dtype=0, **override):
    ptrs = {n: BASE + i * SPAN for i, n in enumerate(("q", "k", "g", "beta", "Aqk", "Akk"))}
    ptrs.update(override)
    vp = ctypes.c_void_p
    args = [vp(ptrs[n]) for n in ("q", "k", "g", "beta", "Aqk", "Akk")]
    return lib.kda_intra_fwd(*args, B, T, H, dtype, vp(0))


@pytest.mark.parametrize("case,want", [
    (dict(q=0), ERR_NULL),
    (dict(Akk=0), ERR_NULL),
    (dict(T=100), ERR_SHAPE),
    (dict(H=0), ERR_SHAPE),
    (dict(B=1 << 16, T=1 << 16), ERR_SHAPE),
    (dict(dtype=5), ERR_DTYPE),
    (dict(g=BASE + 2 * SPAN + 4), ERR_ALIGN),
    (dict(Aqk=BASE + 4 * SPAN + 8), ERR_ALIGN),
    (dict(beta=BASE + 3 * SPAN + 1), ERR_ALIGN),
    (dict(Aqk=BASE + 2 * SPAN), ERR_OVERLAP),        # output aliases g
    (dict(Akk=BASE + 4 * SPAN + 256), ERR_OVERLAP),  # Akk inside Aqk
])
def test_fwd_rejected_before_launch(lib, case, want):
    case = dict(case)
    shape = {k: case.pop(k) for k in ("B", "T", "H", "dtype") if k in case}
    rc = fwd_call(lib, **shape, **case)
    assert rc == want, kda.kda_status_str(rc)


def test_fwd_valid_call_reaches_the_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("would launch on a real device")
    assert fwd_call(lib) in (ERR_CUDA, ERR_DEVICE)


def fwd_ex_call(lib, B=1, T=64, H=1, dtype=0, HV=0, ins=None, **override):
    ptrs = {n: BASE + i * SPAN for i, n in enumerate(("q", "k", "g", "beta", "Aqk", "Akk"))}
    ptrs.update(override)
    vp = ctypes.c_void_p
    opts = kda.KdaFwdOpts()
    opts.HV = HV
    for name, val in (ins or {}).items():
        setattr(opts, name, val)
    args = [vp(ptrs[n]) for n in ("q", "k", "g", "beta", "Aqk", "Akk")]
    return lib.kda_intra_fwd_ex(*args, B, T, H, dtype, ctypes.byref(opts), vp(0))


def test_fwd_ex_rejections(lib):
    assert fwd_ex_call(lib, H=2, HV=3) == ERR_SHAPE
    assert fwd_ex_call(lib, B=2, T=128, ins=varlen_ins()) == ERR_SHAPE
    assert fwd_ex_call(lib, ins=varlen_ins(num_seqs=0)) == ERR_SHAPE
    assert fwd_ex_call(lib, ins=varlen_ins(cu=0)) == ERR_NULL
    assert fwd_ex_call(lib, ins=varlen_ins(ci=BASE + 11 * SPAN + 2)) == ERR_ALIGN
    assert fwd_ex_call(lib, ins=varlen_ins(cu=BASE + 4 * SPAN + 64)) == ERR_OVERLAP  # in Aqk
    assert fwd_ex_call(lib, T=100) == ERR_SHAPE


def test_fwd_ex_accepts_groups_and_varlen(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("would launch on a real device")
    assert fwd_ex_call(lib, H=2, HV=8) in (ERR_CUDA, ERR_DEVICE)
    assert fwd_ex_call(lib, T=100, ins=varlen_ins()) in (ERR_CUDA, ERR_DEVICE)


def test_option_structs_match_the_header(tmp_path):
    """The binding's ctypes option structs have the C header's size and field offsets
    (compiled here with the host C compiler)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no host C compiler")
    structs = {"kda_intra_bwd_opts_t": kda.KdaOpts, "kda_intra_fwd_opts_t": kda.KdaFwdOpts}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "kda.h"', "int main(void) {"]
    for cname, py in structs.items():
        lines.append(f'printf("{cname} size %zu\\n", sizeof({cname}));')
        for field, _ in py._fields_:
            lines.append(f'printf("{cname} {field} %zu\\n", offsetof({cname}, {field}));')
    lines += ["return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    got = {tuple(l.split()[:2]): int(l.split()[2]) for l in out.splitlines()}
    for cname, py in structs.items():
        assert got[(cname, "size")] == ctypes.sizeof(py), cname
        for field, _ in py._fields_:
            assert got[(cname, field)] == getattr(py, field).offset, (cname, field)


def test_release_build_has_no_debug_checks(lib):
    assert lib.kda_debug_checks() == 0
    assert lib.kda_debug_set_flags(None) == 9  # KDA_ERR_OPTION


def test_debug_build_loads_and_takes_a_flag_word():
    dbg = kda.load_library(kda.DEBUG_LIB_PATH)
    for name in declared_functions():
        assert hasattr(dbg, name), f"libkda_debug.so does not export {name}"
    assert dbg.kda_debug_checks() == 1
    assert dbg.kda_abi_version() == kda.kda_abi_version()
    assert dbg.kda_debug_set_flags(ctypes.c_void_p(BASE + 2)) == ERR_ALIGN
    assert dbg.kda_debug_set_flags(None) == OK
    # the same argument checks as the release build
    assert ex_call(dbg, H=2, HV=3) == ERR_SHAPE
    assert ex_call(dbg, ins={"factor_diag": 2}) == 9
