"""Variable-length sequences (cu_seqlens / chunk_indices) through kda_intra_bwd_ex,
against the oracle's variable-length composition, element by element."""

import numpy as np
import pytest
import torch

import gated_delta_rule_intra_gb300 as kda
import kda_inputs
import oracle
from tests import _gpu

pytestmark = pytest.mark.gpu
TOL = _gpu.TOL["kda_intra_bwd"]

# one token, short, whole, ragged chunks; a sequence of whole chunks after a ragged one
EDGE_LENS = [1, 63, 64, 65, 127, 128, 129, 200, 7, 300, 2, 511]


def run_varlen(cpu, cu, chunk_indices=None, outs=None, **opts):
    dev = _gpu.to_device(cpu)
    devopts = {n: (v.cuda() if isinstance(v, torch.Tensor) else v) for n, v in opts.items()}
    ci = None if chunk_indices is None else chunk_indices.cuda()
    extra = {} if outs is None else dict(zip(_gpu.NAMES, outs))
    return kda.kda_intra_bwd_ex(*(dev[n] for n in _gpu.ARGS), cu_seqlens=cu.cuda(),
                                chunk_indices=ci, **extra, **devopts)


def ref_varlen(cpu, cu, **opts):
    return oracle.intra_bwd_varlen(*(cpu[n] for n in _gpu.ARGS), cu.numpy(), **opts)


def test_edge_lengths():
    cpu, cu = kda_inputs.make_varlen_inputs(EDGE_LENS, 3, seed=60)
    _gpu.assert_close(run_varlen(cpu, cu), ref_varlen(cpu, cu), TOL, "varlen edge lengths")


def test_fp16_gate_stress():
    lens = kda_inputs.varlen_seqlens(3000, seed=61, max_len=700)
    cpu, cu = kda_inputs.make_varlen_inputs(lens, 2, gate_lo=-8.0, qk_dtype=torch.float16,
                                            seed=62)
    _gpu.assert_close(run_varlen(cpu, cu), ref_varlen(cpu, cu), TOL, "varlen fp16 stress")


@pytest.mark.parametrize("G", [2, 4])
def test_grouped_value_heads(G):
    cpu, cu = kda_inputs.make_varlen_inputs(EDGE_LENS[:8], 2 * G, HQ=2, seed=63 + G)
    _gpu.assert_close(run_varlen(cpu, cu), ref_varlen(cpu, cu), TOL, f"varlen GVA G={G}")


def test_incoming_gradients_and_fold():
    cpu, cu = kda_inputs.make_varlen_inputs(EDGE_LENS, 2, seed=66)
    T = cpu["g"].shape[1]
    gen = torch.Generator().manual_seed(67)
    ins = dict(dq_in=torch.randn(1, T, 2, 128, generator=gen),
               dk_in=torch.randn(1, T, 2, 128, generator=gen),
               dg_in=torch.randn(1, T, 2, 128, generator=gen),
               db_in=torch.randn(1, T, 2, generator=gen))
    for fold in (False, True):
        _gpu.assert_close(run_varlen(cpu, cu, fold_dg=fold, **ins),
                          ref_varlen(cpu, cu, fold_dg=fold, **ins), TOL,
                          f"varlen accumulate, fold={fold}")


def test_io_dtype_outputs():
    cpu, cu = kda_inputs.make_varlen_inputs(EDGE_LENS[:6], 2, seed=68)
    f32 = run_varlen(cpu, cu)
    low = run_varlen(cpu, cu, dqdk_io_dtype=True)
    assert low[0].dtype == torch.bfloat16
    assert torch.equal(low[0], f32[0].to(torch.bfloat16))
    assert torch.equal(low[1], f32[1].to(torch.bfloat16))
    assert torch.equal(low[2], f32[2]) and torch.equal(low[3], f32[3])


def test_whole_chunks_match_the_fixed_length_kernel_bitwise():
    """Sequences of whole chunks: the same bytes as the fixed-length path on the
    packed tensor (only the dA tensor map and the masking code differ)."""
    cpu, cu = kda_inputs.make_varlen_inputs([128, 64, 320, 512], 4, seed=69)
    dev = _gpu.to_device(cpu)
    fixed = kda.kda_intra_bwd(*(dev[n] for n in _gpu.ARGS))
    var = run_varlen(cpu, cu)
    for n, a, b in zip(_gpu.NAMES, var, fixed):
        assert torch.equal(a, b), n


def test_foreign_rows_are_masked_and_untouched():
    """Rows past a sequence's end belong to the next sequence or to no sequence; the
    kernel reads them but must neither use nor write them.  Tokens after the last
    sequence carry NaN / huge inputs, dA entries outside each chunk's support are NaN,
    and the outputs start as a canary."""
    lens = [70, 33, 100]
    cpu, cu = kda_inputs.make_varlen_inputs(lens + [90], 2, seed=70)
    n = sum(lens)
    cu = cu[:-1].clone()  # the last 90 tokens belong to no sequence
    for name in ("q", "k"):
        cpu[name][0, n:] = float("nan")
    cpu["g"][0, n:] = 3e38
    cpu["beta"][0, n:] = float("nan")
    for name in ("dAqk", "dAkk"):
        x = cpu[name]
        x[x == 0] = float("nan")
        x[0, n:] = float("nan")
    T = cpu["g"].shape[1]
    canary = -7.25
    outs = [torch.full((1, T, 2, 128), canary, device="cuda"),
            torch.full((1, T, 2, 128), canary, device="cuda"),
            torch.full((1, T, 2), canary, device="cuda"),
            torch.full((1, T, 2, 128), canary, device="cuda")]
    got = run_varlen(cpu, cu, outs=outs)
    clean = {k: v.clone() for k, v in cpu.items()}
    for name in ("dAqk", "dAkk"):
        clean[name] = torch.nan_to_num(clean[name], nan=0.0)
    ref = ref_varlen(clean, cu)
    _gpu.assert_close([x[:, :n] for x in got], [r[:, :n] for r in ref], TOL,
                      "varlen with poisoned foreign rows")
    for x in got:
        assert bool((x[:, n:] == canary).all()), "a row outside every sequence was written"


def test_invalid_chunk_entries_are_skipped():
    """Entries naming no chunk (sequence out of range, chunk past the sequence's end,
    negative values) are skipped by the kernel's own checks; valid ones still run."""
    cpu, cu = kda_inputs.make_varlen_inputs([100, 64], 1, seed=71)
    ci = kda.prepare_chunk_indices(cu)  # (0,0) (0,1) (1,0)
    bad = torch.tensor([[0, 0], [5, 0], [0, 2], [-1, 0], [1, -3], [0, 1 << 30]],
                       dtype=torch.int32)
    T = cpu["g"].shape[1]
    canary = 3.5
    outs = [torch.full((1, T, 1, 128), canary, device="cuda"),
            torch.full((1, T, 1, 128), canary, device="cuda"),
            torch.full((1, T, 1), canary, device="cuda"),
            torch.full((1, T, 1, 128), canary, device="cuda")]
    got = run_varlen(cpu, cu, chunk_indices=bad, outs=outs)
    ref = ref_varlen(cpu, cu)
    # only chunk (0, 0) = tokens 0..63 was named validly
    _gpu.assert_close([x[:, :64] for x in got], [r[:, :64] for r in ref], TOL, "valid entry")
    for x in got:
        assert bool((x[:, 64:] == canary).all())
    assert ci.shape == (3, 2)


def test_empty_chunk_table_and_single_token():
    # one token: dq = dAqk[0,0] k, dk = dAqk[0,0] q, db = 0 and dg = 0 exactly (its
    # two terms cancel), so dg is checked in absolute terms
    cpu, cu = kda_inputs.make_varlen_inputs([1], 1, seed=72)
    got, ref = run_varlen(cpu, cu), ref_varlen(cpu, cu)
    _gpu.assert_close(got[:2], ref[:2], TOL, "T = 1")
    assert float(got[2].abs().max()) == 0.0
    assert float(got[3].abs().max()) < 1e-6 and abs(ref[3]).max() < 1e-12
    dev = _gpu.to_device(cpu)
    db = torch.full((1, 1, 1), 9.0, device="cuda")
    kda.kda_intra_bwd_ex(*(dev[n] for n in _gpu.ARGS), db=db,
                         cu_seqlens=torch.tensor([0, 0], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert db.item() == 9.0


def test_varlen_workload_full_size():
    """The variable-length workload (32768 tokens x 16 heads, log-uniform lengths in
    [1, 8192]), every element against the oracle."""
    cpu, cu = kda_inputs.make_varlen_workload()
    _gpu.assert_close(run_varlen(cpu, cu), ref_varlen(cpu, cu), TOL, "varlen workload")


def test_deterministic():
    cpu, cu = kda_inputs.make_varlen_inputs(EDGE_LENS, 2, seed=73)
    a = run_varlen(cpu, cu)
    b = run_varlen(cpu, cu)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    assert np.isfinite(a[3].cpu().numpy()).all()


def test_more_than_32_units_per_cta():
    """About 5,000 units with H = 7: every CTA crosses the 32-unit batches of row ranges
    it looks up ahead, with the head wrapping as it advances; forward and backward."""
    lens = kda_inputs.varlen_seqlens(45000, seed=141, max_len=3000)
    cpu, cu = kda_inputs.make_varlen_inputs(lens, 7, seed=142)
    chunks = int(sum(-(-n // 64) for n in lens))
    assert chunks * 7 > 32 * 152
    _gpu.assert_close(run_varlen(cpu, cu), ref_varlen(cpu, cu), TOL, "varlen, many units per CTA")
    dev = _gpu.to_device(cpu)
    got = kda.kda_intra_fwd(*(dev[n] for n in ("q", "k", "g", "beta")), cu_seqlens=cu.cuda())
    ref = oracle.intra_fwd_ex(*(cpu[n] for n in ("q", "k", "g", "beta")), cu_seqlens=cu.numpy())
    for name, a, b in zip(("Aqk", "Akk"), got, ref):
        a = a.double().cpu().numpy()
        err = float(np.max(np.abs(a - b)) / np.max(np.abs(b)))
        assert err <= TOL, (name, err)
