"""kda_intra_fwd (the score matrices Aqk, Akk) against the oracle's forward, through
the C ABI."""

import numpy as np
import pytest
import torch

import gated_delta_rule_intra_gb300 as kda
import kda_inputs
import oracle
from tests import _gpu

pytestmark = pytest.mark.gpu
TOL = 2e-3  # max|err| / max|ref| per tensor (TF32 cross terms, fp32 diagonal)
IN = ("q", "k", "g", "beta")


def run_fwd(cpu, **kw):
    dev = _gpu.to_device({n: cpu[n] for n in IN})
    return kda.kda_intra_fwd(*(dev[n] for n in IN), **kw)


def ref_fwd(cpu):
    return oracle.intra_fwd(*(cpu[n] for n in IN))


def rel(a, b):
    a = a.detach().double().cpu().numpy() if isinstance(a, torch.Tensor) else a
    return float(np.max(np.abs(a - b)) / np.max(np.abs(b)))


def assert_fwd_close(got, ref, what):
    errs = {n: rel(a, b) for n, a, b in zip(("Aqk", "Akk"), got, ref)}
    assert all(e <= TOL for e in errs.values()), f"{what}: {errs}"


@pytest.mark.parametrize("idx", [kda_inputs.SINGLE_CHUNK, kda_inputs.SMALL, kda_inputs.HEADLINE])
def test_full_workloads(idx):
    cpu = kda_inputs.make_config_inputs(idx)
    assert_fwd_close(run_fwd(cpu), ref_fwd(cpu), kda_inputs.CONFIGS[idx].name)


def per_unit_rel(a, b, bt=64):
    """max|err| / max|ref| of every unit (b, chunk, h) of a [B, T, H, 64] pair: a wrong
    unit whose entries are small cannot hide under the tensor-wide max|ref|."""
    a = a.detach().double().cpu().numpy() if isinstance(a, torch.Tensor) else a
    B, T, H, n = b.shape
    err = np.abs(a - b).reshape(B, T // bt, bt, H, n).max(axis=(2, 4))
    ref = np.abs(b).reshape(B, T // bt, bt, H, n).max(axis=(2, 4))
    return err / np.maximum(ref, 1e-300), ref


@pytest.mark.parametrize("idx", [kda_inputs.LONG, kda_inputs.GATE_STRESS])
def test_large_workloads_element_wise(idx):
    """Every element of the two largest workloads (16,384 and 32,768 units) against the
    oracle, per tensor and per unit."""
    cfg = kda_inputs.CONFIGS[idx]
    cpu = kda_inputs.make_config_inputs(idx)
    got = run_fwd(cpu)
    ref = ref_fwd(cpu)
    assert_fwd_close(got, ref, cfg.name)
    for name, a, b in zip(("Aqk", "Akk"), got, ref):
        unit_err, unit_ref = per_unit_rel(a, b)
        worst = np.unravel_index(np.argmax(unit_err), unit_err.shape)
        print(f"{cfg.name} {name}: per-unit max|err|/max|ref| worst {unit_err.max():.2e} "
              f"at (b, chunk, h) = {tuple(int(i) for i in worst)}, median "
              f"{np.median(unit_err):.2e}; smallest unit max|ref| {unit_ref.min():.2e}")
        assert unit_err.max() <= TOL, (name, unit_err.max(), worst)


def test_strided_q_is_refused():
    """A q view that is not contiguous (every other head of a wider tensor, or a
    transposed one) would be read with dense strides; the binding refuses it."""
    cpu = kda_inputs.make_inputs(2, 64, 4, seed=79)
    dev = _gpu.to_device({n: cpu[n] for n in IN})
    wide = torch.cat([dev["q"], dev["q"]], dim=2)[:, :, ::2]
    assert tuple(wide.shape) == tuple(dev["q"].shape) and not wide.is_contiguous()
    with pytest.raises(ValueError, match="q must be contiguous"):
        kda.kda_intra_fwd(wide, dev["k"], dev["g"], dev["beta"])
    with pytest.raises(ValueError, match="q must be contiguous"):
        kda.kda_intra_fwd(dev["q"].transpose(1, 2), dev["k"], dev["g"], dev["beta"])


def test_outputs_fully_written_and_zero_outside_support():
    cpu = kda_inputs.make_inputs(2, 192, 3, seed=80)
    dev = _gpu.to_device({n: cpu[n] for n in IN})
    Aqk = torch.full((2, 192, 3, 64), float("nan"), device="cuda")
    Akk = torch.full((2, 192, 3, 64), float("nan"), device="cuda")
    kda.kda_intra_fwd(*(dev[n] for n in IN), Aqk=Aqk, Akk=Akk)
    assert bool(torch.isfinite(Aqk).all()) and bool(torch.isfinite(Akk).all())
    lower, strict = kda_inputs.chunk_masks()
    a = Aqk.view(2, 3, 64, 3, 64).cpu()
    b = Akk.view(2, 3, 64, 3, 64).cpu()
    up = ~lower  # s > r
    for r in range(64):
        assert bool((a[:, :, r, :, up[r]] == 0).all()), r
        assert bool((b[:, :, r, :, ~strict[r]] == 0).all()), r
    assert_fwd_close((Aqk, Akk), ref_fwd(cpu), "small")


@pytest.mark.parametrize("B,T,H,dtype", [(1, 64, 1, torch.bfloat16), (3, 128, 5, torch.float16),
                                         (2, 320, 7, torch.bfloat16), (1, 64, 200, torch.float16)])
def test_odd_shapes(B, T, H, dtype):
    cpu = kda_inputs.make_inputs(B, T, H, qk_dtype=dtype, seed=83 + H)
    assert_fwd_close(run_fwd(cpu), ref_fwd(cpu), f"B={B} T={T} H={H}")


def test_fp16_gate_stress_small():
    cpu = kda_inputs.make_inputs(1, 512, 2, gate_lo=-8.0, qk_dtype=torch.float16, seed=81)
    assert_fwd_close(run_fwd(cpu), ref_fwd(cpu), "fp16 stress")


def test_deterministic_and_side_stream():
    cpu = kda_inputs.make_inputs(2, 256, 4, seed=82)
    a = run_fwd(cpu)
    s = torch.cuda.Stream()
    dev = _gpu.to_device({n: cpu[n] for n in IN})
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        b = kda.kda_intra_fwd(*(dev[n] for n in IN), stream=s)
    s.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_forward_and_backward_satisfy_euler_identities():
    """At full size (the headline workload), the two kernels against each other:
    sum q*dq = sum dAqk*Aqk and sum beta*db = sum dAkk*Akk (homogeneity of Aqk in q
    and of Akk in beta)."""
    cpu = kda_inputs.make_config_inputs(kda_inputs.HEADLINE)
    dev = _gpu.to_device(cpu)
    Aqk, Akk = kda.kda_intra_fwd(*(dev[n] for n in IN))
    dq, dk, db, dg = kda.kda_intra_bwd(*(dev[n] for n in _gpu.ARGS))
    lhs1 = (dev["q"].double() * dq.double()).sum().item()
    rhs1 = (dev["dAqk"].double() * Aqk.double()).sum().item()
    lhs2 = (dev["beta"].double() * db.double()).sum().item()
    rhs2 = (dev["dAkk"].double() * Akk.double()).sum().item()
    scale1 = (dev["dAqk"].double().abs() * Aqk.double().abs()).sum().item()
    scale2 = (dev["dAkk"].double().abs() * Akk.double().abs()).sum().item()
    assert abs(lhs1 - rhs1) <= 1e-3 * scale1, (lhs1, rhs1)
    assert abs(lhs2 - rhs2) <= 1e-3 * scale2, (lhs2, rhs2)


# ---------------------------------------------------------------- options (kda_intra_fwd_ex)

def ref_fwd_ex(cpu, cu=None):
    return oracle.intra_fwd_ex(*(cpu[n] for n in IN),
                               cu_seqlens=None if cu is None else cu.numpy())


def run_fwd_ex(cpu, cu=None, chunk_indices=None, **kw):
    dev = _gpu.to_device({n: cpu[n] for n in IN})
    extra = {}
    if cu is not None:
        extra["cu_seqlens"] = cu.cuda()
        if chunk_indices is not None:
            extra["chunk_indices"] = chunk_indices.cuda()
    return kda.kda_intra_fwd(*(dev[n] for n in IN), **extra, **kw)


@pytest.mark.parametrize("G", [2, 4])
def test_grouped_value_heads(G):
    x = kda_inputs.make_inputs(2, 192, 2 * G, seed=90 + G)
    x["q"] = x["q"][:, :, ::G].contiguous()
    x["k"] = x["k"][:, :, ::G].contiguous()
    assert_fwd_close(run_fwd_ex(x), ref_fwd_ex(x), f"fwd GVA G={G}")


VARLEN_LENS = [1, 63, 64, 65, 127, 128, 129, 200, 7, 300, 2, 511]


@pytest.mark.parametrize("qk_dtype,gate_lo", [(torch.bfloat16, -0.5), (torch.float16, -8.0)])
def test_varlen(qk_dtype, gate_lo):
    cpu, cu = kda_inputs.make_varlen_inputs(VARLEN_LENS, 3, gate_lo=gate_lo, qk_dtype=qk_dtype,
                                            seed=94)
    assert_fwd_close(run_fwd_ex(cpu, cu), ref_fwd_ex(cpu, cu), f"fwd varlen {qk_dtype}")


def test_varlen_with_groups():
    cpu, cu = kda_inputs.make_varlen_inputs(VARLEN_LENS[:8], 4, HQ=2, seed=95)
    assert_fwd_close(run_fwd_ex(cpu, cu), ref_fwd_ex(cpu, cu), "fwd varlen GVA")


def test_varlen_whole_chunks_match_the_fixed_length_kernel_bitwise():
    cpu, cu = kda_inputs.make_varlen_inputs([128, 64, 320], 2, seed=96)
    a = run_fwd_ex(cpu, cu)
    b = run_fwd(cpu)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_varlen_foreign_rows_untouched():
    """Tokens after the last sequence carry NaN / huge inputs; the outputs start as a
    canary: valid rows match the oracle, rows outside every sequence stay canary."""
    lens = [70, 33, 100]
    cpu, cu = kda_inputs.make_varlen_inputs(lens + [90], 2, seed=97)
    n = sum(lens)
    cu = cu[:-1].clone()
    for name in ("q", "k", "beta"):
        cpu[name][0, n:] = float("nan")
    cpu["g"][0, n:] = 3e38
    T = cpu["g"].shape[1]
    canary = -5.5
    Aqk = torch.full((1, T, 2, 64), canary, device="cuda")
    Akk = torch.full((1, T, 2, 64), canary, device="cuda")
    got = run_fwd_ex(cpu, cu, Aqk=Aqk, Akk=Akk)
    ref = ref_fwd_ex(cpu, cu)
    assert_fwd_close([x[:, :n] for x in got], [r[:, :n] for r in ref], "fwd varlen poisoned")
    for x in got:
        assert bool((x[:, n:] == canary).all())


def test_varlen_invalid_entries_skipped():
    cpu, cu = kda_inputs.make_varlen_inputs([100, 64], 1, seed=98)
    bad = torch.tensor([[0, 0], [5, 0], [0, 2], [-1, 0], [1, -3]], dtype=torch.int32)
    T = cpu["g"].shape[1]
    Aqk = torch.full((1, T, 1, 64), 2.5, device="cuda")
    Akk = torch.full((1, T, 1, 64), 2.5, device="cuda")
    got = run_fwd_ex(cpu, cu, chunk_indices=bad, Aqk=Aqk, Akk=Akk)
    ref = ref_fwd_ex(cpu, cu)
    assert_fwd_close([x[:, :64] for x in got], [r[:, :64] for r in ref], "valid entry")
    for x in got:
        assert bool((x[:, 64:] == 2.5).all())


def test_varlen_workload_full_size():
    cpu, cu = kda_inputs.make_varlen_workload()
    assert_fwd_close(run_fwd_ex(cpu, cu), ref_fwd_ex(cpu, cu), "fwd varlen workload")
