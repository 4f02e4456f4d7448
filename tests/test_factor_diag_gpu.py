"""The factorized diagonal quadrant (kda_intra_bwd_ex's factor_diag option) against the
oracle, element by element, and against the exact diagonal form of the same kernel."""

import numpy as np
import pytest
import torch

import gated_delta_rule_intra_gb300 as kda
import kda_inputs
import oracle
from tests import _gpu

pytestmark = pytest.mark.gpu
TOL = _gpu.TOL["kda_intra_bwd"]


def run_fd(dev, factor=True, **opts):
    return kda.kda_intra_bwd_ex(*(dev[n] for n in _gpu.ARGS), factor_diag=factor, **opts)


@pytest.mark.parametrize("cfg", [kda_inputs.SINGLE_CHUNK, kda_inputs.SMALL, kda_inputs.HEADLINE])
def test_configs_every_element(cfg):
    cpu = kda_inputs.make_config_inputs(cfg)
    got = run_fd(_gpu.to_device(cpu))
    _gpu.assert_close(got, _gpu.oracle_outputs(cpu), TOL, f"factor_diag config {cfg}")


@pytest.mark.parametrize("cfg", [kda_inputs.LONG, kda_inputs.GATE_STRESS])
def test_large_configs_sampled_units(cfg):
    """B=1 T=32768 H=32 and the fp16 gate-stress workload (g down to about -500)."""
    cpu = kda_inputs.make_config_inputs(cfg)
    dev = _gpu.to_device(cpu)
    outs = run_fd(dev)
    torch.cuda.synchronize()
    for x in outs:
        assert bool(torch.isfinite(x).all())
    _gpu.sampled_parity("kda_intra_bwd", cfg, cpu, dev, outs=outs, n_units=24)


@pytest.mark.parametrize("gate_lo", [-8.0, -40.0])
def test_steep_gates(gate_lo):
    """Per-step log2 gates down to -40: inside a 16-row block the exact E spans 2^-600,
    so both factors of the quadrant underflow in places; every exponent stays <= 0."""
    cpu = kda_inputs.make_inputs(2, 256, 3, gate_lo=gate_lo, qk_dtype=torch.float16, seed=110)
    got = run_fd(_gpu.to_device(cpu))
    for x in got:
        assert bool(torch.isfinite(x).all())
    _gpu.assert_close(got, _gpu.oracle_outputs(cpu), TOL, f"factor_diag gate_lo={gate_lo}")


def test_close_to_the_exact_diagonal_at_full_size():
    """Same kernel, same inputs: the two diagonal forms differ by rounding only."""
    cpu = kda_inputs.make_config_inputs(kda_inputs.HEADLINE)
    dev = _gpu.to_device(cpu)
    exact = run_fd(dev, factor=False)
    fact = run_fd(dev, factor=True)
    for n, a, b in zip(_gpu.NAMES, exact, fact):
        rel = ((a - b).abs().max() / a.abs().max()).item()
        assert rel <= 1e-5, (n, rel)


def test_exact_form_is_the_default():
    cpu = kda_inputs.make_inputs(2, 192, 2, seed=111)
    dev = _gpu.to_device(cpu)
    plain = kda.kda_intra_bwd(*(dev[n] for n in _gpu.ARGS))
    off = run_fd(dev, factor=False)
    for n, a, b in zip(_gpu.NAMES, plain, off):
        assert torch.equal(a, b), n


def test_with_every_other_option():
    """GVA, incoming gradients and fold_dg together with the factorized quadrant."""
    G = 2
    x = kda_inputs.make_inputs(2, 192, 2 * G, seed=112)
    x["q"] = x["q"][:, :, ::G].contiguous()
    x["k"] = x["k"][:, :, ::G].contiguous()
    gen = torch.Generator().manual_seed(113)
    ins = dict(dq_in=torch.randn(2, 192, 2 * G, 128, generator=gen),
               dk_in=torch.randn(2, 192, 2 * G, 128, generator=gen),
               dg_in=torch.randn(2, 192, 2 * G, 128, generator=gen),
               db_in=torch.randn(2, 192, 2 * G, generator=gen))
    dev = _gpu.to_device(x)
    got = run_fd(dev, fold_dg=True, **{n: v.cuda() for n, v in ins.items()})
    ref = oracle.intra_bwd_ex(*(x[n] for n in _gpu.ARGS), fold_dg=True, **ins)
    _gpu.assert_close(got, ref, TOL, "factor_diag + GVA + accumulate + fold")


def test_io_dtype_outputs_are_the_rounded_fp32_results():
    cpu = kda_inputs.make_inputs(2, 128, 3, qk_dtype=torch.float16, seed=114)
    dev = _gpu.to_device(cpu)
    f32 = run_fd(dev)
    low = run_fd(dev, dqdk_io_dtype=True)
    assert torch.equal(low[0], f32[0].to(torch.float16))
    assert torch.equal(low[1], f32[1].to(torch.float16))
    assert torch.equal(low[2], f32[2]) and torch.equal(low[3], f32[3])


EDGE_LENS = [1, 63, 64, 65, 127, 128, 129, 200, 7, 300, 2, 511]


def test_varlen_edge_lengths():
    cpu, cu = kda_inputs.make_varlen_inputs(EDGE_LENS, 3, seed=115)
    got = run_fd(_gpu.to_device(cpu), cu_seqlens=cu.cuda())
    ref = oracle.intra_bwd_varlen(*(cpu[n] for n in _gpu.ARGS), cu.numpy())
    _gpu.assert_close(got, ref, TOL, "factor_diag varlen")


def test_varlen_whole_chunks_match_fixed_length_bitwise():
    cpu, cu = kda_inputs.make_varlen_inputs([128, 64, 320], 2, seed=116)
    dev = _gpu.to_device(cpu)
    a = run_fd(dev, cu_seqlens=cu.cuda())
    b = run_fd(dev)
    for n, x, y in zip(_gpu.NAMES, a, b):
        assert torch.equal(x, y), n


def test_varlen_poisoned_foreign_rows():
    """Tokens after the last sequence carry NaN / huge inputs and dA entries outside the
    support are NaN: the quadrant reads only pairs s < r of valid rows."""
    lens = [70, 33, 100]
    cpu, cu = kda_inputs.make_varlen_inputs(lens + [90], 2, seed=117)
    n = sum(lens)
    cu = cu[:-1].clone()
    for name in ("q", "k", "beta"):
        cpu[name][0, n:] = float("nan")
    cpu["g"][0, n:] = 3e38
    for name in ("dAqk", "dAkk"):
        x = cpu[name]
        x[x == 0] = float("nan")
        x[0, n:] = float("nan")
    T = cpu["g"].shape[1]
    canary = 9.5
    outs = [torch.full((1, T, 2, 128), canary, device="cuda"),
            torch.full((1, T, 2, 128), canary, device="cuda"),
            torch.full((1, T, 2), canary, device="cuda"),
            torch.full((1, T, 2, 128), canary, device="cuda")]
    got = run_fd(_gpu.to_device(cpu), cu_seqlens=cu.cuda(), **dict(zip(_gpu.NAMES, outs)))
    clean = {k: v.clone() for k, v in cpu.items()}
    for name in ("dAqk", "dAkk"):
        clean[name] = torch.nan_to_num(clean[name], nan=0.0)
    ref = oracle.intra_bwd_varlen(*(clean[k] for k in _gpu.ARGS), cu.numpy())
    _gpu.assert_close([x[:, :n] for x in got], [np.asarray(r)[:, :n] for r in ref], TOL,
                      "factor_diag varlen poisoned")
    for x in got:
        assert bool((x[:, n:] == canary).all())
