"""kda_intra_bwd_ex against the oracle's extended contract, through the C ABI."""

import pytest
import torch

import gated_delta_rule_intra_gb300 as kda
import kda_inputs
import oracle
from tests import _gpu

pytestmark = pytest.mark.gpu
TOL = _gpu.TOL["kda_intra_bwd"]


def grouped_inputs(B, T, H, G, seed, qk_dtype=torch.bfloat16, gate_lo=-0.5):
    """q, k with H heads; everything else with H*G heads."""
    x = kda_inputs.make_inputs(B, T, H * G, gate_lo=gate_lo, qk_dtype=qk_dtype, seed=seed)
    x["q"] = x["q"][:, :, ::G].contiguous()
    x["k"] = x["k"][:, :, ::G].contiguous()
    return x


def incoming(B, T, HV, seed):
    gen = torch.Generator().manual_seed(seed)
    return dict(dq_in=torch.randn(B, T, HV, 128, generator=gen),
                dk_in=torch.randn(B, T, HV, 128, generator=gen),
                dg_in=torch.randn(B, T, HV, 128, generator=gen),
                db_in=torch.randn(B, T, HV, generator=gen))


def run_ex(cpu, **opts):
    dev = _gpu.to_device(cpu)
    devopts = {n: (v.cuda() if isinstance(v, torch.Tensor) else v) for n, v in opts.items()}
    return kda.kda_intra_bwd_ex(*(dev[n] for n in _gpu.ARGS), **devopts)


def ref_ex(cpu, **opts):
    return oracle.intra_bwd_ex(*(cpu[n] for n in _gpu.ARGS), **opts)


@pytest.mark.parametrize("G", [1, 2, 4])
def test_grouped_value_heads(G):
    cpu = grouped_inputs(2, 128, 2, G, seed=30 + G)
    _gpu.assert_close(run_ex(cpu), ref_ex(cpu), TOL, f"GVA G={G}")


def test_grouped_value_heads_fp16_stress():
    cpu = grouped_inputs(1, 256, 3, 2, seed=40, qk_dtype=torch.float16, gate_lo=-8.0)
    _gpu.assert_close(run_ex(cpu), ref_ex(cpu), TOL, "GVA fp16 stress")


@pytest.mark.parametrize("G", [2, 4])
def test_split_tf32_with_grouped_value_heads(G):
    """The split-TF32 cross sums with HV = G*H value heads (q/k read per group), held to
    the FP32 path's tolerance; 3 q/k heads x 64 chunks so that the persistent CTAs walk
    several units each and the group index wraps across them."""
    cpu = grouped_inputs(2, 2048, 3, G, seed=60 + G)
    got = run_ex(cpu, split_tf32=True)
    _gpu.assert_close(got, ref_ex(cpu), _gpu.TOL["split_tf32"], f"split_tf32 G={G}")


def test_incoming_gradients_added():
    cpu = kda_inputs.make_inputs(2, 192, 3, seed=41)
    ins = incoming(2, 192, 3, seed=42)
    _gpu.assert_close(run_ex(cpu, **ins), ref_ex(cpu, **ins), TOL, "accumulate")


def test_incoming_gradients_partial_and_in_place():
    cpu = kda_inputs.make_inputs(1, 128, 2, seed=43)
    ins = incoming(1, 128, 2, seed=44)
    only = {"dk_in": ins["dk_in"], "db_in": ins["db_in"]}
    _gpu.assert_close(run_ex(cpu, **only), ref_ex(cpu, **only), TOL, "partial accumulate")
    # in place: the output tensors are the incoming gradients
    dev = _gpu.to_device(cpu)
    bufs = {n: v.cuda() for n, v in ins.items()}
    out = kda.kda_intra_bwd_ex(*(dev[n] for n in _gpu.ARGS), dq=bufs["dq_in"], dk=bufs["dk_in"],
                               db=bufs["db_in"], dg=bufs["dg_in"], **bufs)
    assert out[0].data_ptr() == bufs["dq_in"].data_ptr()
    ref = run_ex(cpu, **ins)
    for n, a, b in zip(_gpu.NAMES, out, ref):
        assert torch.equal(a, b), f"in-place {n} differs from out-of-place"


@pytest.mark.parametrize("fold", [False, True])
@pytest.mark.parametrize("varlen", [False, True])
def test_in_place_accumulation_matches_out_of_place(fold, varlen):
    """dq_in, dk_in, dg_in given as the outputs themselves: the stores add to them in L2
    (dg_in is read before the fold); bitwise the out-of-place result, for whole and short
    chunks.  Partly in place (dq only) takes the loading path and agrees too."""
    if varlen:
        lens = [70, 1, 130, 64]
        B, T = 1, sum(lens)
        cpu, cu = kda_inputs.make_varlen_inputs(lens, 3, seed=47)
        extra = {"cu_seqlens": cu.cuda()}
    else:
        B, T = 2, 192
        cpu = kda_inputs.make_inputs(B, T, 3, seed=47)
        extra = {}
    ins = incoming(B, T, 3, seed=48)
    dev = _gpu.to_device(cpu)
    ref = kda.kda_intra_bwd_ex(*(dev[n] for n in _gpu.ARGS), fold_dg=fold,
                               **{n: v.cuda() for n, v in ins.items()}, **extra)
    bufs = {n: v.cuda() for n, v in ins.items()}
    out = kda.kda_intra_bwd_ex(*(dev[n] for n in _gpu.ARGS), dq=bufs["dq_in"], dk=bufs["dk_in"],
                               db=bufs["db_in"], dg=bufs["dg_in"], fold_dg=fold, **bufs, **extra)
    for n, a, b in zip(_gpu.NAMES, out, ref):
        assert torch.equal(a, b), f"in-place {n} differs from out-of-place"
    part = {n: v.cuda() for n, v in ins.items()}
    dq = part["dq_in"]
    got = kda.kda_intra_bwd_ex(*(dev[n] for n in _gpu.ARGS), dq=dq, fold_dg=fold, **part, **extra)
    for n, a, b in zip(_gpu.NAMES, got, ref):
        assert torch.equal(a, b), f"partly in-place {n} differs from out-of-place"


def test_fold_dg():
    cpu = kda_inputs.make_inputs(2, 256, 3, seed=45)
    _gpu.assert_close(run_ex(cpu, fold_dg=True), ref_ex(cpu, fold_dg=True), TOL, "fold_dg")


def test_fold_dg_with_incoming_and_groups():
    cpu = grouped_inputs(1, 192, 2, 2, seed=46)
    ins = incoming(1, 192, 4, seed=47)
    _gpu.assert_close(run_ex(cpu, fold_dg=True, **ins), ref_ex(cpu, fold_dg=True, **ins), TOL,
                      "fold + accumulate + GVA")


def test_fold_dg_is_the_reverse_cumsum_of_the_plain_dg():
    """Property at full size (the headline workload): folding is a chunk-local suffix sum
    of the unfolded dg, checked on the GPU outputs themselves."""
    cpu = kda_inputs.make_config_inputs(kda_inputs.HEADLINE)
    dev = _gpu.to_device(cpu)
    plain = kda.kda_intra_bwd_ex(*(dev[n] for n in _gpu.ARGS))
    folded = kda.kda_intra_bwd_ex(*(dev[n] for n in _gpu.ARGS), fold_dg=True)
    for a, b in zip(plain[:3], folded[:3]):
        assert torch.equal(a, b)
    B, T, H = 8, 4096, 16
    want = plain[3].double().view(B, T // 64, 64, H, 128).flip(2).cumsum(2).flip(2)
    got = folded[3].double().view(B, T // 64, 64, H, 128)
    err = ((got - want).abs().max() / want.abs().max()).item()
    assert err < 1e-5, err


@pytest.mark.parametrize("qk_dtype", [torch.bfloat16, torch.float16])
def test_io_dtype_outputs_are_the_rounded_fp32_results(qk_dtype):
    cpu = kda_inputs.make_inputs(2, 128, 3, qk_dtype=qk_dtype, seed=48)
    f32 = run_ex(cpu)
    low = run_ex(cpu, dqdk_io_dtype=True)
    assert low[0].dtype == qk_dtype and low[1].dtype == qk_dtype
    assert torch.equal(low[0], f32[0].to(qk_dtype))
    assert torch.equal(low[1], f32[1].to(qk_dtype))
    assert torch.equal(low[2], f32[2]) and torch.equal(low[3], f32[3])


def test_plain_options_match_the_plain_entry_point():
    cpu = kda_inputs.make_inputs(2, 192, 2, seed=49)
    dev = _gpu.to_device(cpu)
    a = kda.kda_intra_bwd(*(dev[n] for n in _gpu.ARGS))
    b = kda.kda_intra_bwd_ex(*(dev[n] for n in _gpu.ARGS))
    for n, x, y in zip(_gpu.NAMES, a, b):
        assert torch.equal(x, y), n


def test_full_size_all_options():
    """The headline workload with every option on, every element against the oracle."""
    cpu = kda_inputs.make_config_inputs(kda_inputs.HEADLINE)
    ins = incoming(8, 4096, 16, seed=50)
    got = run_ex(cpu, fold_dg=True, **ins)
    ref = ref_ex(cpu, fold_dg=True, **ins)
    _gpu.assert_close(got, ref, TOL, "headline, all options")
