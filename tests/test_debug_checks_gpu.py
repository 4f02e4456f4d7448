"""Every path through the bounds-checked debug build (libkda_debug.so, compiled with
KDA_DEBUG_CHECKS): no kernel computes a global index outside its buffer and no wait
gives up (the flag word stays 0), and the checks change no result (the outputs equal
the normal build's bitwise)."""

import pytest
import torch

import gated_delta_rule_intra_gb300 as kda
import kda_inputs
from tests import _gpu

pytestmark = pytest.mark.gpu

EDGE_LENS = [1, 63, 64, 65, 127, 128, 129, 200, 7, 300, 2, 511]


def _same_under_checks(call):
    """Run `call` with the normal library, then with the debug build reporting into a
    fresh flag word; compare the outputs bitwise and require a clean flag word."""
    ref = [t.clone() for t in call()]
    word = torch.zeros(1, dtype=torch.int32, device="cuda")
    with kda.use_library(kda.DEBUG_LIB_PATH):
        assert kda.kda_debug_checks()
        kda.kda_debug_set_flags(word)
        try:
            got = [t.clone() for t in call()]
            torch.cuda.synchronize()
        finally:
            kda.kda_debug_set_flags(None)
    assert word.item() == 0, f"debug checks reported flags {word.item():#x}"
    assert len(got) == len(ref)
    for i, (a, b) in enumerate(zip(got, ref)):
        assert torch.equal(a, b) or (a.isnan() == b.isnan()).all() and torch.equal(
            a.nan_to_num(), b.nan_to_num()), f"output {i} differs under the checks"


def _dev(cpu):
    return _gpu.to_device(cpu)


@pytest.mark.parametrize("shape,dtype", [((2, 1024, 4), torch.bfloat16),
                                         ((3, 192, 5), torch.float16),
                                         ((1, 64, 200), torch.bfloat16)])
def test_fast_and_fp32_paths(shape, dtype):
    dev = _dev(kda_inputs.make_inputs(*shape, qk_dtype=dtype, seed=130))
    args = [dev[n] for n in _gpu.ARGS]
    _same_under_checks(lambda: kda.kda_intra_bwd(*args))
    _same_under_checks(lambda: kda.kda_intra_bwd_fp32(*args))
    _same_under_checks(lambda: kda.kda_intra_bwd_ex(*args, factor_diag=True))
    _same_under_checks(lambda: kda.kda_intra_bwd_ex(*args, split_tf32=True))
    _same_under_checks(lambda: kda.kda_intra_fwd(*args[:4]))


def test_headline_workload():
    """8192 units: every CTA of the persistent grid runs many units and both stages."""
    dev = _dev(kda_inputs.make_config_inputs(kda_inputs.HEADLINE))
    args = [dev[n] for n in _gpu.ARGS]
    _same_under_checks(lambda: kda.kda_intra_bwd(*args))
    _same_under_checks(lambda: kda.kda_intra_fwd(*args[:4]))


def test_every_option_together():
    G = 2
    x = kda_inputs.make_inputs(2, 320, 2 * G, seed=131)
    x["q"] = x["q"][:, :, ::G].contiguous()
    x["k"] = x["k"][:, :, ::G].contiguous()
    dev = _dev(x)
    args = [dev[n] for n in _gpu.ARGS]
    gen = torch.Generator().manual_seed(132)
    ins = {n: torch.randn(2, 320, 2 * G, 128, generator=gen).cuda()
           for n in ("dq_in", "dk_in", "dg_in")}
    ins["db_in"] = torch.randn(2, 320, 2 * G, generator=gen).cuda()
    for fd in (False, True):
        _same_under_checks(lambda: kda.kda_intra_bwd_ex(*args, fold_dg=True, factor_diag=fd,
                                                        **ins))
    _same_under_checks(lambda: kda.kda_intra_fwd(*args[:4]))
    plain = _dev(kda_inputs.make_inputs(2, 192, 3, seed=133))
    pargs = [plain[n] for n in _gpu.ARGS]
    _same_under_checks(lambda: kda.kda_intra_bwd_ex(*pargs, dqdk_io_dtype=True))


def test_variable_length():
    cpu, cu = kda_inputs.make_varlen_inputs(EDGE_LENS, 2, seed=134)
    dev = _dev(cpu)
    args = [dev[n] for n in _gpu.ARGS]
    cu_d = cu.cuda()
    T = cpu["g"].shape[1]
    gen = torch.Generator().manual_seed(135)
    ins = {n: torch.randn(1, T, 2, 128, generator=gen).cuda() for n in ("dq_in", "dg_in")}
    for fold in (False, True):
        _same_under_checks(lambda: kda.kda_intra_bwd_ex(*args, cu_seqlens=cu_d,
                                                        fold_dg=fold, **ins))
    _same_under_checks(lambda: kda.kda_intra_bwd_ex(*args, cu_seqlens=cu_d, factor_diag=True))
    _same_under_checks(lambda: kda.kda_intra_fwd(*args[:4], cu_seqlens=cu_d))


def test_variable_length_invalid_entries_and_untouched_rows():
    """Table entries that name no chunk are skipped; rows no entry names keep their
    canary.  The outputs are pre-filled the same way for both builds."""
    cpu, cu = kda_inputs.make_varlen_inputs([100, 64], 1, seed=136)
    dev = _dev(cpu)
    args = [dev[n] for n in _gpu.ARGS]
    bad = torch.tensor([[0, 0], [5, 0], [0, 2], [-1, 0], [1, -3], [1, 0]],
                       dtype=torch.int32).cuda()
    T = cpu["g"].shape[1]

    def bwd():
        outs = [torch.full((1, T, 1, 128), 2.5, device="cuda"),
                torch.full((1, T, 1, 128), 2.5, device="cuda"),
                torch.full((1, T, 1), 2.5, device="cuda"),
                torch.full((1, T, 1, 128), 2.5, device="cuda")]
        return kda.kda_intra_bwd_ex(*args, *outs, cu_seqlens=cu.cuda(), chunk_indices=bad)

    def fwd():
        outs = [torch.full((1, T, 1, 64), 2.5, device="cuda") for _ in range(2)]
        return kda.kda_intra_fwd(*args[:4], *outs, cu_seqlens=cu.cuda(), chunk_indices=bad)

    _same_under_checks(bwd)
    _same_under_checks(fwd)


def test_host_entry_point():
    cpu = kda_inputs.make_inputs(2, 256, 3, seed=137)
    host = {n: v.pin_memory() for n, v in cpu.items()}
    ws = torch.empty(kda.kda_intra_bwd_host_workspace_bytes(2, 256, 3, torch.bfloat16),
                     dtype=torch.uint8, device="cuda")

    def call():
        outs = [torch.empty(2, 256, 3, 128).pin_memory(), torch.empty(2, 256, 3, 128).pin_memory(),
                torch.empty(2, 256, 3).pin_memory(), torch.empty(2, 256, 3, 128).pin_memory()]
        kda.kda_intra_bwd_host(*(host[n] for n in _gpu.ARGS), *outs, workspace=ws)
        torch.cuda.synchronize()
        return outs

    _same_under_checks(call)
