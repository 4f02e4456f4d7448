"""Repeated launches of every path on a workload where each persistent CTA runs many
units, compared bitwise with the first launch.

Every kernel sums in a fixed order, so identical inputs give identical outputs; a
hand-off between warps that went wrong only now and then (a stage refilled too early,
an mbarrier phase confused, an operand read before it was written) would show up as a
launch that differs.  Some launches start while a large matrix product runs on another
stream, so that CTAs start and proceed at different times than in a quiet launch.
"""

import pytest
import torch

import gated_delta_rule_intra_gb300 as kda
import kda_inputs
from tests import _gpu

pytestmark = pytest.mark.gpu

REPEATS = 24
B, T, H = 4, 4096, 8  # 2048 units: about 13 per CTA on 152 SMs


# the same token count cut into sequences whose chunks end mid-way (257 chunks x 8 heads)
SEQLENS = (3635, 461, 2048, 8448, 1792)


@pytest.fixture(scope="module")
def problem():
    dev = _gpu.to_device(kda_inputs.make_inputs(B, T, H, seed=170))
    vin, cu = kda_inputs.make_varlen_inputs(SEQLENS, H, seed=171)
    vdev = _gpu.to_device(vin)
    noise = torch.randn(4096, 4096, device="cuda", dtype=torch.bfloat16)
    yield dev, vdev, cu.cuda(), noise
    del dev, vdev, noise
    torch.cuda.empty_cache()


def _call(path, dev, vdev, cu):
    args = [dev[n] for n in _gpu.ARGS]
    vargs = [vdev[n] for n in _gpu.ARGS]
    if path == "kda_intra_fwd":
        return lambda: kda.kda_intra_fwd(*args[:4])
    if path == "kda_intra_fwd_varlen":
        return lambda: kda.kda_intra_fwd(*vargs[:4], cu_seqlens=cu)
    if path == "factor_diag":
        return lambda: kda.kda_intra_bwd_ex(*args, factor_diag=True)
    if path == "varlen":
        return lambda: kda.kda_intra_bwd_ex(*vargs, cu_seqlens=cu)
    return lambda: _gpu.run(path, dev)


@pytest.mark.parametrize("path", list(_gpu.PATHS) + ["factor_diag", "varlen", "kda_intra_fwd",
                                                     "kda_intra_fwd_varlen"])
def test_repeated_launches_are_bitwise_identical(problem, path):
    dev, vdev, cu, noise = problem
    assert sum(SEQLENS) == B * T
    call = _call(path, dev, vdev, cu)
    first = [x.clone() for x in call()]
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    for n in range(REPEATS):
        if n % 2:
            # a matrix product on another stream, queued just before the launch
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                torch.mm(noise, noise)
        got = call()
        torch.cuda.synchronize()
        for a, b in zip(first, got):
            assert torch.equal(a, b), f"{path}: launch {n + 1} differs from the first"
    for x in first:
        assert torch.isfinite(x).all()
