"""The fp64 oracle against pins that do not come from the oracle itself."""

import zlib

import numpy as np
import pytest
import torch

import kda_inputs
import oracle
from tests import _pins


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


CASES = {
    # (B, T, H, K, bt, gate_lo)
    "tiny_two_chunks": (1, 16, 2, 4, 8, -1.0),
    "tiny_two_batches": (2, 8, 1, 3, 8, -0.5),
    "tiny_steep_gate": (1, 8, 1, 4, 8, -8.0),
    "wide_chunk": (1, 64, 1, 8, 16, -1.0),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_pins_tiny(lib, case):
    B, T, H, K, bt, lo = CASES[case]
    inp = _pins.tiny_inputs(B, T, H, K, bt, gate_lo=lo, seed=zlib.crc32(case.encode()) % 1000)
    fails = _pins.run_all(lib, inp, bt, with_fd=(K * T * H * B <= 256))
    assert not fails, "\n".join(fails)


def test_finite_differences_full_width_chunk(lib):
    """FD at the kernel's own chunk geometry (BT=64) on one channel-narrow unit."""
    inp = _pins.tiny_inputs(1, 64, 1, 2, 64, gate_lo=-0.5, seed=5)
    fails = _pins.check_finite_differences(lib, inp, 64)
    assert not fails, "\n".join(fails)


def _quantised_config0():
    x = kda_inputs.make_config_inputs(0)
    return {n: v.to(torch.float64).numpy() for n, v in x.items()}


def test_config0_against_autograd(lib):
    """The single-chunk workload (bf16 q/k, K=128, BT=64) against torch autograd."""
    inp = _quantised_config0()
    fails = _pins.check_autograd_backward(lib, inp, 64, tol=1e-12)
    fails += _pins.check_separable_forward(lib, inp, 64)
    fails += _pins.check_masks(lib, inp, 64)
    fails += _pins.check_dbeta_identity(lib, inp, 64)
    fails += _pins.check_euler(lib, inp, 64)
    assert not fails, "\n".join(fails)


def test_gate_stress_unit_against_autograd(lib):
    """Cumulative gates down to about -300 (fp16 q/k): the separable fp64 form still holds."""
    cfg = kda_inputs.CONFIGS[4]
    inp = kda_inputs.make_inputs(1, 128, 2, gate_lo=cfg.gate_lo, qk_dtype=cfg.qk_dtype,
                                 seed=99)
    inp = {n: v.to(torch.float64).numpy() for n, v in inp.items()}
    assert inp["g"].min() < -250.0
    fails = _pins.check_autograd_backward(lib, inp, 64, tol=1e-12)
    assert not fails, "\n".join(fails)


def test_thread_count_does_not_change_results(lib):
    inp = _pins.tiny_inputs(2, 32, 3, 8, 16, seed=11)
    args = [inp[n] for n in ("q", "k", "g", "beta", "dAqk", "dAkk")]
    one = oracle.intra_bwd(*args, bt=16, nthreads=1, lib=lib)
    many = oracle.intra_bwd(*args, bt=16, nthreads=4, lib=lib)
    for a, b in zip(one, many):
        assert np.array_equal(a, b)


def test_rejects_bad_shapes(lib):
    inp = _pins.tiny_inputs(1, 16, 1, 4, 8)
    args = [inp[n] for n in ("q", "k", "g", "beta", "dAqk", "dAkk")]
    with pytest.raises(ValueError):
        oracle.intra_bwd(*args, bt=5, lib=lib)  # T % bt != 0
