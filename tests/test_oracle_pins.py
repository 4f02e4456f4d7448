"""The fp64 oracle against pins that do not come from the oracle itself."""

import zlib

import numpy as np
import pytest
import torch

import kda_inputs
import oracle
from tests import _pins


_ARGS = ("q", "k", "g", "beta", "dAqk", "dAkk")


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
    x = kda_inputs.make_config_inputs(kda_inputs.SINGLE_CHUNK)
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
    cfg = kda_inputs.CONFIGS[kda_inputs.GATE_STRESS]
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


# ---------------------------------------------------------------- extended contract

def test_chunk_reverse_cumsum_pins():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((2, 24, 3, 5))
    y = oracle.chunk_reverse_cumsum(x, bt=8)
    for c in range(3):
        sl = slice(8 * c, 8 * c + 8)
        xc, yc = x[:, sl], y[:, sl]
        assert np.allclose(yc[:, -1], xc[:, -1], rtol=0, atol=0)          # last row
        assert np.allclose(yc[:, :-1] - yc[:, 1:], xc[:, :-1], atol=1e-14)  # differences
        assert np.allclose(yc[:, 0], xc.sum(axis=1), atol=1e-13)           # first row


def test_grouped_heads_pinned_by_finite_differences():
    """With q/k shared by G value heads, the sum of the per-value-head dq (dk) over a
    group is dL/d(shared q) (dk), by central differences of the summed loss."""
    B, T, H, G, K, bt = 1, 16, 1, 3, 3, 8
    rng = np.random.default_rng(17)
    base = _pins.tiny_inputs(B, T, H * G, K, bt, seed=17)
    q = rng.standard_normal((B, T, H, K))
    k = rng.standard_normal((B, T, H, K))
    lib = oracle.load()

    def loss(qq, kk):
        qx, kx = np.repeat(qq, G, axis=2), np.repeat(kk, G, axis=2)
        Aqk, Akk = oracle.intra_fwd(qx, kx, base["g"], base["beta"], bt=bt, lib=lib)
        return float(np.sum(base["dAqk"] * Aqk) + np.sum(base["dAkk"] * Akk))

    dq, dk, _, _ = oracle.intra_bwd_ex(q, k, base["g"], base["beta"], base["dAqk"],
                                       base["dAkk"], bt=bt, lib=lib)
    for name, x, grad in (("q", q, dq), ("k", k, dk)):
        shared = grad.reshape(B, T, H, G, K).sum(axis=3)
        fd = np.zeros_like(x)
        h = 1e-6
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + h
            lp = loss(q, k)
            x[idx] = old - h
            lm = loss(q, k)
            x[idx] = old
            fd[idx] = (lp - lm) / (2 * h)
        assert _pins.rel_err(shared, fd) < 1e-6, name


def test_grouped_heads_with_one_group_is_the_plain_backward():
    inp = _pins.tiny_inputs(1, 16, 2, 4, 8, seed=21)
    a = oracle.intra_bwd(*(inp[n] for n in ("q", "k", "g", "beta", "dAqk", "dAkk")), bt=8)
    b = oracle.intra_bwd_ex(*(inp[n] for n in ("q", "k", "g", "beta", "dAqk", "dAkk")), bt=8)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


# ------------------------------------------------------------ variable-length sequences

VARLEN_LENS = [3, 8, 11, 1, 16, 5, 9]  # chunks of 8: short, whole, ragged, single row


def _varlen_tiny(H=2, K=4, bt=8, seed=11, lens=VARLEN_LENS, gate_lo=-1.0, HQ=None):
    x, cu = kda_inputs.make_varlen_inputs(lens, H, gate_lo=gate_lo, qk_dtype=torch.float32,
                                          seed=seed, k_dim=K, bt=bt, HQ=HQ)
    return {n: v.double().numpy() for n, v in x.items()}, cu.numpy()


def test_varlen_against_ragged_autograd(lib):
    """Short and ragged chunks against autograd of the per-chunk forward on the valid
    rows only (the oracle pads; the pin does not)."""
    inp, cu = _varlen_tiny()
    got = oracle.intra_bwd_varlen(*(inp[n] for n in _ARGS), cu, bt=8, lib=lib)
    want = _pins.ragged_autograd_backward(inp, cu, 8)
    for name, a, b in zip(("dq", "dk", "db", "dg"), got, want):
        assert _pins.rel_err(a, b) < 1e-12, name


def test_varlen_options_against_ragged_autograd(lib):
    """Grouped value heads, incoming gradients and the fold on ragged chunks."""
    inp, cu = _varlen_tiny(H=4, HQ=2, seed=12, gate_lo=-3.0)
    rng = np.random.default_rng(3)
    T = inp["g"].shape[1]
    ins = dict(dq_in=rng.standard_normal((1, T, 4, 4)), dk_in=rng.standard_normal((1, T, 4, 4)),
               dg_in=rng.standard_normal((1, T, 4, 4)), db_in=rng.standard_normal((1, T, 4)))
    got = oracle.intra_bwd_varlen(*(inp[n] for n in _ARGS), cu, fold_dg=True, bt=8, lib=lib,
                                  **ins)
    rep = dict(inp, q=np.repeat(inp["q"], 2, axis=2), k=np.repeat(inp["k"], 2, axis=2))
    dq, dk, db, dg = _pins.ragged_autograd_backward(rep, cu, 8)
    want = (dq + ins["dq_in"], dk + ins["dk_in"], db + ins["db_in"],
            _pins.ragged_reverse_cumsum(dg + ins["dg_in"], cu, 8))
    for name, a, b in zip(("dq", "dk", "db", "dg"), got, want):
        assert _pins.rel_err(a, b) < 1e-12, name


def test_varlen_whole_chunks_equal_the_fixed_length_oracle(lib):
    """Sequences of whole chunks: the packed problem is the fixed-length one."""
    inp, cu = _varlen_tiny(lens=[16, 8, 24], seed=13)
    got = oracle.intra_bwd_varlen(*(inp[n] for n in _ARGS), cu, bt=8, lib=lib)
    want = oracle.intra_bwd(*(inp[n] for n in _ARGS), bt=8, lib=lib)
    for a, b in zip(got, want):
        assert np.array_equal(a, b)


def test_varlen_rows_outside_every_sequence_are_nan(lib):
    inp, _ = _varlen_tiny(lens=[5, 7], seed=14)
    got = oracle.intra_bwd_varlen(*(inp[n] for n in _ARGS), np.array([0, 5, 9]), bt=8, lib=lib)
    assert np.isnan(got[0][0, 9:]).all() and np.isfinite(got[0][0, :9]).all()


def test_forward_varlen_and_groups_against_ragged_separable_forward(lib):
    """The forward's composition (GVA + ragged chunks) against the per-chunk separable
    forward over valid rows only."""
    inp, cu = _varlen_tiny(H=4, HQ=2, seed=15, gate_lo=-2.0)
    got = oracle.intra_fwd_ex(inp["q"], inp["k"], inp["g"], inp["beta"], cu_seqlens=cu, bt=8,
                              lib=lib)
    rep = dict(inp, q=np.repeat(inp["q"], 2, axis=2), k=np.repeat(inp["k"], 2, axis=2))
    want = _pins.ragged_separable_forward(rep, cu, 8)
    for a, b in zip(got, want):
        assert _pins.rel_err(a, b) < 1e-12
