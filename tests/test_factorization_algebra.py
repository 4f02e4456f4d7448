"""The factorizations the GPU kernels use, restated in fp64 numpy and checked against the
oracle's direct sums (CPU only; no GPU code is shared or called).

Per unit (64-token chunk, rows r, s, channels d, E[r,s,d] = 2^(g[r,d] - g[s,d])), the
backward needs the row-side sums accq, acck and the column-side sum dkt.  The kernels
evaluate them in three ways (bwd_intra page, module docstring and diagonal-block section):

* cross sub-block terms, target block t and source block j < t, through the block
  boundaries: E[r,s] = 2^(g_r - g_16t) * 2^(g_16t - g_s) on the row side (the middle
  factor folded into the operand A_t), and 2^(g_e(i) - g_s) * 2^(g_16j - g_e(i)) *
  2^(g_r - g_16j) on the column side, e(i) = 16(i + 1);
* the 16x16 diagonal blocks pair by pair, one exp2 per (r, s, d);
* with factor_diag, each diagonal block's lower-left 8x8 quadrant through the block's
  row 8: E[r,s] = 2^(g_r - g_8) * 2^(g_8 - g_s).

Every exponent any of them evaluates must be <= 0, so nothing can overflow; the test
records them all and checks that too.
"""

import math

import numpy as np
import pytest

import kda_inputs
import oracle

BT, BC, NB = 64, 16, 4


class Exps:
    """Collects the largest exponent passed to exp2."""

    def __init__(self):
        self.max = -math.inf

    def __call__(self, x):
        x = np.asarray(x, dtype=np.float64)
        if x.size:
            self.max = max(self.max, float(x.max()))
        return np.exp2(x)


def restated_sums(q, k, g, beta, daq, dak, factor_diag: bool, exp2: Exps):
    """accq, acck [64, K] and dkt [64, K] of one unit the way the kernels evaluate them."""
    K = q.shape[1]
    accq = np.zeros((BT, K))
    acck = np.zeros((BT, K))
    dkt = np.zeros((BT, K))
    # row side, cross: A_t[s, d] = k_s 2^(g_16t - g_s), X_t[n, d] = sum_s dA[16t+n, s] A_t
    for t in range(1, NB):
        b0 = BC * t
        A = k[:b0] * exp2(g[b0] - g[:b0])                       # [16t, K]
        post = exp2(g[b0:b0 + BC] - g[b0])                       # [16, K]
        accq[b0:b0 + BC] += post * (daq[b0:b0 + BC, :b0] @ A)
        acck[b0:b0 + BC] += post * (dak[b0:b0 + BC, :b0] @ A)
    # column side, cross: P_j[s, d] = sum_{r in blk j} (q_r dAqk[r,s] + beta_r k_r dAkk[r,s])
    # 2^(g_r - g_16j); dkt[s] = 2^(g_e(i) - g_s) sum_{j>i} 2^(g_16j - g_e(i)) P_j[s]
    for i in range(NB - 1):
        s0, e = BC * i, BC * (i + 1)
        tot = np.zeros((BC, K))
        for j in range(i + 1, NB):
            r0 = BC * j
            f = exp2(g[r0:r0 + BC] - g[r0])                      # [16, K]
            qa = q[r0:r0 + BC] * f
            ka = (beta[r0:r0 + BC, None] * k[r0:r0 + BC]) * f
            P = daq[r0:r0 + BC, s0:e].T @ qa + dak[r0:r0 + BC, s0:e].T @ ka
            tot += exp2(g[r0] - g[e]) * P
        dkt[s0:e] += exp2(g[e] - g[s0:e]) * tot
    # diagonal blocks
    for i in range(NB):
        b = BC * i
        for rr in range(BC):
            r = b + rr
            for ss in range(rr + 1):
                s = b + ss
                if factor_diag and rr >= BC // 2 and ss < BC // 2:
                    m = b + BC // 2
                    E = exp2(g[r] - g[m]) * exp2(g[m] - g[s])
                else:
                    E = exp2(g[r] - g[s])
                accq[r] += daq[r, s] * k[s] * E
                dkt[s] += daq[r, s] * q[r] * E
                if ss < rr:
                    acck[r] += dak[r, s] * k[s] * E
                    dkt[s] += dak[r, s] * beta[r] * k[r] * E
    return accq, acck, dkt


def outputs_from_sums(q, k, beta, accq, acck, dkt):
    """The epilogue: dq, dk, db, dg from the three sums (dg in log2-gate units)."""
    dq = accq
    dk = beta[:, None] * acck + dkt
    db = (acck * k).sum(axis=1)
    dg = math.log(2.0) * (q * accq + (beta[:, None] * acck - dkt) * k)
    return dq, dk, db, dg


@pytest.mark.parametrize("factor_diag", [False, True])
@pytest.mark.parametrize("gate_lo,seed", [(-0.5, 150), (-8.0, 151), (-40.0, 152)])
def test_factorized_sums_equal_the_direct_sums(factor_diag, gate_lo, seed):
    inp = kda_inputs.make_inputs(1, 2 * BT, 1, gate_lo=gate_lo, seed=seed, k_dim=16)
    arr = {n: v.double().numpy() for n, v in inp.items()}
    ref = oracle.intra_bwd(*(inp[n] for n in ("q", "k", "g", "beta", "dAqk", "dAkk")))
    for c in range(2):
        rows = slice(c * BT, (c + 1) * BT)
        q, k, g = (arr[n][0, rows, 0] for n in ("q", "k", "g"))
        beta = arr["beta"][0, rows, 0]
        daq, dak = arr["dAqk"][0, rows, 0], arr["dAkk"][0, rows, 0]
        exp2 = Exps()
        sums = restated_sums(q, k, g, beta, daq, dak, factor_diag, exp2)
        assert exp2.max <= 0.0, f"an exponent above zero: {exp2.max}"
        got = outputs_from_sums(q, k, beta, *sums)
        for name, a, r in zip(("dq", "dk", "db", "dg"), got, ref):
            want = np.asarray(r)[0, rows, 0]
            scale = max(np.abs(want).max(), 1e-300)
            assert np.abs(a - want).max() <= 1e-12 * scale, (name, c)


def test_quadrant_through_a_block_start_would_overflow():
    """The reason the quadrant goes through row 8 and not through the block's first row:
    with steep gates the first-row split needs 2^(g_0 - g_s) with a positive exponent
    that leaves the fp32 range, while both row-8 factors stay <= 1."""
    inp = kda_inputs.make_inputs(1, BT, 1, gate_lo=-40.0, seed=153, k_dim=8)
    g = inp["g"][0, :, 0].double().numpy()
    # 2^(g_0 - g_s) for the block's sources: positive exponents, past fp32's range
    with np.errstate(over="ignore"):
        assert np.isinf(np.exp2((g[0] - g[1:16]).astype(np.float32)).max())
    # the row-8 split: 2^(g_r - g_8) for r in 8..15 and 2^(g_8 - g_s) for s in 0..7
    assert (g[8:16] - g[8]).max() <= 0 and (g[8] - g[:8]).max() <= 0
