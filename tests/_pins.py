"""Checks that pin the fp64 oracle to something other than itself.

Each check takes an oracle library handle (``oracle.load()`` or a deliberately
mutated build) and returns a list of failure strings (empty = pass).  They are
used twice: by test_oracle_pins.py on the real oracle, and by
test_oracle_mutants.py on oracle builds with a planted mistake, which must each
trip at least one check.

What pins what:
  * separable forward  -- Aqk/Akk equal the masked product (q*2^g)(k*2^-g)^T
                          computed by a library matmul (an identity of exp2).
  * autograd backward  -- torch fp64 autograd of that separable forward gives a
                          second, independent dq/dk/dbeta/dg.
  * finite differences -- central differences of L = sum dAqk*Aqk + sum dAkk*Akk.
  * gate-free form     -- g == 0 reduces everything to masked matmuls.
  * masks, dbeta identity, gate-shift invariance, Euler identities, linearity.
"""

from __future__ import annotations

import math

import numpy as np
import torch

import oracle

LN2 = math.log(2.0)


def tiny_inputs(B=1, T=16, H=2, K=4, bt=8, gate_lo=-1.0, seed=0):
    """fp64 inputs for tiny problems (no quantisation: the oracle is exact in fp64)."""
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, T, H, K))
    k = rng.standard_normal((B, T, H, K))
    step = rng.uniform(gate_lo, 0.0, (B, T, H, K))
    g = step.reshape(B, T // bt, bt, H, K).cumsum(axis=2).reshape(B, T, H, K)
    beta = rng.uniform(0.0, 1.0, (B, T, H))
    r = np.arange(bt)[:, None]
    s = np.arange(bt)[None, :]
    lower = (s <= r).astype(np.float64)
    strict = (s < r).astype(np.float64)
    nt = T // bt
    dAqk = (rng.standard_normal((B, nt, bt, H, bt)) * lower[None, None, :, None, :]
            ).reshape(B, T, H, bt)
    dAkk = (rng.standard_normal((B, nt, bt, H, bt)) * strict[None, None, :, None, :]
            ).reshape(B, T, H, bt)
    return dict(q=q, k=k, g=g, beta=beta, dAqk=dAqk, dAkk=dAkk)


def _units(x, bt):
    """[B, T, H, X] -> [B, H, NT, bt, X] (torch view helper)."""
    B, T, H = x.shape[:3]
    rest = x.shape[3:]
    x = x.reshape(B, T // bt, bt, H, *rest)
    if rest:
        return x.permute(0, 3, 1, 2, 4)
    return x.permute(0, 3, 1, 2)


def separable_forward(inp, bt):
    """Aqk, Akk via (q*2^g)(k*2^-g)^T with library matmuls, fp64 torch."""
    t = {n: torch.as_tensor(np.asarray(v, dtype=np.float64)) for n, v in inp.items()}
    return _separable(t, bt)


def _separable(t, bt):
    q, k, g, beta = (_units(t[n], bt) for n in ("q", "k", "g", "beta"))
    lower = torch.tril(torch.ones(bt, bt, dtype=torch.float64))
    strict = torch.tril(torch.ones(bt, bt, dtype=torch.float64), -1)
    up = torch.exp2(g)
    dn = torch.exp2(-g)
    Aqk = ((q * up) @ (k * dn).transpose(-1, -2)) * lower
    Akk = beta.unsqueeze(-1) * ((k * up) @ (k * dn).transpose(-1, -2)) * strict
    return Aqk, Akk


def _to_btx(a, B, T, H):
    """[B, H, NT, bt, X] -> [B, T, H, X] numpy."""
    a = a.permute(0, 2, 3, 1, *range(4, a.dim())).reshape(B, T, H, *a.shape[4:])
    return a.detach().numpy()


def autograd_backward(inp, bt):
    """dq, dk, db, dg from torch fp64 autograd of the separable forward."""
    t = {n: torch.tensor(np.asarray(v, dtype=np.float64), requires_grad=True)
         for n, v in inp.items() if n in ("q", "k", "g", "beta")}
    Aqk, Akk = _separable(t, bt)
    dAqk = _units(torch.as_tensor(np.asarray(inp["dAqk"], dtype=np.float64)), bt)
    dAkk = _units(torch.as_tensor(np.asarray(inp["dAkk"], dtype=np.float64)), bt)
    L = (dAqk * Aqk).sum() + (dAkk * Akk).sum()
    L.backward()
    return (t["q"].grad.numpy(), t["k"].grad.numpy(), t["beta"].grad.numpy(),
            t["g"].grad.numpy())


def ragged_autograd_backward(inp, cu_seqlens, bt):
    """dq, dk, db, dg of packed variable-length sequences (B == 1) from torch fp64
    autograd of the separable forward written per chunk over its valid rows only:
    chunks start at each sequence start, the last one of a sequence may be short.
    No padding and nothing shared with the oracle's composition."""
    t = {n: torch.tensor(np.asarray(v, dtype=np.float64), requires_grad=True)
         for n, v in inp.items() if n in ("q", "k", "g", "beta")}
    dAqk = torch.as_tensor(np.asarray(inp["dAqk"], dtype=np.float64))
    dAkk = torch.as_tensor(np.asarray(inp["dAkk"], dtype=np.float64))
    cu = [int(v) for v in np.asarray(cu_seqlens).reshape(-1)]
    L = torch.zeros((), dtype=torch.float64)
    for a, b in zip(cu[:-1], cu[1:]):
        for c0 in range(a, b, bt):
            m = min(c0 + bt, b) - c0
            sl = slice(c0, c0 + m)
            q, k, g = (t[n][0, sl].transpose(0, 1) for n in ("q", "k", "g"))  # [H, m, K]
            beta = t["beta"][0, sl].transpose(0, 1)                             # [H, m]
            lower = torch.tril(torch.ones(m, m, dtype=torch.float64))
            strict = torch.tril(torch.ones(m, m, dtype=torch.float64), -1)
            up, dn = torch.exp2(g), torch.exp2(-g)
            Aqk = ((q * up) @ (k * dn).transpose(-1, -2)) * lower
            Akk = beta.unsqueeze(-1) * ((k * up) @ (k * dn).transpose(-1, -2)) * strict
            gq = dAqk[0, sl, :, :m].transpose(0, 1)  # [H, m, m]
            gk = dAkk[0, sl, :, :m].transpose(0, 1)
            L = L + (gq * Aqk).sum() + (gk * Akk).sum()
    L.backward()
    return (t["q"].grad.numpy(), t["k"].grad.numpy(), t["beta"].grad.numpy(),
            t["g"].grad.numpy())


def ragged_separable_forward(inp, cu_seqlens, bt):
    """Aqk, Akk of packed variable-length sequences (B == 1) as [1, T, H, bt] arrays:
    per chunk, over its valid rows only, (q 2^g)(k 2^-g)^T masked, in torch fp64;
    rows outside every sequence are NaN."""
    t = {n: torch.as_tensor(np.asarray(v, dtype=np.float64)) for n, v in inp.items()}
    T, H = t["g"].shape[1], t["g"].shape[2]
    Aqk = torch.full((1, T, H, bt), float("nan"), dtype=torch.float64)
    Akk = torch.full((1, T, H, bt), float("nan"), dtype=torch.float64)
    cu = [int(v) for v in np.asarray(cu_seqlens).reshape(-1)]
    for a, b in zip(cu[:-1], cu[1:]):
        for c0 in range(a, b, bt):
            m = min(c0 + bt, b) - c0
            sl = slice(c0, c0 + m)
            q, k, g = (t[n][0, sl].transpose(0, 1) for n in ("q", "k", "g"))
            beta = t["beta"][0, sl].transpose(0, 1)
            lower = torch.tril(torch.ones(m, m, dtype=torch.float64))
            strict = torch.tril(torch.ones(m, m, dtype=torch.float64), -1)
            up, dn = torch.exp2(g), torch.exp2(-g)
            aq = ((q * up) @ (k * dn).transpose(-1, -2)) * lower
            ak = beta.unsqueeze(-1) * ((k * up) @ (k * dn).transpose(-1, -2)) * strict
            Aqk[0, sl, :, :] = 0.0
            Akk[0, sl, :, :] = 0.0
            Aqk[0, sl, :, :m] = aq.transpose(0, 1)
            Akk[0, sl, :, :m] = ak.transpose(0, 1)
    return Aqk.numpy(), Akk.numpy()


def ragged_reverse_cumsum(x, cu_seqlens, bt):
    """Inclusive reverse cumsum along tokens inside each (possibly short) chunk of
    packed variable-length sequences, by explicit loops over tokens."""
    x = np.asarray(x, dtype=np.float64)
    out = np.array(x)
    cu = [int(v) for v in np.asarray(cu_seqlens).reshape(-1)]
    for a, b in zip(cu[:-1], cu[1:]):
        for c0 in range(a, b, bt):
            c1 = min(c0 + bt, b)
            run = np.zeros(x.shape[2:])
            for tkn in range(c1 - 1, c0 - 1, -1):
                run = run + x[0, tkn]
                out[0, tkn] = run
    return out


def rel_err(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    scale = max(np.max(np.abs(b)), 1e-300)
    return float(np.max(np.abs(a - b)) / scale)


def _cmp(fails, name, got, want, tol):
    e = rel_err(got, want)
    if not np.isfinite(e) or e > tol:
        fails.append(f"{name}: rel err {e:.3e} > {tol:.1e}")


def _loss(lib, inp, bt):
    Aqk, Akk = oracle.intra_fwd(inp["q"], inp["k"], inp["g"], inp["beta"], bt=bt,
                                nthreads=1, lib=lib)
    return float(np.sum(inp["dAqk"] * Aqk) + np.sum(inp["dAkk"] * Akk))


def bwd(lib, inp, bt):
    return oracle.intra_bwd(inp["q"], inp["k"], inp["g"], inp["beta"], inp["dAqk"],
                            inp["dAkk"], bt=bt, nthreads=1, lib=lib)


# ----------------------------------------------------------------------------- checks

def check_separable_forward(lib, inp, bt, tol=1e-12):
    fails = []
    Aqk, Akk = oracle.intra_fwd(inp["q"], inp["k"], inp["g"], inp["beta"], bt=bt,
                                nthreads=1, lib=lib)
    sq, sk = separable_forward(inp, bt)
    B, T, H = inp["beta"].shape
    _cmp(fails, "Aqk vs separable", Aqk, _to_btx(sq, B, T, H), tol)
    _cmp(fails, "Akk vs separable", Akk, _to_btx(sk, B, T, H), tol)
    return fails


def check_autograd_backward(lib, inp, bt, tol=1e-11):
    fails = []
    dq, dk, db, dg = bwd(lib, inp, bt)
    aq, ak, ab, ag = autograd_backward(inp, bt)
    _cmp(fails, "dq vs autograd", dq, aq, tol)
    _cmp(fails, "dk vs autograd", dk, ak, tol)
    _cmp(fails, "db vs autograd", db, ab, tol)
    _cmp(fails, "dg vs autograd", dg, ag, tol)
    return fails


def check_finite_differences(lib, inp, bt, h=1e-6, tol=1e-6):
    """Central differences of the oracle's own forward loss, every input element."""
    fails = []
    inp = {n: np.array(v, dtype=np.float64) for n, v in inp.items()}
    dq, dk, db, dg = bwd(lib, inp, bt)
    grads = {"q": dq, "k": dk, "beta": db, "g": dg}
    for name, grad in grads.items():
        base = inp[name]
        fd = np.zeros_like(base)
        flat = base.reshape(-1)
        for idx in range(flat.size):
            old = flat[idx]
            flat[idx] = old + h
            lp = _loss(lib, inp, bt)
            flat[idx] = old - h
            lm = _loss(lib, inp, bt)
            flat[idx] = old
            fd.reshape(-1)[idx] = (lp - lm) / (2 * h)
        _cmp(fails, f"d{name} vs finite differences", grad, fd, tol)
    return fails


def check_gate_free_closed_form(lib, inp, bt, tol=1e-12):
    """g == 0: every output is a masked matmul (numpy, per unit)."""
    fails = []
    inp = dict(inp)
    inp["g"] = np.zeros_like(inp["g"])
    dq, dk, db, dg = bwd(lib, inp, bt)
    B, T, H, K = inp["q"].shape
    lower = np.tril(np.ones((bt, bt)))
    strict = np.tril(np.ones((bt, bt)), -1)
    want = {n: np.zeros_like(v) for n, v in (("dq", dq), ("dk", dk), ("db", db),
                                             ("dg", dg))}
    for b in range(B):
        for h in range(H):
            for c in range(T // bt):
                sl = slice(c * bt, (c + 1) * bt)
                q = inp["q"][b, sl, h]
                k = inp["k"][b, sl, h]
                be = inp["beta"][b, sl, h]
                Pq = inp["dAqk"][b, sl, h] * lower
                Pk = inp["dAkk"][b, sl, h] * strict
                Pkb = be[:, None] * Pk  # dL/dS for S = k k^T on the Akk term
                want["dq"][b, sl, h] = Pq @ k
                want["dk"][b, sl, h] = Pq.T @ q + Pkb @ k + Pkb.T @ k
                want["db"][b, sl, h] = np.sum(Pk * (k @ k.T), axis=1)
                want["dg"][b, sl, h] = LN2 * (q * (Pq @ k) - k * (Pq.T @ q)
                                              + k * (Pkb @ k) - k * (Pkb.T @ k))
    for n, got in (("dq", dq), ("dk", dk), ("db", db), ("dg", dg)):
        _cmp(fails, f"{n} vs gate-free closed form", got, want[n], tol)
    return fails


def check_masks(lib, inp, bt, tol=0.0):
    """Entries outside the support change nothing; first-row special cases."""
    fails = []
    base = bwd(lib, inp, bt)
    poisoned = dict(inp)
    r = np.arange(bt)[:, None]
    s = np.arange(bt)[None, :]
    B, T, H, _ = inp["q"].shape
    upper_q = np.tile((s > r), (T // bt, 1))[None, :, None, :]
    upper_k = np.tile((s >= r), (T // bt, 1))[None, :, None, :]
    poisoned["dAqk"] = np.where(upper_q, 1e6, inp["dAqk"])
    poisoned["dAkk"] = np.where(upper_k, -1e6, inp["dAkk"])
    got = bwd(lib, poisoned, bt)
    for n, a, b in zip(("dq", "dk", "db", "dg"), got, base):
        if not np.array_equal(a, b):
            fails.append(f"{n} changed when out-of-support dA entries were poisoned")
    dq, dk, db, dg = base
    for c in range(T // bt):
        row = c * bt
        want_dq0 = inp["dAqk"][:, row, :, 0:1] * inp["k"][:, row]
        _cmp(fails, "dq at chunk row 0", dq[:, row], want_dq0, 1e-15)
        if np.any(db[:, row] != 0.0):
            fails.append("db at chunk row 0 is not exactly 0")
    return fails


def check_dbeta_identity(lib, inp, bt, tol=1e-12):
    fails = []
    dq, dk, db, dg = bwd(lib, inp, bt)
    Aqk, Akk = oracle.intra_fwd(inp["q"], inp["k"], inp["g"], inp["beta"], bt=bt,
                                nthreads=1, lib=lib)
    want = np.sum(inp["dAkk"] * Akk, axis=-1) / inp["beta"]
    _cmp(fails, "db vs sum_s dAkk*Akk/beta", db, want, tol)
    return fails


def check_gate_shift(lib, inp, bt, tol=1e-10):
    """A per-(chunk, channel) constant added to g changes no output; sum_t dg = 0."""
    fails = []
    base = bwd(lib, inp, bt)
    B, T, H, K = inp["g"].shape
    rng = np.random.default_rng(123)
    shift = rng.uniform(-3.0, 3.0, (B, T // bt, 1, H, K))
    shifted = dict(inp)
    shifted["g"] = (inp["g"].reshape(B, T // bt, bt, H, K) + shift).reshape(B, T, H, K)
    got = bwd(lib, shifted, bt)
    for n, a, b in zip(("dq", "dk", "db", "dg"), got, base):
        _cmp(fails, f"{n} under a chunk-constant gate shift", a, b, tol)
    dg = base[3].reshape(B, T // bt, bt, H, K)
    colsum = np.abs(dg.sum(axis=2)).max()
    if colsum > 1e-12 * max(np.abs(dg).max(), 1e-300) * bt:
        fails.append(f"sum_t dg[t, d] over a chunk is {colsum:.3e}, not 0")
    return fails


def check_euler(lib, inp, bt, tol=1e-11):
    """Degree-1/2 homogeneity identities, per unit."""
    fails = []
    dq, dk, db, dg = bwd(lib, inp, bt)
    Aqk, Akk = oracle.intra_fwd(inp["q"], inp["k"], inp["g"], inp["beta"], bt=bt,
                                nthreads=1, lib=lib)
    B, T, H, K = inp["q"].shape
    nt = T // bt

    def per_unit(x):  # [B, T, H, ...] -> sum over chunk rows and trailing dims
        x = x.reshape(B, nt, bt, H, -1)
        return x.sum(axis=(2, 4))

    Lq = per_unit(inp["dAqk"] * Aqk)
    Lk = per_unit(inp["dAkk"] * Akk)
    _cmp(fails, "sum q*dq = sum dAqk*Aqk", per_unit(inp["q"] * dq), Lq, tol)
    _cmp(fails, "sum beta*db = sum dAkk*Akk", per_unit(inp["beta"][..., None] * db[..., None]),
         Lk, tol)
    _cmp(fails, "sum k*dk = Lq + 2 Lk", per_unit(inp["k"] * dk), Lq + 2 * Lk, tol)
    # sum_d dg[t, d] = ln2 * (row sum - column sum) of W = dAqk*Aqk + dAkk*Akk
    W = (inp["dAqk"] * Aqk + inp["dAkk"] * Akk).reshape(B, nt, bt, H, bt)
    rows = W.sum(axis=4)                                   # [B, nt, bt(r), H]
    cols = W.sum(axis=2).transpose(0, 1, 3, 2)             # [B, nt, bt(s), H]
    want = (LN2 * (rows - cols)).reshape(B, T, H)
    _cmp(fails, "sum_d dg = ln2 (rowsum - colsum)", dg.sum(axis=-1), want, tol)
    return fails


def check_linearity(lib, inp, bt, tol=1e-12):
    fails = []
    a = bwd(lib, inp, bt)
    only_q = dict(inp, dAkk=np.zeros_like(inp["dAkk"]))
    only_k = dict(inp, dAqk=np.zeros_like(inp["dAqk"]))
    bq = bwd(lib, only_q, bt)
    bk = bwd(lib, only_k, bt)
    for n, x, y, z in zip(("dq", "dk", "db", "dg"), a, bq, bk):
        _cmp(fails, f"{n} linear in (dAqk, dAkk)", x, y + z, tol)
    if np.any(bq[2] != 0.0):
        fails.append("db is not exactly 0 when dAkk == 0")
    if np.any(bk[0] != 0.0):
        fails.append("dq is not exactly 0 when dAqk == 0")
    return fails


def check_unit_permutation(lib, inp, bt):
    """Swapping two heads swaps the outputs exactly (units are independent)."""
    fails = []
    B, T, H, K = inp["q"].shape
    if H < 2:
        return fails
    perm = np.arange(H)[::-1].copy()
    sw = {n: v[:, :, perm] for n, v in inp.items()}
    a = bwd(lib, inp, bt)
    b = bwd(lib, sw, bt)
    for n, x, y in zip(("dq", "dk", "db", "dg"), a, b):
        if not np.array_equal(x[:, :, perm], y):
            fails.append(f"{n} is not permuted with the heads")
    return fails


ALL_CHECKS = (
    check_separable_forward,
    check_autograd_backward,
    check_gate_free_closed_form,
    check_masks,
    check_dbeta_identity,
    check_gate_shift,
    check_euler,
    check_linearity,
    check_unit_permutation,
)


def run_all(lib, inp, bt, with_fd=True):
    fails = []
    for chk in ALL_CHECKS:
        fails += chk(lib, inp, bt)
    if with_fd:
        fails += check_finite_differences(lib, inp, bt)
    return fails
