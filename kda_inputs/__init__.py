"""Seeded synthetic inputs for the KDA intra-chunk backward.

This module is shared by the tests, the benchmark and the fp64 oracle's callers.
It holds the input recipe only -- distributions, shapes, masks, the chunk-local
gate cumsum that defines the ``g`` input -- and none of the backward's arithmetic.

Recipe (one "unit" = one (batch, head, 64-token chunk)):

* q, k  : N(0, 1) per element, each (b, t, h) row L2-normalised over the head
          dimension in fp32, then rounded to the io dtype (bf16 or fp16).
* gate  : per-step log2 gate, fp32, uniform in (gate_lo, 0].
* g     : inclusive cumulative sum of the per-step gate inside each 64-token
          chunk, restarted at every chunk boundary, in fp32 (the chunk-local
          cumsum that the bwd_intra page's host wrapper receives as ``g``).
* beta  : fp32 uniform in [0, 1).
* dAqk  : fp32 N(0, 1), lower-triangular inside each chunk *including* the
          diagonal (row = token, column = in-chunk source index), zero elsewhere.
* dAkk  : fp32 N(0, 1), strictly lower-triangular inside each chunk, zero elsewhere.

All draws come from one ``torch.Generator`` on the CPU seeded with ``seed``; the
order of draws is fixed, so a (config, seed) pair always yields the same tensors
on a given torch build.
"""

from __future__ import annotations

import dataclasses

import torch

BT = 64
K = 128
SEED0 = 20261202


@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    B: int
    T: int
    H: int
    gate_lo: float
    qk_dtype: torch.dtype = torch.bfloat16

    @property
    def units(self) -> int:
        return self.B * self.H * (self.T // BT)

    @property
    def tokens_heads(self) -> int:
        return self.B * self.T * self.H


# The five workloads: a single chunk, a small multi-chunk case, the headline
# B=8,T=4096,H=16 throughput case, a long sequence and the gate-magnitude stress.
CONFIGS = (
    Config("single_chunk_B1_T64_H1", 1, 64, 1, -0.5),
    Config("small_B2_T1024_H4", 2, 1024, 4, -0.5),
    Config("headline_B8_T4096_H16", 8, 4096, 16, -0.5),
    Config("long_B1_T32768_H32", 1, 32768, 32, -1.0),
    Config("gate_stress_B4_T8192_H64_fp16", 4, 8192, 64, -8.0, torch.float16),
)
# their positions in CONFIGS (each one's seed is SEED0 + its position)
SINGLE_CHUNK, SMALL, HEADLINE, LONG, GATE_STRESS = range(len(CONFIGS))


def chunk_masks(bt: int = BT):
    """Boolean [bt, bt] masks: (lower incl. diagonal, strictly lower)."""
    r = torch.arange(bt).view(bt, 1)
    s = torch.arange(bt).view(1, bt)
    return s <= r, s < r


def make_inputs(B: int, T: int, H: int, *, gate_lo: float = -0.5,
                qk_dtype: torch.dtype = torch.bfloat16, seed: int = SEED0,
                k_dim: int = K, bt: int = BT) -> dict:
    """Draw one seeded input set in the [B, T, H, *] layout (CPU tensors)."""
    if T % bt:
        raise ValueError(f"T={T} is not a multiple of the chunk size {bt}")
    gen = torch.Generator().manual_seed(int(seed))
    f32 = torch.float32

    def unit_rows(x):
        return (x / x.norm(dim=-1, keepdim=True)).to(qk_dtype)

    q = unit_rows(torch.randn(B, T, H, k_dim, generator=gen, dtype=f32))
    k = unit_rows(torch.randn(B, T, H, k_dim, generator=gen, dtype=f32))
    step = torch.rand(B, T, H, k_dim, generator=gen, dtype=f32) * gate_lo
    g = (step.view(B, T // bt, bt, H, k_dim).cumsum(dim=2, dtype=f32)
         .view(B, T, H, k_dim).contiguous())
    beta = torch.rand(B, T, H, generator=gen, dtype=f32)
    lower, strict = chunk_masks(bt)
    nchunk = T // bt

    def masked_grad(mask):
        a = torch.randn(B, nchunk, bt, H, bt, generator=gen, dtype=f32)
        a = a * mask.view(1, 1, bt, 1, bt).to(f32)
        return a.view(B, T, H, bt).contiguous()

    dAqk = masked_grad(lower)
    dAkk = masked_grad(strict)
    return dict(q=q, k=k, g=g, beta=beta, dAqk=dAqk, dAkk=dAkk)


def varlen_seqlens(total: int, *, seed: int = SEED0, min_len: int = 1,
                   max_len: int = 8192) -> list:
    """A seeded mix of sequence lengths summing to exactly ``total``: lengths drawn
    log-uniformly in [min_len, max_len] (many short sequences, most tokens in long
    ones), the last one cut to fit."""
    gen = torch.Generator().manual_seed(int(seed))
    lo, hi = torch.log(torch.tensor(float(min_len))), torch.log(torch.tensor(float(max_len)))
    out, left = [], int(total)
    while left > 0:
        u = torch.rand((), generator=gen)
        n = int(torch.exp(lo + (hi - lo) * u).round().clamp(min_len, max_len))
        n = min(n, left)
        out.append(n)
        left -= n
    return out


def make_varlen_inputs(seqlens, H: int, *, gate_lo: float = -0.5,
                       qk_dtype: torch.dtype = torch.bfloat16, seed: int = SEED0,
                       k_dim: int = K, bt: int = BT, HQ: int | None = None):
    """Packed variable-length inputs: B = 1, T = sum(seqlens), sequence n at tokens
    [cu[n], cu[n+1]).  Same distributions as make_inputs; the gate cumsum and the dA
    triangles restart at every chunk of every sequence (chunks start at the sequence
    start, the last one may be short).  q and k get HQ heads (default H).
    Returns (inputs, cu_seqlens) with cu_seqlens an int32 CPU tensor."""
    lens = [int(n) for n in seqlens]
    if any(n < 0 for n in lens):
        raise ValueError("sequence lengths must be >= 0")
    T = sum(lens)
    HQ = H if HQ is None else HQ
    gen = torch.Generator().manual_seed(int(seed))
    f32 = torch.float32

    def unit_rows(x):
        return (x / x.norm(dim=-1, keepdim=True)).to(qk_dtype)

    q = unit_rows(torch.randn(1, T, HQ, k_dim, generator=gen, dtype=f32))
    k = unit_rows(torch.randn(1, T, HQ, k_dim, generator=gen, dtype=f32))
    step = torch.rand(1, T, H, k_dim, generator=gen, dtype=f32) * gate_lo
    beta = torch.rand(1, T, H, generator=gen, dtype=f32)
    cu = torch.tensor([0] + lens, dtype=torch.int64).cumsum(0)
    # in-chunk position of every token
    pos = torch.empty(T, dtype=torch.int64)
    g = torch.empty(1, T, H, k_dim, dtype=f32)
    for a, b in zip(cu[:-1].tolist(), cu[1:].tolist()):
        for c0 in range(a, b, bt):
            c1 = min(c0 + bt, b)
            pos[c0:c1] = torch.arange(c1 - c0)
            g[:, c0:c1] = step[:, c0:c1].cumsum(dim=1, dtype=f32)
    cols = torch.arange(bt).view(1, bt)
    lower = (cols <= pos.view(T, 1)).to(f32).view(1, T, 1, bt)
    strict = (cols < pos.view(T, 1)).to(f32).view(1, T, 1, bt)
    dAqk = (torch.randn(1, T, H, bt, generator=gen, dtype=f32) * lower).contiguous()
    dAkk = (torch.randn(1, T, H, bt, generator=gen, dtype=f32) * strict).contiguous()
    inputs = dict(q=q, k=k, g=g.contiguous(), beta=beta, dAqk=dAqk, dAkk=dAkk)
    return inputs, cu.to(torch.int32)


# The variable-length workload: the headline's 32768 tokens x 16 heads, cut into a
# seeded log-uniform mix of sequence lengths in [1, 8192].
VARLEN_WORKLOAD = dict(name="varlen_T32768_H16", total=32768, H=16, gate_lo=-0.5,
                       max_len=8192)


def make_varlen_workload(seed: int = SEED0):
    w = VARLEN_WORKLOAD
    lens = varlen_seqlens(w["total"], seed=seed, max_len=w["max_len"])
    return make_varlen_inputs(lens, w["H"], gate_lo=w["gate_lo"], seed=seed + 1)


def make_config_inputs(idx: int, seed: int | None = None) -> dict:
    cfg = CONFIGS[idx]
    return make_inputs(cfg.B, cfg.T, cfg.H, gate_lo=cfg.gate_lo,
                       qk_dtype=cfg.qk_dtype,
                       seed=SEED0 + idx if seed is None else seed)


def gather_units(inputs: dict, units, H: int, T: int, bt: int = BT) -> dict:
    """Slice whole units out of a [B, T, H, *] input set.

    ``units`` is an iterable of (b, h, chunk) triples.  The result holds the
    same tensors with shape [n, bt, 1, *] (n units as a batch of single-chunk,
    single-head problems), so any consumer can process exactly those units.
    """
    out = {}
    for name, x in inputs.items():
        parts = []
        for (b, h, c) in units:
            parts.append(x[b, c * bt:(c + 1) * bt, h].unsqueeze(1))
        out[name] = torch.stack(parts, dim=0).contiguous()
    return out


def sample_units(cfg: Config, n: int, seed: int = 7):
    """A deterministic spread of n unit ids, always including the first and last."""
    nchunk = cfg.T // BT
    total = cfg.units
    gen = torch.Generator().manual_seed(seed)
    picks = {0, total - 1}
    if n > 2:
        picks.update(torch.randint(0, total, (n - 2,), generator=gen).tolist())
    out = []
    for u in sorted(picks):
        h = u % cfg.H
        c = (u // cfg.H) % nchunk
        b = u // (cfg.H * nchunk)
        out.append((b, h, c))
    return out
