"""Helpers for the GPU parity tests: run the library, run the oracle, compare."""

from __future__ import annotations

import numpy as np
import torch

import gated_delta_rule_intra_gb300 as kda
import kda_inputs
import oracle

NAMES = ("dq", "dk", "db", "dg")
ARGS = ("q", "k", "g", "beta", "dAqk", "dAkk")

# max|err| / max|ref| per output tensor; "split_tf32" is kda_intra_bwd_ex with the
# split-TF32 cross sums, held to the FP32 path's tolerance
TOL = {"kda_intra_bwd": 2e-3, "kda_intra_bwd_fp32": 1e-4, "split_tf32": 1e-4}
PATHS = tuple(TOL)


def to_device(inp: dict, device="cuda") -> dict:
    return {n: v.to(device) for n, v in inp.items()}


def run(path: str, dev: dict, **kw):
    if path == "split_tf32":
        return kda.kda_intra_bwd_ex(*(dev[n] for n in ARGS), split_tf32=True, **kw)
    fn = getattr(kda, path)
    return fn(*(dev[n] for n in ARGS), **kw)


def oracle_outputs(inp: dict, nthreads: int = 0):
    return oracle.intra_bwd(*(inp[n] for n in ARGS), nthreads=nthreads)


def rel_errors(got, ref) -> dict:
    out = {}
    for n, a, b in zip(NAMES, got, ref):
        a = a.detach().to("cpu", torch.float64).numpy() if isinstance(a, torch.Tensor) else a
        b = np.asarray(b, dtype=np.float64)
        out[n] = float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))
    return out


def assert_close(got, ref, tol, what=""):
    errs = rel_errors(got, ref)
    bad = {n: e for n, e in errs.items() if not (e <= tol)}
    assert not bad, f"{what}: max|err|/max|ref| above {tol:g}: {bad} (all: {errs})"
    return errs


def gather_outputs(outs, units, bt=64):
    """Slice the GPU outputs at the given (b, h, c) units -> [n, bt, 1, *] CPU tensors."""
    idx_b = torch.tensor([u[0] for u in units])
    idx_h = torch.tensor([u[1] for u in units])
    rows = torch.stack([torch.arange(u[2] * bt, (u[2] + 1) * bt) for u in units])
    res = []
    for x in outs:
        xb = x[idx_b.to(x.device)[:, None], rows.to(x.device), idx_h.to(x.device)[:, None]]
        res.append(xb.unsqueeze(2).cpu())
    return res


def sampled_parity(path, cfg_idx, inp_cpu, dev, outs=None, n_units=16):
    cfg = kda_inputs.CONFIGS[cfg_idx]
    units = kda_inputs.sample_units(cfg, n_units)
    if outs is None:
        outs = run(path, dev)
    got = gather_outputs(outs, units)
    sub = kda_inputs.gather_units(inp_cpu, units, cfg.H, cfg.T)
    ref = oracle_outputs(sub)
    return assert_close(got, ref, TOL[path], f"{path} on {cfg.name} (sampled units)")
