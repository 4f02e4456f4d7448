#!/usr/bin/env python
"""Throughput benchmark of the KDA intra-chunk backward (tokens*heads/s, HBM roofline).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one call of the library's intra-chunk backward over the whole workload
(the B=8, T=4096, H=16 headline case by default: 8192 units of one (batch, head,
64-token chunk)), inputs resident in HBM.  The working set (1.61 GB read+written)
is far larger than the 129 MB L2, so steps run back to back without an L2 flush.
``--config`` picks another workload (an index, a name such as ``gate_stress``, or
``all`` for one JSON line per workload).  A workload whose bytes fit in twice the L2
(the single chunk and the small case) is timed call by call with a 258 MB write
between calls that evicts the L2, and its line adds the host cost per call.

Under torchrun (N > 1) every rank runs its own independent shard of the same size
(weak scaling, no collective on the data path); rank 0 prints the JSON line.

``--impl reference`` times the fp64 CPU oracle on the host cores instead (a
bounded sample of the same workload per step).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import kda_inputs  # noqa: E402

METRIC = "KDA intra-chunk bwd tokens·heads/s and achieved HBM GB/s (B=8,T=4096,H=16)"
UNIT = "tokens*heads/s"
FALLBACK_HBM_GBS = 8000.0  # nominal GB300 HBM3e, used only without MEASURED_PEAKS.json
L2_BYTES = 129 * 2 ** 20
KERNEL_NAMES = {
    "kda_intra_bwd": "kda_intra_bwd_tc_kernel",
    "kda_intra_bwd_fp32": "kda_intra_bwd_fp32_kernel",
    "kda_intra_fwd": "kda_intra_fwd_tc_kernel",
}
# forward: q, k, g, beta in; Aqk, Akk ([64 x 64] fp32 each, zeros included) out
FWD_BYTES_PER_UNIT = 2 * 64 * 128 * 2 + 64 * 128 * 4 + 64 * 4 + 2 * 64 * 64 * 4


def algorithmic_bytes_per_unit(qk_bytes: int = 2, group: int = 1, accumulate: bool = False,
                               io_out: bool = False) -> float:
    """Bytes one unit must move at minimum: q, k (shared by `group` value heads),
    g, beta, the ten lower 16x16 blocks of dAqk and dAkk, the dq, dk, dg, db outputs
    (dq, dk in the io dtype when `io_out`), and the incoming gradients when
    `accumulate`."""
    bt, kd, bc = kda_inputs.BT, kda_inputs.K, 16
    qk = 2 * bt * kd * qk_bytes / group
    g = bt * kd * 4
    beta = bt * 4
    da = 2 * 10 * bc * bc * 4
    out = 2 * bt * kd * (qk_bytes if io_out else 4) + bt * kd * 4 + bt * 4
    acc = 3 * bt * kd * 4 + bt * 4 if accumulate else 0
    return qk + g + beta + da + out + acc


def varlen_algorithmic_bytes(lens, H: int, qk_bytes: int = 2, accumulate: bool = False,
                             io_out: bool = False) -> float:
    """algorithmic_bytes_per_unit summed over the chunks of variable-length sequences
    (chunks restart at each sequence start; a short chunk moves its valid rows and the
    lower-block part of their dA rows only), times H heads."""
    bt, kd, bc = kda_inputs.BT, kda_inputs.K, 16
    per_row = (2 * kd * qk_bytes + kd * 4 + 4                # q, k, g, beta
               + 2 * kd * (qk_bytes if io_out else 4) + kd * 4 + 4  # dq, dk, dg, db
               + (3 * kd * 4 + 4 if accumulate else 0))
    total = 0
    for n in lens:
        for c0 in range(0, n, bt):
            m = min(bt, n - c0)
            total += m * per_row + 2 * 4 * sum(bc * (r // bc + 1) for r in range(m))
    return float(total * H)


class VarlenWorkload:
    """The variable-length workload, with the attributes of a kda_inputs.Config."""

    def __init__(self, cu):
        w = kda_inputs.VARLEN_WORKLOAD
        self.lens = (cu[1:] - cu[:-1]).tolist()
        self.name, self.B, self.T, self.H = w["name"], 1, int(cu[-1]), w["H"]
        self.gate_lo, self.qk_dtype = w["gate_lo"], torch.bfloat16
        self.chunks = sum(-(-n // kda_inputs.BT) for n in self.lens)
        self.units = self.chunks * self.H
        self.tokens_heads = self.T * self.H


KERNEL_SOURCES = {
    "kda_intra_bwd_tc_kernel": ("kda_intra_tc.cuh", "kda_intra_tc.cu", "tc_ptx.cuh", "kda_common.cuh"),
    "kda_intra_bwd_fp32_kernel": ("kda_intra_fp32.cu", "kda_intra_tc.cuh", "tc_ptx.cuh",
                                  "kda_common.cuh"),
    "kda_intra_fwd_tc_kernel": ("kda_intra_fwd_tc.cu", "tc_ptx.cuh", "kda_common.cuh"),
}


def code_only(text: str) -> str:
    """C/C++/CUDA source without its comments and blank lines (string and character
    literals kept, trailing blanks dropped): what the compiler sees, so that an edit of
    comments alone leaves a kernel's hash unchanged."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c and text[j] != "\n":
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    lines = (line.rstrip() for line in "".join(out).split("\n"))
    return "\n".join(line for line in lines if line)


def source_hash(kernel: str) -> str:
    """Hash of the code (comments left out) of the source files one kernel is compiled
    from: ties an ncu summary to the code it measured."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "gated_delta_rule_intra_gb300", "csrc")
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            h.update(f.encode())
            h.update(code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.txt")
    try:
        fields = {}
        with open(path) as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    fields[k.strip()] = v.strip()
        if fields.get("source_sha256") != source_hash(kernel):
            return None
        return float(fields["dram_bytes_per_launch"])
    except Exception:
        return None


def summary_name(args, workload: str):
    """Which committed ncu summary covers this run's launch: the plain launch of each
    path on its workload, and on their own the split-TF32, factor_diag and
    variable-length launches of the backward (whose summaries carry the option's name
    or the variable-length workload's).  Other options have none (None)."""
    if args.gva > 1 or args.accumulate or args.fold_dg or args.io_dtype_out:
        return None
    picked = [n for n, on in (("split_tf32", args.split_tf32),
                               ("factor_diag", args.factor_diag),
                               ("varlen", args.varlen)) if on]
    if not picked:
        return workload
    if len(picked) > 1 or args.path != "kda_intra_bwd":
        return None
    return workload if picked == ["varlen"] else f"{picked[0]}_{workload}"


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples taken while the timed region runs."""

    QUERY = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, device_id: str):
        self.samples = []
        self.proc = None
        self.device_id = device_id
        self.window = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.device_id, f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.monotonic(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.samples or self.window is None:
            return None
        t0, t1 = self.window
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        note = "during timed region"
        if not inside:  # timed region shorter than the sampling period
            inside = sorted(self.samples, key=lambda s: min(abs(s[0] - t0), abs(s[0] - t1)))[:2]
            note = "nearest samples (timed region shorter than 100 ms)"
        sm, mx, reasons = [], [], set()
        for _, line in inside:
            parts = [p.strip() for p in line.split(",")]
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except (ValueError, IndexError):
                continue
            for name, val in zip(self.REASONS, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm), "note": note}


def device_selector(dev: torch.device) -> str:
    try:
        return "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        return str(dev.index or 0)


def setup_dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if torch.cuda.is_available():
            torch.cuda.set_device(local)  # before the process group: NCCL binds this device
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def config_dict(cfg, path, opts=None, flushed=False):
    d = {
        "workload": cfg.name, "B": cfg.B, "T": cfg.T, "H": cfg.H, "K": kda_inputs.K,
        "BT": kda_inputs.BT, "BC": 16, "units": cfg.units,
        "qk_dtype": str(cfg.qk_dtype).replace("torch.", ""),
        "gate_lo": cfg.gate_lo, "entry_point": path,
        "l2": "no flush: inputs+outputs of one step (%.2f GB) exceed the 129 MB L2"
              % (cfg.units * algorithmic_bytes_per_unit() / 1e9),
    }
    if path == "kda_intra_fwd":
        d["l2"] = "no flush: inputs+outputs of one step (%.2f GB) exceed the 129 MB L2" % (
            cfg.units * FWD_BYTES_PER_UNIT / 1e9)
    if opts:
        d["options"] = opts
    if flushed:
        d["l2"] = ("flushed: a 258 MB write before every call; each call timed alone "
                   "with CUDA events (the workload fits in the 129 MB L2)")
    if isinstance(cfg, VarlenWorkload):
        d["sequences"] = {"count": len(cfg.lens), "min": min(cfg.lens), "max": max(cfg.lens),
                          "not_whole_chunks": sum(1 for n in cfg.lens if n % kda_inputs.BT),
                          "chunks": cfg.chunks,
                          "recipe": "log-uniform lengths in [1, 8192], seeded"}
        d["l2"] = "no flush: inputs+outputs of one step (%.2f GB) exceed the 129 MB L2" % (
            varlen_algorithmic_bytes(cfg.lens, cfg.H) / 1e9)
    return d


CONFIG_ALIASES = {"single_chunk": kda_inputs.SINGLE_CHUNK, "small": kda_inputs.SMALL,
                  "headline": kda_inputs.HEADLINE, "long": kda_inputs.LONG,
                  "gate_stress": kda_inputs.GATE_STRESS}


def parse_configs(text: str):
    """--config value -> list of indices into kda_inputs.CONFIGS: an index, a short
    name (single_chunk, small, headline, long, gate_stress), a workload name, or
    'all'."""
    t = str(text).strip().lower()
    if t == "all":
        return list(range(len(kda_inputs.CONFIGS)))
    if t.lstrip("-").isdigit():
        i = int(t)
        if not 0 <= i < len(kda_inputs.CONFIGS):
            raise ValueError(f"--config {i}: no such workload")
        return [i]
    if t in CONFIG_ALIASES:
        return [CONFIG_ALIASES[t]]
    for i, c in enumerate(kda_inputs.CONFIGS):
        if c.name.lower() == t:
            return [i]
    raise ValueError(f"--config {text!r}: unknown workload")


# --------------------------------------------------------------------------- oracle

def oracle_rate(cpu_inputs, units_sample, bt=64, nthreads=0):
    """Time the fp64 oracle on a sample; returns (tokens*heads/s, seconds, cores)."""
    import oracle
    lib = oracle.load()
    t = time.perf_counter()
    oracle.intra_bwd(*(cpu_inputs[n] for n in ("q", "k", "g", "beta", "dAqk", "dAkk")),
                     lib=lib, nthreads=nthreads)
    dt = time.perf_counter() - t
    return units_sample * bt / dt, dt, (nthreads or oracle.max_threads(lib))


def cpu_baseline(cpu, cfg):
    """The oracle as it stands on the host cores: the first half of the batch."""
    nb = max(1, cfg.B // 2)
    sample = {n: v[:nb] for n, v in cpu.items()}
    units = nb * cfg.H * (cfg.T // kda_inputs.BT)
    value, secs, cores = oracle_rate(sample, units)
    # the same oracle on one thread, on 64 sampled units (scaled by the unit count)
    few = kda_inputs.sample_units(cfg, 64)
    one, one_secs, _ = oracle_rate(kda_inputs.gather_units(cpu, few, cfg.H, cfg.T), len(few),
                                   nthreads=1)
    return {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"batch elements 0..{nb - 1} of {cfg.B} ({units} of {cfg.units} "
                      f"units), one pass, {secs:.2f} s wall on {cores} threads",
            "single_core": {"value": one, "unit": UNIT, "cores": 1,
                            "sample": f"{len(few)} sampled units, {one_secs:.2f} s, "
                                      "scaled by unit count"}}


def sampled_check(cpu, cfg, outs, n_units=8):
    """max|err|/max|ref| per output on a few sampled units of the last timed step."""
    import numpy as np

    import oracle
    units = kda_inputs.sample_units(cfg, n_units)
    sub = kda_inputs.gather_units(cpu, units, cfg.H, cfg.T)
    ref = oracle.intra_bwd(*(sub[n] for n in ("q", "k", "g", "beta", "dAqk", "dAkk")))
    bt = kda_inputs.BT
    res = {}
    for name, x, r in zip(("dq", "dk", "db", "dg"), outs, ref):
        got = torch.stack([x[b, c * bt:(c + 1) * bt, h] for (b, h, c) in units])
        got = got.unsqueeze(2).double().cpu().numpy()
        res[name] = float(np.max(np.abs(got - r)) / np.max(np.abs(r)))
    res["units"] = len(units)
    return res


def run_reference(args, cfg):
    world, rank, _ = setup_dist()
    if rank != 0:
        return
    import oracle
    oracle.load()
    cpu = kda_inputs.make_config_inputs(args.config)
    nchunk = cfg.T // kda_inputs.BT
    # calibrate, then size each step so the whole run stays within ~2 minutes
    cal_units = kda_inputs.sample_units(cfg, 32)
    cal = kda_inputs.gather_units(cpu, cal_units, cfg.H, cfg.T)
    rate_units = oracle_rate(cal, len(cal_units))[0] / kda_inputs.BT
    per_step = int(max(1, min(cfg.units, 120.0 * rate_units / (args.steps + args.warmup))))
    # a contiguous run of whole (batch, chunk) rows: every head of the first chunks
    chunks = max(1, per_step // cfg.H)
    nb = min(cfg.B, (chunks + nchunk - 1) // nchunk)
    sample = {n: v[:nb, : min(cfg.T, chunks * kda_inputs.BT)] for n, v in cpu.items()}
    units = sample["q"].shape[0] * (sample["q"].shape[1] // kda_inputs.BT) * cfg.H
    for _ in range(args.warmup):
        oracle_rate(sample, units)
    times = []
    for _ in range(args.steps):
        times.append(oracle_rate(sample, units)[1])
    secs = sum(times)
    value = args.steps * units * kda_inputs.BT / secs
    cores = oracle.max_threads()
    desc = (f"{units} of {cfg.units} units per step (batch 0..{nb - 1}, first "
            f"{sample['q'].shape[1]} tokens, all heads)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * secs / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(cfg, "oracle.intra_bwd (fp64 C, OpenMP)"),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- ours

def launch_bytes(args, cfg, qk_bytes: int, fwd: bool) -> float:
    """Algorithmic bytes of one launch of the path and options being timed."""
    if fwd:
        # per valid token row and head: q, k, g, beta in; both 64-column rows out
        per_row = 2 * kda_inputs.K * qk_bytes / args.gva + kda_inputs.K * 4 + 4 + 2 * 64 * 4
        rows = cfg.T * cfg.B if args.varlen else cfg.units * kda_inputs.BT / cfg.H
        return rows * cfg.H * per_row
    if args.varlen:
        b = varlen_algorithmic_bytes(cfg.lens, cfg.H, qk_bytes, accumulate=args.accumulate,
                                     io_out=args.io_dtype_out)
        if args.gva > 1:
            b -= cfg.T * cfg.H * 2 * kda_inputs.K * qk_bytes * (1 - 1 / args.gva)
        return b
    return cfg.units * algorithmic_bytes_per_unit(
        qk_bytes, group=args.gva, accumulate=args.accumulate, io_out=args.io_dtype_out)


def host_cost(step, c_call, dev, n=200):
    """Host wall time per call of n back-to-back calls with no synchronisation between
    them (fewer than the launch queue holds, so the host never waits for the GPU):
    through the C ABI directly (ctypes, arguments built once) and through the Python
    binding (argument checks and marshalling included)."""
    def per_call(f):
        torch.cuda.synchronize(dev)
        t = time.perf_counter()
        for _ in range(n):
            f()
        secs = time.perf_counter() - t
        torch.cuda.synchronize(dev)
        return 1e6 * secs / n
    res = {"calls": n}
    if c_call is not None:
        per_call(c_call)
        res["c_abi_us_per_call"] = per_call(c_call)
    res["binding_us_per_call"] = per_call(step)
    return res


def end_to_end(kda, args, cfg, cpu, outs, stream, dev, world):
    """The metric through kda_intra_bwd_host with pinned host buffers (every step copies
    the inputs up and the outputs down), and beside it the same bytes copied alone, up
    and down at once on two streams: the ceiling the host link sets on this machine.  The
    host side of the link is shared with whatever else the machine runs, so the two are
    timed alternately, E2E_ROUNDS rounds each, and each reports its median round."""
    names = ("q", "k", "g", "beta", "dAqk", "dAkk")
    pin = {n: v.pin_memory() for n, v in cpu.items()}
    hout = [torch.empty_like(o, device="cpu").pin_memory() for o in outs]
    ws = torch.empty(kda.kda_intra_bwd_host_workspace_bytes(cfg.B, cfg.T, cfg.H, cfg.qk_dtype),
                     dtype=torch.uint8, device=dev)
    hin = [pin[n] for n in names]
    for _ in range(2):
        kda.kda_intra_bwd_host(*hin, *hout, workspace=ws, stream=stream)
    bi = sum(t.numel() * t.element_size() for t in hin)
    bo = sum(t.numel() * t.element_size() for t in hout)
    with_link = bi + bo >= LINK_MIN_BYTES
    link = LinkCopies(hin, hout, ws, stream, dev) if with_link else None

    def timed(fn):
        barrier(world)
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.e2e_steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        return max_over_ranks(e0.elapsed_time(e1), world, dev)

    e_ms, link_ms = [], []
    for _ in range(E2E_ROUNDS):
        e_ms.append(timed(lambda: kda.kda_intra_bwd_host(*hin, *hout, workspace=ws,
                                                         stream=stream)))
        if link:
            link_ms.append(timed(link.copies) / args.e2e_steps)
    e_med = statistics.median(e_ms)
    res = {"value": world * cfg.tokens_heads * args.e2e_steps / (e_med / 1e3),
           "unit": UNIT, "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
           "steps": args.e2e_steps, "rounds": E2E_ROUNDS,
           "ms_per_step": e_med / args.e2e_steps,
           "ms_per_step_rounds": [t / args.e2e_steps for t in e_ms],
           "entry_point": "kda_intra_bwd_host (pinned host buffers)"}
    if link:
        lm = statistics.median(link_ms)
        res.update({"link_ms_per_step": lm,
                    "link_ms_per_step_rounds": link_ms,
                    "link_gbs": (bi + bo) / (lm / 1e3) / 1e9,
                    "link_frac": lm / (e_med / args.e2e_steps),
                    "link_how": "the same bytes copied alone: pinned host buffers, pieces of "
                                "about 96 MB, inputs up on one stream and outputs down on "
                                "another, interleaved, no kernel; timed alternately with the "
                                "end-to-end call, median round of each"})
    del ws
    return res


E2E_ROUNDS = 5
LINK_MIN_BYTES = 256 << 20  # below this a copy's fixed cost, not the link, sets the time
LINK_PIECE = 96 << 20


class LinkCopies:
    """One step's inputs copied up and its outputs down with no kernel, the way
    kda_intra_bwd_host moves data: the ceiling the host link sets."""

    def __init__(self, hin, hout, ws, stream, dev):
        views, off = [], 0
        for h in hin + hout:
            nb = h.numel() * h.element_size()
            views.append(ws[off:off + nb])
            off += (nb + 255) // 256 * 256

        def pieces(hosts, devs):
            out = []
            for h, d in zip(hosts, devs):
                hb = h.view(-1).view(torch.uint8)
                for o in range(0, hb.numel(), LINK_PIECE):
                    out.append((hb[o:o + LINK_PIECE], d[o:o + LINK_PIECE]))
            return out

        self.ups = pieces(hin, views[:len(hin)])
        self.downs = pieces(hout, views[len(hin):])
        self.up, self.down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        self.stream = stream
        self.copies()
        torch.cuda.synchronize(dev)

    def copies(self):
        start = torch.cuda.Event()
        start.record(self.stream)
        self.up.wait_event(start)
        self.down.wait_event(start)
        for n in range(max(len(self.ups), len(self.downs))):
            if n < len(self.ups):
                with torch.cuda.stream(self.up):
                    self.ups[n][1].copy_(self.ups[n][0], non_blocking=True)
            if n < len(self.downs):
                with torch.cuda.stream(self.down):
                    self.downs[n][0].copy_(self.downs[n][1], non_blocking=True)
        self.stream.wait_stream(self.up)
        self.stream.wait_stream(self.down)



def run_ours(args, cfg):
    world, rank, local = setup_dist()
    import gated_delta_rule_intra_gb300 as kda

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    kda.load_library()
    stream = torch.cuda.current_stream(dev)
    seed = kda_inputs.SEED0 + args.config + 1000 * rank
    if args.varlen:
        cpu, cu = kda_inputs.make_varlen_workload(kda_inputs.SEED0 + 1000 * rank)
        cfg = VarlenWorkload(cu)
        varlen = {"cu_seqlens": cu.to(dev),
                  "chunk_indices": kda.prepare_chunk_indices(cu).to(dev)}
    else:
        cpu = kda_inputs.make_inputs(cfg.B, cfg.T, cfg.H, gate_lo=cfg.gate_lo,
                                     qk_dtype=cfg.qk_dtype, seed=seed)
        varlen = {}
    if args.gva > 1:  # q/k shared by groups of value heads
        cpu["q"] = cpu["q"][:, :, ::args.gva].contiguous()
        cpu["k"] = cpu["k"][:, :, ::args.gva].contiguous()
    x = {n: v.to(dev) for n, v in cpu.items()}
    ins = [x[n] for n in ("q", "k", "g", "beta", "dAqk", "dAkk")]
    fwd = args.path == "kda_intra_fwd"
    extended = (args.gva > 1 or args.accumulate or args.fold_dg or args.io_dtype_out
                or args.varlen or args.factor_diag or args.split_tf32)
    opts = None
    if fwd:
        if (args.accumulate or args.fold_dg or args.io_dtype_out or args.factor_diag
                or args.split_tf32):
            raise SystemExit("the forward takes --gva and --varlen only")
        outs = list(kda.kda_intra_fwd(*ins[:4], **varlen))
        if extended:
            opts = {"value_heads_per_qk_head": args.gva, "varlen": args.varlen}

        def step():
            kda.kda_intra_fwd(*ins[:4], *outs, **varlen, stream=stream)
    elif extended:
        if args.path != "kda_intra_bwd":
            raise SystemExit("options run on the tensor-core path (--path kda_intra_bwd) only")
        gen = torch.Generator().manual_seed(seed + 1)
        extra = dict(varlen)
        if args.accumulate:
            shp = (cfg.B, cfg.T, cfg.H, kda_inputs.K)
            extra.update({n: torch.randn(*shp, generator=gen).to(dev)
                          for n in ("dq_in", "dk_in", "dg_in")})
            extra["db_in"] = torch.randn(cfg.B, cfg.T, cfg.H, generator=gen).to(dev)
        extra["factor_diag"] = args.factor_diag
        extra["split_tf32"] = args.split_tf32
        if args.in_place:
            if not args.accumulate or args.io_dtype_out:
                raise SystemExit("--in-place needs --accumulate and fp32 outputs")
            outs = [extra["dq_in"], extra["dk_in"], extra["db_in"], extra["dg_in"]]
        else:
            outs = list(kda.kda_intra_bwd_ex(*ins, **extra, fold_dg=args.fold_dg,
                                             dqdk_io_dtype=args.io_dtype_out))
        opts = {"value_heads_per_qk_head": args.gva, "accumulate": args.accumulate,
                "fold_dg": args.fold_dg, "dqdk_io_dtype": args.io_dtype_out,
                "varlen": args.varlen, "factor_diag": args.factor_diag,
                "split_tf32": args.split_tf32, "in_place": args.in_place}

        def step():
            kda.kda_intra_bwd_ex(*ins, *outs, **extra, fold_dg=args.fold_dg,
                                 dqdk_io_dtype=args.io_dtype_out, stream=stream)
    else:
        fn = getattr(kda, args.path)
        outs = kda._outputs(x["q"], None, None, None, None)

        def step():
            fn(*ins, *outs, stream=stream)

    qk_bytes = torch.tensor([], dtype=cfg.qk_dtype).element_size()
    bytes_per_launch = launch_bytes(args, cfg, qk_bytes, fwd)
    # a working set that fits in the L2 would be served from it by back-to-back steps:
    # such workloads are timed call by call, each after a write that evicts the L2
    flushed = bytes_per_launch < 2 * L2_BYTES
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if flushed else None

    for _ in range(args.warmup):
        step()
    sampler = ClockSampler(device_selector(dev))
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize(dev)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    t0 = time.monotonic()
    if flushed:
        pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(args.steps)]
        for a, b in pairs:
            flush.zero_()
            a.record(stream)
            step()
            b.record(stream)
    else:
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.monotonic()
    barrier(world)
    sampler.window = (t0, t1)
    time.sleep(0.25)
    sampler.stop()
    if flushed:
        per_call = sorted(a.elapsed_time(b) for a, b in pairs)
        ms = sum(per_call)
    else:
        ms = ev0.elapsed_time(ev1)
    ms_max = max_over_ranks(ms, world, dev)
    ms_per_step = ms_max / args.steps

    host = None
    if flushed and rank == 0:
        c_call = None
        if not extended:  # the C entry point itself, arguments built once
            import ctypes
            lib = kda.load_library()
            vp = ctypes.c_void_p
            c_fn = getattr(lib, args.path)
            c_args = ([vp(t.data_ptr()) for t in (ins[:4] if fwd else ins)]
                      + [vp(t.data_ptr()) for t in outs]
                      + [cfg.B, cfg.T, cfg.H, kda._DTYPES[cfg.qk_dtype], vp(stream.cuda_stream)])
            c_call = lambda: c_fn(*c_args)  # noqa: E731
        host = host_cost(step, c_call, dev)
        host["device_ms_per_call"] = {"median": per_call[len(per_call) // 2],
                                      "min": per_call[0], "max": per_call[-1]}

    # end to end through the host-buffer entry point
    e2e = None
    if not args.no_e2e and not extended and not fwd:
        e2e = end_to_end(kda, args, cfg, cpu, outs, stream, dev, world)

    cpu_base = None
    if world == 1 and rank == 0 and not args.no_cpu_baseline and not extended and not fwd:
        cpu_base = cpu_baseline(cpu, cfg)
        cpu_base["parity_check"] = sampled_check(cpu, cfg, outs)

    if rank != 0:
        return
    achieved = bytes_per_launch / (ms / args.steps / 1e3) / 1e9
    clocks = sampler.summary()
    if clocks:  # time x clock: a step's length in SM cycles at the sampled clock
        clocks["kcycles_per_step"] = ms_per_step * clocks["sm_mhz"]
    peak, peak_kind = hbm_peak()
    kname = KERNEL_NAMES[args.path]
    summary = summary_name(args, cfg.name)
    traffic = ncu_traffic(kname, summary) if summary else None
    line = {
        "metric": METRIC,
        "value": world * cfg.tokens_heads / (ms_per_step / 1e3),
        "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32" if args.path.endswith("fp32") else
                 "split-tf32+f32" if args.split_tf32 else "tf32+f32",
        "data": "synthetic",
        "config": config_dict(cfg, args.path if fwd else
                              "kda_intra_bwd_ex" if extended else args.path, opts,
                              flushed=flushed),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback: nominal 8 TB/s",
                     "kernel": kname, "algorithmic_bytes_per_launch": bytes_per_launch},
        "cpu_baseline": cpu_base,
        "clocks": clocks,
        "e2e": e2e,
        "gpu_launches": args.steps,
    }
    if host is not None:
        line["host"] = host
    print(json.dumps(line), flush=True)


def main():
    p = argparse.ArgumentParser(description=__doc__,
                                formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--config", default=str(kda_inputs.HEADLINE),
                   help="workload: an index into kda_inputs.CONFIGS, a short name "
                        "(single_chunk, small, headline, long, gate_stress), a workload "
                        "name, or 'all' for one JSON line per workload (default: the "
                        "headline workload, B=8 T=4096 H=16)")
    p.add_argument("--path", choices=tuple(KERNEL_NAMES), default="kda_intra_bwd")
    p.add_argument("--e2e-steps", type=int, default=10)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--gva", type=int, default=1,
                   help="value heads per q/k head (kda_intra_bwd_ex); heads stay H")
    p.add_argument("--accumulate", action="store_true",
                   help="add incoming dq/dk/dg/db in-kernel (kda_intra_bwd_ex)")
    p.add_argument("--in-place", action="store_true",
                   help="with --accumulate: the incoming gradients are the outputs themselves")
    p.add_argument("--fold-dg", action="store_true",
                   help="dg as its chunk-local reverse cumsum (kda_intra_bwd_ex)")
    p.add_argument("--io-dtype-out", action="store_true",
                   help="dq, dk written in the q/k dtype (kda_intra_bwd_ex)")
    p.add_argument("--varlen", action="store_true",
                   help="the variable-length workload (32768 tokens x 16 heads in "
                        "sequences of log-uniform length) through cu_seqlens")
    p.add_argument("--factor-diag", action="store_true",
                   help="diagonal blocks' lower-left quadrant factorized through row 8 "
                        "(kda_intra_bwd_ex)")
    p.add_argument("--split-tf32", action="store_true",
                   help="cross sums in split TF32, FP32-level accuracy (kda_intra_bwd_ex)")
    args = p.parse_args()
    args.warmup = max(3, args.warmup)  # at least three untimed warm-up steps
    for idx in parse_configs(args.config):
        args.config = idx
        cfg = kda_inputs.CONFIGS[idx]
        if args.impl == "reference":
            run_reference(args, cfg)
        else:
            run_ours(args, cfg)
            torch.cuda.empty_cache()


if __name__ == "__main__":
    main()
