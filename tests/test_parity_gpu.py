"""CUDA path against the fp64 oracle, element by element, through the C ABI."""

import numpy as np
import pytest
import torch

import gated_delta_rule_intra_gb300 as kda
import kda_inputs
import oracle
from tests import _gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def config_inputs():
    cache = {}

    def get(idx):
        if idx not in cache:
            cpu = kda_inputs.make_config_inputs(idx)
            cache.clear()  # keep at most one large config resident
            cache[idx] = (cpu, _gpu.to_device(cpu))
        return cache[idx]
    yield get
    cache.clear()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("path", _gpu.PATHS)
@pytest.mark.parametrize("cfg", [kda_inputs.SINGLE_CHUNK, kda_inputs.SMALL])
def test_full_parity_small_configs(config_inputs, path, cfg):
    cpu, dev = config_inputs(cfg)
    got = _gpu.run(path, dev)
    torch.cuda.synchronize()
    ref = _gpu.oracle_outputs(cpu)
    _gpu.assert_close(got, ref, _gpu.TOL[path], f"{path} config {cfg}")


@pytest.mark.parametrize("path", _gpu.PATHS)
@pytest.mark.parametrize("cfg", [kda_inputs.HEADLINE, kda_inputs.LONG, kda_inputs.GATE_STRESS])
def test_full_parity_full_size(config_inputs, path, cfg):
    """Full-size launch (the benchmark's configuration), every element vs the oracle."""
    cpu, dev = config_inputs(cfg)
    outs = _gpu.run(path, dev)
    torch.cuda.synchronize()
    ref = _gpu.oracle_outputs(cpu)
    _gpu.assert_close(outs, ref, _gpu.TOL[path], f"{path} config {cfg}")
    del ref
    # properties that hold at any size, checked on every unit of the launch
    cf = kda_inputs.CONFIGS[cfg]
    for x in outs:
        assert torch.isfinite(x).all()
    dg = outs[3].view(cf.B, cf.T // 64, 64, cf.H, 128)
    colsum = dg.sum(dim=2).abs().max().item()
    assert colsum <= 1e-4 * dg.abs().max().item() * 8, "sum_t dg over a chunk != 0"


@pytest.mark.parametrize("path", _gpu.PATHS)
@pytest.mark.parametrize("shape", [(1, 64, 1), (3, 192, 5), (1, 128, 7), (2, 64, 3)])
def test_odd_shapes(path, shape):
    B, T, H = shape
    cpu = kda_inputs.make_inputs(B, T, H, seed=B * 1000 + T + H)
    got = _gpu.run(path, _gpu.to_device(cpu))
    _gpu.assert_close(got, _gpu.oracle_outputs(cpu), _gpu.TOL[path], f"{path} {shape}")


@pytest.mark.parametrize("path", _gpu.PATHS)
def test_fp16_gate_stress_small(path):
    cpu = kda_inputs.make_inputs(2, 256, 3, gate_lo=-8.0, qk_dtype=torch.float16, seed=4)
    got = _gpu.run(path, _gpu.to_device(cpu))
    _gpu.assert_close(got, _gpu.oracle_outputs(cpu), _gpu.TOL[path], f"{path} stress")


@pytest.mark.parametrize("path", _gpu.PATHS)
def test_out_of_support_entries_are_ignored(path):
    """Poison dAqk above the diagonal and dAkk on/above it: bitwise same outputs."""
    cpu = kda_inputs.make_inputs(2, 128, 2, seed=11)
    dev = _gpu.to_device(cpu)
    base = _gpu.run(path, dev)
    lower, strict = kda_inputs.chunk_masks()
    up_q = (~lower).repeat(2, 1).view(1, 128, 1, 64).cuda()
    up_k = (~strict).repeat(2, 1).view(1, 128, 1, 64).cuda()
    dev["dAqk"] = torch.where(up_q, torch.full_like(dev["dAqk"], 3e38), dev["dAqk"])
    dev["dAkk"] = torch.where(up_k, torch.full_like(dev["dAkk"], float("nan")), dev["dAkk"])
    got = _gpu.run(path, dev)
    for n, a, b in zip(_gpu.NAMES, got, base):
        assert torch.equal(a, b), f"{n} depends on out-of-support dA entries"


@pytest.mark.parametrize("path", _gpu.PATHS)
def test_every_output_written_and_nothing_else(path):
    """NaN-prefilled outputs inside canary-padded buffers."""
    B, T, H = 2, 192, 3
    cpu = kda_inputs.make_inputs(B, T, H, seed=12)
    dev = _gpu.to_device(cpu)
    pad = 4096
    outs = []
    for shape in ((B, T, H, 128), (B, T, H, 128), (B, T, H), (B, T, H, 128)):
        n = int(np.prod(shape))
        buf = torch.full((n + 2 * pad,), float("nan"), device="cuda")
        buf[:pad] = 1234.5
        buf[-pad:] = -4321.5
        outs.append((buf, buf[pad:pad + n].view(shape)))
    dq, dk, db, dg = (o[1] for o in outs)
    _gpu.run(path, dev, dq=dq, dk=dk, db=db, dg=dg)
    torch.cuda.synchronize()
    for buf, view in outs:
        assert torch.isfinite(view).all()
        assert (buf[:pad] == 1234.5).all() and (buf[-pad:] == -4321.5).all()
    _gpu.assert_close((dq, dk, db, dg), _gpu.oracle_outputs(cpu), _gpu.TOL[path], path)


@pytest.mark.parametrize("path", _gpu.PATHS)
def test_deterministic(path):
    cpu = kda_inputs.make_inputs(2, 256, 4, seed=13)
    dev = _gpu.to_device(cpu)
    a = _gpu.run(path, dev)
    b = _gpu.run(path, dev)
    for n, x, y in zip(_gpu.NAMES, a, b):
        assert torch.equal(x, y), f"{n} differs between identical calls"


@pytest.mark.parametrize("path", _gpu.PATHS)
def test_zero_gradients_give_zero_outputs(path):
    cpu = kda_inputs.make_inputs(1, 128, 2, seed=14)
    cpu["dAqk"].zero_()
    cpu["dAkk"].zero_()
    got = _gpu.run(path, _gpu.to_device(cpu))
    for n, x in zip(_gpu.NAMES, got):
        assert torch.count_nonzero(x).item() == 0, n


@pytest.mark.parametrize("path", _gpu.PATHS)
def test_gate_free(path):
    cpu = kda_inputs.make_inputs(1, 128, 2, seed=15)
    cpu["g"].zero_()
    got = _gpu.run(path, _gpu.to_device(cpu))
    _gpu.assert_close(got, _gpu.oracle_outputs(cpu), _gpu.TOL[path], f"{path} g=0")


def test_side_stream_and_paths_agree():
    cpu = kda_inputs.make_inputs(2, 256, 2, seed=16)
    dev = _gpu.to_device(cpu)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        got = _gpu.run("kda_intra_bwd", dev, stream=s)
    s.synchronize()
    ref = _gpu.run("kda_intra_bwd_fp32", dev)
    _gpu.assert_close(got, [x.cpu().double().numpy() for x in ref], 2e-3, "fast vs fp32")


def test_host_entry_point_matches_device_path():
    B, T, H = 2, 256, 3
    cpu = kda_inputs.make_inputs(B, T, H, seed=17)
    pinned = {n: v.pin_memory() for n, v in cpu.items()}
    outs = [torch.empty(B, T, H, 128).pin_memory(), torch.empty(B, T, H, 128).pin_memory(),
            torch.empty(B, T, H).pin_memory(), torch.empty(B, T, H, 128).pin_memory()]
    nbytes = kda.kda_intra_bwd_host_workspace_bytes(B, T, H, torch.bfloat16)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    kda.kda_intra_bwd_host(*(pinned[n] for n in _gpu.ARGS), *outs, workspace=ws)
    torch.cuda.current_stream().synchronize()
    ref = _gpu.run("kda_intra_bwd", _gpu.to_device(cpu))
    for n, a, b in zip(_gpu.NAMES, outs, ref):
        assert torch.equal(a, b.cpu()), n


@pytest.mark.parametrize("pinned_host", [True, False])
def test_host_entry_point_pipelined_pieces(pinned_host):
    """About 300 MB of input: the host entry point splits it into three pieces of
    85-86 chunks on its internal streams (beta and db move whole); the result is
    bitwise the device path's."""
    B, T, H = 4, 4096, 12
    cpu = kda_inputs.make_inputs(B, T, H, seed=19)
    host = {n: (v.pin_memory() if pinned_host else v.clone()) for n, v in cpu.items()}
    mk = (lambda *shape: torch.empty(*shape).pin_memory()) if pinned_host else torch.empty
    outs = [mk(B, T, H, 128), mk(B, T, H, 128), mk(B, T, H), mk(B, T, H, 128)]
    ws = torch.empty(kda.kda_intra_bwd_host_workspace_bytes(B, T, H, torch.bfloat16),
                     dtype=torch.uint8, device="cuda")
    side = torch.cuda.Stream()
    kda.kda_intra_bwd_host(*(host[n] for n in _gpu.ARGS), *outs, workspace=ws, stream=side)
    side.synchronize()
    ref = _gpu.run("kda_intra_bwd", _gpu.to_device(cpu))
    for n, a, b in zip(_gpu.NAMES, outs, ref):
        assert torch.equal(a, b.cpu()), n


def test_host_entry_point_from_several_threads():
    """Four host threads call kda_intra_bwd_host at once, each with its own buffers,
    workspace and stream (the calls share the library's internal copy streams and
    events, taken under a per-device lock; ctypes releases the GIL): every result is
    bitwise the device path's."""
    import threading
    B, T, H = 1, 2048, 4
    jobs = []
    for n in range(4):
        cpu = kda_inputs.make_inputs(B, T, H, seed=150 + n)
        host = {k: v.pin_memory() for k, v in cpu.items()}
        outs = [torch.empty(B, T, H, 128).pin_memory(), torch.empty(B, T, H, 128).pin_memory(),
                torch.empty(B, T, H).pin_memory(), torch.empty(B, T, H, 128).pin_memory()]
        ws = torch.empty(kda.kda_intra_bwd_host_workspace_bytes(B, T, H, torch.bfloat16),
                         dtype=torch.uint8, device="cuda")
        jobs.append((cpu, host, outs, ws, torch.cuda.Stream()))
    errors = []

    def work(job):
        cpu, host, outs, ws, stream = job
        try:
            for _ in range(3):
                kda.kda_intra_bwd_host(*(host[n] for n in _gpu.ARGS), *outs, workspace=ws,
                                       stream=stream)
            stream.synchronize()
        except Exception as e:  # pragma: no cover - reported below
            errors.append(e)

    threads = [threading.Thread(target=work, args=(j,)) for j in jobs]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for cpu, host, outs, ws, stream in jobs:
        ref = _gpu.run("kda_intra_bwd", _gpu.to_device(cpu))
        for n, a, b in zip(_gpu.NAMES, outs, ref):
            assert torch.equal(a, b.cpu()), n


def test_misaligned_pointer_is_a_status_not_a_fault():
    cpu = kda_inputs.make_inputs(1, 64, 1, seed=18)
    dev = _gpu.to_device(cpu)
    buf = torch.empty(64 * 128 + 1, device="cuda")
    bad = buf[1:].view(1, 64, 1, 128)  # 4 bytes off a 16-byte boundary
    bad.copy_(dev["g"])
    for path in _gpu.PATHS:
        with pytest.raises(kda.KdaError, match="ALIGN"):
            _gpu.run(path, {**dev, "g": bad})


def test_sampled_units_match_full_launch():
    """The sampled-unit helper the benchmark uses agrees with the full launch."""
    cpu = kda_inputs.make_config_inputs(kda_inputs.SMALL)
    dev = _gpu.to_device(cpu)
    _gpu.sampled_parity("kda_intra_bwd", 1, cpu, dev, n_units=8)


def _device_inputs(B, T, H, seed):
    """The input recipe of kda_inputs, drawn on the GPU (for sizes too large to draw on
    the host in reasonable time)."""
    gen = torch.Generator(device="cuda").manual_seed(seed)
    f32 = torch.float32

    def rows(x):
        return (x / x.norm(dim=-1, keepdim=True)).to(torch.bfloat16)

    q = rows(torch.randn(B, T, H, 128, generator=gen, device="cuda"))
    k = rows(torch.randn(B, T, H, 128, generator=gen, device="cuda"))
    step = torch.rand(B, T, H, 128, generator=gen, device="cuda") * -0.5
    g = step.view(B, T // 64, 64, H, 128).cumsum(2, dtype=f32).view(B, T, H, 128)
    del step
    beta = torch.rand(B, T, H, generator=gen, device="cuda")
    lower, strict = (m.cuda() for m in kda_inputs.chunk_masks())
    dAqk = (torch.randn(B, T // 64, 64, H, 64, generator=gen, device="cuda") *
            lower.view(1, 1, 64, 1, 64)).view(B, T, H, 64)
    dAkk = (torch.randn(B, T // 64, 64, H, 64, generator=gen, device="cuda") *
            strict.view(1, 1, 64, 1, 64)).view(B, T, H, 64)
    return dict(q=q, k=k, g=g.contiguous(), beta=beta, dAqk=dAqk.contiguous(),
                dAkk=dAkk.contiguous())


def test_maximum_head_count():
    """H = KDA_MAX_H = 65536 (one chunk, 65536 units, about 430 per SM): sampled heads of
    every output of both backward paths and of the forward against the oracle."""
    B, T, H = 1, 64, 65536
    dev = _device_inputs(B, T, H, seed=31)
    heads = [0, 1, 12345, 40000, H - 2, H - 1]
    sub = {n: v[:, :, heads].cpu().contiguous() for n, v in dev.items()}
    ref = _gpu.oracle_outputs(sub)
    for path in _gpu.PATHS:
        outs = _gpu.run(path, dev)
        got = [o[:, :, heads].cpu() for o in outs]
        del outs
        _gpu.assert_close(got, ref, _gpu.TOL[path], f"{path} at H = {H}")
    fref = oracle.intra_fwd(*(sub[n] for n in ("q", "k", "g", "beta")))
    fouts = kda.kda_intra_fwd(*(dev[n] for n in ("q", "k", "g", "beta")))
    for name, a, b in zip(("Aqk", "Akk"), fouts, fref):
        a = a[:, :, heads].double().cpu().numpy()
        assert float(np.max(np.abs(a - b)) / np.max(np.abs(b))) <= 2e-3, name


@pytest.mark.parametrize("path", _gpu.PATHS)
def test_many_units_per_cta_with_an_odd_head_count(path):
    """896 units with H = 7: each persistent CTA runs about six units and the unit's head
    wraps around H as it advances by the grid stride; every element against the oracle."""
    cpu = kda_inputs.make_inputs(2, 4096, 7, seed=140)
    got = _gpu.run(path, _gpu.to_device(cpu))
    _gpu.assert_close(got, _gpu.oracle_outputs(cpu), _gpu.TOL[path], f"{path} H=7 B=2 T=4096")
