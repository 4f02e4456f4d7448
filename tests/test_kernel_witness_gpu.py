"""Kernel-name witness: each entry point launches the library's own kernel, and no
library GEMM or other vendor kernel, on the device.

The bwd_intra page names its kernels so that a launch trace shows which one ran; here
the CUDA activity of one small call, recorded by torch.profiler, must hold exactly the
expected kernel of libkda (once) and nothing that looks like a cuBLAS, cuDNN or CUTLASS
GEMM.  The inputs are created and copied before the profiled region, so the call is
the only thing recorded.
"""

import json

import pytest
import torch
from torch.profiler import ProfilerActivity, profile

import gated_delta_rule_intra_gb300 as kda
import kda_inputs
from tests import _gpu

pytestmark = pytest.mark.gpu

LIBRARY_GEMM = ("gemm", "cublas", "cutlass", "cudnn", "xmma", "sm90_", "sm100_", "nvjet")


def _kernels(fn, tmp_path):
    """Names of the kernels the device ran during fn(), from the profiler's raw trace
    (launches made inside libkda have no torch operator around them, so they appear
    only as device activity, not in the operator view)."""
    torch.cuda.synchronize()
    with profile(activities=[ProfilerActivity.CPU, ProfilerActivity.CUDA]) as prof:
        fn()
        torch.cuda.synchronize()
    path = tmp_path / "trace.json"
    prof.export_chrome_trace(str(path))
    events = json.loads(path.read_text()).get("traceEvents", [])
    return [e["name"] for e in events if e.get("cat") == "kernel"]


@pytest.fixture(scope="module", autouse=True)
def _profiler_warmed_up(tmp_path_factory):
    """The first profiling session of a process can miss device activity while the
    profiler starts up; one throw-away session on a torch kernel comes first."""
    x = torch.ones(1024, device="cuda")
    _kernels(lambda: x.add_(1.0), tmp_path_factory.mktemp("warmup"))
    yield


def _inputs():
    cpu = kda_inputs.make_inputs(1, 128, 2, seed=90)
    dev = _gpu.to_device(cpu)
    return [dev[n] for n in _gpu.ARGS]


@pytest.mark.parametrize("entry,kernel", [
    ("kda_intra_bwd", "kda_intra_bwd_tc_kernel"),
    ("kda_intra_bwd_fp32", "kda_intra_bwd_fp32_kernel"),
    ("kda_intra_bwd_ex", "kda_intra_bwd_tc_kernel"),
    ("split_tf32", "kda_intra_bwd_tc_kernel"),
    ("kda_intra_fwd", "kda_intra_fwd_tc_kernel"),
])
def test_entry_point_launches_its_own_kernel(entry, kernel, tmp_path):
    ins = _inputs()
    if entry == "kda_intra_fwd":
        outs = [torch.empty(1, 128, 2, 64, device="cuda") for _ in range(2)]
        call = lambda: kda.kda_intra_fwd(*ins[:4], *outs)  # noqa: E731
    else:
        outs = list(kda._outputs(ins[0], None, None, None, None))
        extra = {"factor_diag": True} if entry == "kda_intra_bwd_ex" else \
            {"split_tf32": True} if entry == "split_tf32" else {}
        fn = kda.kda_intra_bwd_ex if entry == "split_tf32" else getattr(kda, entry)
        call = lambda: fn(*ins, *outs, **extra)  # noqa: E731
    call()  # first call outside the trace: the module loads, attributes are set
    names = _kernels(call, tmp_path)
    ours = [n for n in names if kernel in n]
    assert len(ours) == 1, f"{entry}: expected one {kernel} launch, saw {names}"
    vendor = [n for n in names if any(tag in n.lower() for tag in LIBRARY_GEMM)]
    assert not vendor, f"{entry}: library kernels launched: {vendor}"
    assert len(names) == 1, f"{entry}: unexpected extra launches: {names}"
