"""kda_intra_bwd_host_static: the host-buffer entry point that allocates nothing.

Some callers hold only host buffers and may not allocate device memory: a plugin whose
host application's allocator owns the GPU's memory, or a caller under a fixed memory
budget or on a path where cudaMalloc's implicit device synchronisation is not allowed.
For them the library stages the problem in its own fixed device array, so the problem
must fit that array.  These tests call the entry point through the C ABI and compare it
with kda_intra_bwd_host, the entry point that takes a caller-owned workspace.

The file sorts last so that a run stopping at the first failure has run every other
test before it; it also passes alone in a fresh process.
"""

import ctypes
import os
import re

import pytest
import torch

import gated_delta_rule_intra_gb300 as kda
import kda_inputs
from tests import _gpu

TOL = _gpu.TOL["kda_intra_bwd"]
ROW_BYTES = 3080  # staging bytes per token-head row (inputs and outputs)


def _host_problem(B, T, H, seed, dtype):
    cpu = kda_inputs.make_inputs(B, T, H, seed=seed, qk_dtype=dtype)
    host = {n: v.pin_memory() for n, v in cpu.items()}
    return host


def _outputs(B, T, H):
    return [torch.full((B, T, H, 128), float("nan")).pin_memory(),
            torch.full((B, T, H, 128), float("nan")).pin_memory(),
            torch.full((B, T, H), float("nan")).pin_memory(),
            torch.full((B, T, H, 128), float("nan")).pin_memory()]


def _static_call(lib, host, outs, B, T, H, dtype, stream):
    vp = ctypes.c_void_p
    ptrs = [vp(host[n].data_ptr()) for n in _gpu.ARGS] + [vp(o.data_ptr()) for o in outs]
    return lib.kda_intra_bwd_host_static(*ptrs, B, T, H, kda._DTYPES[dtype],
                                         vp(stream.cuda_stream))


@pytest.mark.gpu
def test_two_calls_in_a_row_match_the_workspace_entry_point():
    """Two calls in a row on one stream, the second smaller than the first (so the array
    still holds the first call's bytes beyond the second's extent), each checked against
    kda_intra_bwd_host on the same inputs with a caller-owned workspace."""
    lib = kda.load_library()
    stream = torch.cuda.Stream()
    cases = ((2, 1024, 4, 31, torch.bfloat16),   # 8192 rows, 25.2 MB of staging
             (1, 192, 3, 32, torch.float16))      # a smaller call after it
    for B, T, H, seed, dtype in cases:
        assert B * T * H * ROW_BYTES <= kda.HOST_STATIC_MAX_BYTES
        host = _host_problem(B, T, H, seed, dtype)
        got = _outputs(B, T, H)
        rc = _static_call(lib, host, got, B, T, H, dtype, stream)
        assert rc == kda.KDA_OK, kda.kda_status_str(rc)
        stream.synchronize()

        want = _outputs(B, T, H)
        ws = torch.empty(kda.kda_intra_bwd_host_workspace_bytes(B, T, H, dtype),
                         dtype=torch.uint8, device="cuda")
        kda.kda_intra_bwd_host(*(host[n] for n in _gpu.ARGS), *want, workspace=ws,
                               stream=stream)
        stream.synchronize()
        _gpu.assert_close(got, [w.double().numpy() for w in want], TOL,
                          f"kda_intra_bwd_host_static B={B} T={T} H={H} {dtype}")
        # the same kernel on the same inputs: the results are in fact identical
        for n, a, b in zip(_gpu.NAMES, got, want):
            assert torch.equal(a, b), n


def test_too_large_is_rejected_before_anything_runs():
    """A problem whose staging exceeds the fixed array is refused with its own status,
    before any CUDA call (the pointers here are never dereferenced)."""
    lib = kda.load_library()
    header = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                               "include", "kda.h")).read()
    limit = int(re.search(r"#define KDA_HOST_STATIC_MAX_BYTES (\d+)u", header).group(1))
    assert limit == kda.HOST_STATIC_MAX_BYTES
    vp = ctypes.c_void_p
    base, span = 1 << 40, 1 << 34
    ptrs = [vp(base + i * span) for i in range(10)]
    B, T, H = 1, 64 * 171, 1   # 10,944 rows: one chunk past the 10,880 that fit
    assert kda.kda_intra_bwd_host_workspace_bytes(B, T, H) > kda.HOST_STATIC_MAX_BYTES
    assert kda.kda_intra_bwd_host_workspace_bytes(1, 64 * 170, 1) <= kda.HOST_STATIC_MAX_BYTES
    rc = lib.kda_intra_bwd_host_static(*ptrs, B, T, H, 0, vp(0))
    assert rc == kda.KDA_ERR_TOO_LARGE
    assert "KDA_ERR_TOO_LARGE" in kda.kda_status_str(rc)
    # the ordinary argument checks still come first
    bad = list(ptrs)
    bad[0] = vp(0)
    assert lib.kda_intra_bwd_host_static(*bad, B, T, H, 0, vp(0)) == 1  # KDA_ERR_NULL
