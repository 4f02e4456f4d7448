import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the built libkda.so")


def _cuda_available() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:  # pragma: no cover
        return False


def pytest_collection_modifyitems(config, items):
    if _cuda_available():
        return
    skip = pytest.mark.skip(reason="no CUDA device in this process")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(scope="session", autouse=True)
def _built_library():
    """Build libkda.so and its bounds-checked debug build in-tree if either is missing
    or older than its sources."""
    import concurrent.futures
    import glob

    from gated_delta_rule_intra_gb300 import build
    srcs = glob.glob(os.path.join(build.CSRC, "*")) + glob.glob(
        os.path.join(ROOT, "include", "*.h"))
    newest = max(os.path.getmtime(s) for s in srcs)
    jobs = [fn for path, fn in ((build.LIB, build.build_library),
                                (build.DEBUG_LIB, build.build_debug_library))
            if not os.path.exists(path) or os.path.getmtime(path) < newest]
    if jobs:
        with concurrent.futures.ThreadPoolExecutor(len(jobs)) as ex:
            for f in [ex.submit(fn) for fn in jobs]:
                f.result()
    yield
