import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def has_gpu() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(params=["ring", "ring-static", "direct"])
def append_kernel(request):
    """Run a test once with each append kernel: the TMA ring and the direct-load kernel.
    The library picks one by the size of the call; the host switch
    NVFP4KV_TEST_APPEND_KERNEL (read on every call) overrides that choice, so both kernels
    meet every case. "ring-static" runs the ring kernels (append, dequantize, materialize)
    with a fixed share of the work per CTA instead of the shared work counter, so both
    schedules meet every case too."""
    import nvfp4_paged_kv_02_gb300 as nv
    old = os.environ.get("NVFP4KV_TEST_APPEND_KERNEL")
    os.environ["NVFP4KV_TEST_APPEND_KERNEL"] = request.param.split("-")[0]
    nv.set_dynamic_schedule(request.param != "ring-static")
    try:
        yield request.param
    finally:
        nv.set_dynamic_schedule(True)
        if old is None:
            os.environ.pop("NVFP4KV_TEST_APPEND_KERNEL", None)
        else:
            os.environ["NVFP4KV_TEST_APPEND_KERNEL"] = old


@pytest.fixture(scope="session")
def gpu_lib():
    """The CUDA library, built for sm_103a. On a GPU machine a missing or broken build is
    an error, never a skip."""
    import nvfp4_paged_kv_02_gb300 as nv
    nv.load()
    return nv
