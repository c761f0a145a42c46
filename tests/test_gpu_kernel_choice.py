"""The append (and the contiguous quantize) pick a kernel by the size of the call: at most
2^18 16-element blocks per tensor run the direct-load kernel, larger calls run the TMA ring.
Here the library makes its own choice (the test override is cleared) on both sides of that
boundary, and every byte matches the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from tests import pipelines as PL

pytestmark = pytest.mark.gpu

# 8 heads of 128 elements: 64 blocks per token and tensor, so 4096 tokens are 2^18 blocks
H, D = 8, 128
BOUNDARY_TOKENS = (1 << 18) // (H * D // 16)


@pytest.fixture(scope="module", autouse=True)
def _cuda(gpu_lib):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    yield


@pytest.fixture(autouse=True)
def _library_choice(monkeypatch):
    monkeypatch.delenv("NVFP4KV_TEST_APPEND_KERNEL", raising=False)


@pytest.mark.parametrize("extra", [-1, 0, 1, 37])
def test_paged_append_either_side_of_the_kernel_boundary(extra):
    lens = np.array([1024, 1024, 1024, 1024 + extra], np.int64)
    assert lens.sum() == BOUNDARY_TOKENS + extra
    w = W.make_paged(f"boundary{extra}", 900 + extra, B=4, H=H, D=D, ps=16, layout=W.HND,
                     dtype=torch.bfloat16, lens_old=np.zeros(4, np.int64), lens_new=lens,
                     recipe=W.Recipe(256.0, 0, True), slack=0.1)
    PL.assert_same(PL.run_gpu(w), PL.run_oracle(w), f"boundary {extra:+d}")


@pytest.mark.parametrize("extra", [0, 1])
def test_contiguous_quantize_either_side_of_the_kernel_boundary(extra):
    import nvfp4_paged_kv_02_gb300 as nv
    rows = BOUNDARY_TOKENS + extra
    rng = np.random.Generator(np.random.PCG64(950 + extra))
    x = torch.from_numpy(rng.standard_normal((rows, H * D)).astype(np.float32) * 2.5)
    x = x.to(torch.float16)
    recipe = W.Recipe(256.0, 1, False)
    gs = float(np.float32(float(x.float().abs().max()) / (6 * 256.0)))
    g = torch.tensor([gs], dtype=torch.float32, device="cuda")
    fp4, sf = nv.nvfp4_kv_quantize(x.cuda(), g, PL.gpu_recipe(recipe))
    codes, scales = O.kv_quantize(W.bits16(x), False, gs, PL.oracle_recipe(recipe))
    assert np.array_equal(fp4.cpu().numpy(), codes)
    assert np.array_equal(sf.cpu().numpy(), scales)
