"""Contiguous quantize / dequantize ("FP4 KV Cache Quantization": nvfp4_kv_quantize,
nvfp4_kv_dequantize) through the C ABI against the CPU oracle, bit-exact on the packed
codes, the scale bytes and the dequantized fp16/bf16 values. Sizes span several pipeline
tiles with a ragged tail, strided input rows, rows too long for a shared-memory stage (the
direct-load kernel), the recipes and both dtypes. Every test runs once with each quantize
kernel (the TMA ring and the direct-load kernel); the dequantize's two kernels are chosen
by alignment and size, and one test runs each."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("append_kernel")]


@pytest.fixture(scope="module", autouse=True)
def _cuda(gpu_lib):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    yield


RECIPES = [None, W.Recipe(256.0, 0, False), W.Recipe(256.0, 1, False),
           W.Recipe(256.0, 0, True), W.Recipe(256.0, 1, True), W.Recipe(448.0, 1, False)]


def _gpu_recipe(nv, r):
    if r is None:
        return None
    return nv.NVFP44Over6Config(r.e4m3_max, "MSE" if r.err_mode else "MAE",
                                bool(r.err_use_fast_math))


def _input(seed, rows, cols, dtype, pad=0):
    rng = np.random.Generator(np.random.PCG64(seed + 7000))
    x = rng.standard_normal((rows, cols + pad)).astype(np.float32)
    x *= rng.uniform(0.05, 30.0, size=(rows, 1)).astype(np.float32)
    if rows * cols >= 64:  # a few outlier columns
        x[:, rng.integers(0, cols, size=2)] *= 20.0
    return torch.from_numpy(x).to(dtype)


CASES = []
for i, (rows, cols, pad) in enumerate([(1, 16, 0), (37, 128, 0), (1000, 64, 0), (257, 1024, 0),
                                       (129, 256, 64), (5, 16384, 0), (3, 32768, 0),
                                       (2049, 48, 16)]):
    for j, recipe in enumerate(RECIPES):
        for dt in (torch.bfloat16, torch.float16):
            CASES.append((100 * i + 10 * j + (dt == torch.float16), rows, cols, pad, recipe, dt))


@pytest.mark.parametrize("seed,rows,cols,pad,recipe,dtype", CASES)
def test_kv_quantize_dequantize(seed, rows, cols, pad, recipe, dtype):
    import nvfp4_paged_kv_02_gb300 as nv
    dev = torch.device("cuda")
    xfull = _input(seed, rows, cols, dtype, pad)
    x_host = xfull[:, :cols]
    cap = 448.0 if recipe is None else recipe.e4m3_max
    gs = float(np.float32(float(x_host.float().abs().max()) / (6.0 * cap)))
    xd = xfull.to(dev)[:, :cols]
    g = torch.tensor([gs], dtype=torch.float32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    fp4, sf = nv.nvfp4_kv_quantize(xd, g, _gpu_recipe(nv, recipe), dev_status=st)
    o_codes, o_sf = O.kv_quantize(W.bits16(x_host), dtype == torch.bfloat16, gs, recipe)
    assert int(st.item()) == 0
    assert np.array_equal(sf.cpu().numpy(), o_sf), "scale bytes"
    assert np.array_equal(fp4.cpu().numpy(), o_codes), "codes"
    for out_dt in (torch.bfloat16, torch.float16):
        y = nv.nvfp4_kv_dequantize(fp4, sf, g, out_dt)
        want = O.kv_dequantize(o_codes, o_sf, gs, out_dt == torch.bfloat16)
        assert np.array_equal(W.bits16(y.cpu()), want), out_dt


@pytest.mark.parametrize("rows,cols", [(64, 256), (257, 1024), (2049, 48), (5, 16384)])
def test_kv_dequantize_each_kernel(rows, cols):
    """The dequantize reads aligned codes and scales of at least 1024 blocks through its
    bulk-copy ring (the blocks after the last whole chunk of 1024 directly), and anything
    else with direct loads: scales one byte off a 16-byte boundary, or an output 16 bytes
    off a 32-byte boundary (16-byte stores). Each must match the oracle."""
    import nvfp4_paged_kv_02_gb300 as nv
    dev = torch.device("cuda")
    x = _input(4242 + rows, rows, cols, torch.bfloat16)
    gs = float(np.float32(float(x.float().abs().max()) / 2688.0))
    c, s = O.kv_quantize(W.bits16(x), True, gs, None)
    g = torch.tensor([gs], dtype=torch.float32, device=dev)
    fp4 = torch.from_numpy(c).to(dev)
    sf = torch.from_numpy(s).to(dev)
    sf_buf = torch.zeros(s.size + 16, dtype=torch.uint8, device=dev)
    sf_off = sf_buf[1:1 + s.size].view(rows, cols // 16)  # 1 byte past an aligned base
    sf_off.copy_(sf)
    for out_dt in (torch.bfloat16, torch.float16):
        want = O.kv_dequantize(c, s, gs, out_dt == torch.bfloat16)
        out_buf = torch.full((rows * cols + 16,), float("nan"), dtype=out_dt, device=dev)
        shifted = out_buf[8:8 + rows * cols].view(rows, cols)  # 16 bytes past a 32-byte base
        for name, scales, out in (("ring", sf, None), ("scales off 16 B", sf_off, None),
                                  ("output off 32 B", sf, shifted)):
            st = torch.zeros(1, dtype=torch.int32, device=dev)
            y = nv.nvfp4_kv_dequantize(fp4, scales, g, out_dt, out=out, dev_status=st)
            torch.cuda.synchronize()
            assert int(st.item()) == 0, name
            assert np.array_equal(W.bits16(y.cpu()), want), (name, out_dt)
        assert bool(out_buf[:8].isnan().all()) and bool(out_buf[8 + rows * cols:].isnan().all())


def test_kv_quantize_leading_dims_and_out():
    """[..., D] inputs keep their leading dimensions; caller-provided outputs are filled."""
    import nvfp4_paged_kv_02_gb300 as nv
    dev = torch.device("cuda")
    x = _input(5, 6 * 8, 128, torch.bfloat16).view(6, 8, 128)
    gs = float(np.float32(float(x.float().abs().max()) / 2688.0))
    g = torch.tensor([gs], dtype=torch.float32, device=dev)
    out = (torch.full((6, 8, 64), 0xA5, dtype=torch.uint8, device=dev),
           torch.full((6, 8, 8), 0xA5, dtype=torch.uint8, device=dev))
    fp4, sf = nv.nvfp4_kv_quantize(x.to(dev), g, None, out=out)
    assert fp4.data_ptr() == out[0].data_ptr() and fp4.shape == (6, 8, 64) and sf.shape == (6, 8, 8)
    c, s = O.kv_quantize(W.bits16(x.reshape(48, 128)), True, gs, None)
    assert np.array_equal(fp4.cpu().numpy().reshape(48, 64), c)
    assert np.array_equal(sf.cpu().numpy().reshape(48, 8), s)
    y = nv.nvfp4_kv_dequantize(fp4, sf, g, torch.float16)
    assert y.shape == (6, 8, 128)


def test_kv_quantize_bad_device_scale_is_reported():
    """A global scale that is not positive finite is reported and nothing is written."""
    import nvfp4_paged_kv_02_gb300 as nv
    dev = torch.device("cuda")
    x = _input(9, 64, 128, torch.float16).to(dev)
    for bad in (0.0, -1.0, float("inf"), float("nan")):
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        out = (torch.full((64, 64), 0x5A, dtype=torch.uint8, device=dev),
               torch.full((64, 8), 0x5A, dtype=torch.uint8, device=dev))
        nv.nvfp4_kv_quantize(x, torch.tensor([bad], device=dev), None, out=out, dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) & nv.DEV_BAD_SCALE
        assert bool((out[0] == 0x5A).all()) and bool((out[1] == 0x5A).all())


def test_kv_quantize_large_sampled():
    """A bench-sized contiguous tensor (the large-pool K rows, 2.3 M x 1024) compared with the
    oracle on sampled rows."""
    import nvfp4_paged_kv_02_gb300 as nv
    dev = torch.device("cuda")
    rows, cols = 2_290_174, 1024
    gen = torch.Generator(device=dev)
    gen.manual_seed(11)
    x = torch.randn((rows, cols), generator=gen, device=dev).mul_(2.0).to(torch.bfloat16)
    recipe = W.Recipe(256.0, 0, True)
    gs = float(np.float32(float(x.float().abs().max()) / 1536.0))
    g = torch.tensor([gs], dtype=torch.float32, device=dev)
    fp4, sf = nv.nvfp4_kv_quantize(x, g, _gpu_recipe(nv, recipe))
    y = nv.nvfp4_kv_dequantize(fp4, sf, g, torch.bfloat16)
    idx = torch.tensor(sorted(set(np.random.default_rng(3).integers(0, rows, 200).tolist())
                              | {0, rows - 1}), device=dev)
    xs = x[idx].cpu()
    c, s = O.kv_quantize(W.bits16(xs), True, gs, recipe)
    assert np.array_equal(fp4[idx].cpu().numpy(), c)
    assert np.array_equal(sf[idx].cpu().numpy(), s)
    assert np.array_equal(W.bits16(y[idx].cpu()), O.kv_dequantize(c, s, gs, True))


def test_kv_ops_past_2_gib_of_codes():
    """4.3 M rows of 1024 elements: the codes (2.2 GB) and the output run past 2^31 bytes, so
    every offset in both bulk-copy rings must be 64-bit. Sampled rows, the last ones
    included, are compared with the oracle."""
    import nvfp4_paged_kv_02_gb300 as nv
    dev = torch.device("cuda")
    rows, cols = 4_300_000, 1024
    gen = torch.Generator(device=dev)
    gen.manual_seed(29)
    x = torch.empty((rows, cols), dtype=torch.bfloat16, device=dev)
    for r0 in range(0, rows, 1 << 20):  # in slices, to bound the binary32 temporaries
        x[r0:r0 + (1 << 20)] = torch.randn((min(1 << 20, rows - r0), cols), generator=gen,
                                           device=dev).mul_(2.0)
    gs = float(np.float32(float(x.abs().max()) / 2688.0))
    g = torch.tensor([gs], dtype=torch.float32, device=dev)
    fp4, sf = nv.nvfp4_kv_quantize(x, g, None)
    y = nv.nvfp4_kv_dequantize(fp4, sf, g, torch.bfloat16)
    assert fp4.numel() > (1 << 31)
    idx = torch.tensor(sorted(set(np.random.default_rng(31).integers(0, rows, 100).tolist())
                              | {0, rows // 2, rows - 2, rows - 1}), device=dev)
    xs = x[idx].cpu()
    c, s = O.kv_quantize(W.bits16(xs), True, gs, None)
    assert np.array_equal(fp4[idx].cpu().numpy(), c)
    assert np.array_equal(sf[idx].cpu().numpy(), s)
    assert np.array_equal(W.bits16(y[idx].cpu()), O.kv_dequantize(c, s, gs, True))
