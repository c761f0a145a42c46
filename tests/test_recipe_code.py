"""Recipe int64 code ("NVFP4 4over6 Recipes": nvfp4_4over6_code / nvfp4_4over6_from_code)
through the C ABI, host only (no GPU): the documented bit layout, the round trip of every
recipe field combination, and rejection of codes outside the layout."""
import struct

import pytest

import nvfp4_paged_kv_02_gb300 as nv


def f32_bits(x: float) -> int:
    return struct.unpack("<I", struct.pack("<f", x))[0]


def test_standard_nvfp4_is_code_zero():
    assert nv.nvfp4_4over6_code(None) == 0
    assert nv.nvfp4_4over6_from_code(0) is None


@pytest.mark.parametrize("e4m3_max", [256.0, 448.0, 384.0, 1.0, 2.0 ** -9, 447.5])
@pytest.mark.parametrize("mode", ["MAE", "MSE"])
@pytest.mark.parametrize("fast", [False, True])
def test_layout_and_round_trip(e4m3_max, mode, fast):
    r = nv.NVFP44Over6Config(e4m3_max, mode, fast)
    code = nv.nvfp4_4over6_code(r)
    want = (f32_bits(e4m3_max) << 32) | 1 | (2 if mode == "MSE" else 0) | (4 if fast else 0)
    assert code == (want - (1 << 64) if want >= 1 << 63 else want)
    back = nv.nvfp4_4over6_from_code(code)
    assert back == nv.NVFP44Over6Config(float(struct.unpack("<f", struct.pack("<f", e4m3_max))[0]),
                                        mode, fast)


def test_worked_example():
    # e4m3_max = 256 is 0x43800000 in binary32; MSE and fast math set bits 1 and 2
    assert nv.nvfp4_4over6_code(nv.NVFP44Over6Config(256.0, "MSE", True)) == 0x4380000000000007


@pytest.mark.parametrize("code", [
    2,                                    # bit 0 clear but not zero
    0x4380000000000001 | 8,               # reserved bit set
    (f32_bits(449.0) << 32) | 1,          # e4m3_max above 448
    (f32_bits(0.0) << 32) | 1,            # e4m3_max zero
    (f32_bits(float("nan")) << 32) | 1,   # not finite
    -1,
])
def test_invalid_codes_are_rejected(code):
    if code >= 1 << 63:
        code -= 1 << 64
    with pytest.raises(nv.NVFP4KVError):
        nv.nvfp4_4over6_from_code(code)


def test_invalid_recipe_has_no_code():
    with pytest.raises(nv.NVFP4KVError):
        nv.nvfp4_4over6_code(nv.NVFP44Over6Config(500.0, "MAE", False))
