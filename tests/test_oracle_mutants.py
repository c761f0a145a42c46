"""Planted mistakes in the oracle must be caught by its pins (CPU only).

Each case copies oracle/nvfp4_oracle.c, makes one plausible mistake (a dropped term, a
wrong sign, index, rounding rule or operand order), compiles the copy into a temporary
directory and runs every pin against it. A mutant that passes every pin means the pins
would not notice that mistake in the oracle, and fails this test.
"""
import os

import pytest

import oracle as O
from tests import pins

SRC = os.path.join(os.path.dirname(O.__file__), "nvfp4_oracle.c")

MUTANTS = {
    "ties_away_from_zero": (
        "if (fr > 0.5 || (fr == 0.5 && fmod(fl, 2.0) == 1.0)) fl += 1.0;",
        "if (fr >= 0.5) fl += 1.0;"),
    "no_subnormal_spacing": ("  if (e < emin) e = emin;\n  double q", "  double q"),
    "e2m1_drops_negative_zero": (
        "uint32_t s = signbit(v) ? 8u : 0u;", "uint32_t s = (v < 0) ? 8u : 0u;"),
    "e2m1_no_saturation": ("  if (a > 6.0) a = 6.0;\n", "  if (a > 8.0) a = 8.0;\n"),
    "e4m3_no_saturation": ("  if (a > 448.0) a = 448.0;\n", ""),
    "nibbles_swapped": (
        "codes[k] = (uint8_t)(q[2 * k] | (q[2 * k + 1] << 4));",
        "codes[k] = (uint8_t)(q[2 * k + 1] | (q[2 * k] << 4));"),
    "amax_is_signed_max": (
        "  for (int i = 0; i < 16; ++i) {\n    float a = fabsf(x[i]);",
        "  for (int i = 0; i < 16; ++i) {\n    float a = x[i];"),
    "standard_scale_uses_4": ("float g6 = 6.0f * gs;", "float g6 = 4.0f * gs;"),
    "candidate_b_uses_6": ("float g4 = 4.0f * gs;", "float g4 = 6.0f * gs;"),
    "candidate_b_capped_like_a": (
        "if (rb > 448.0f) rb = 448.0f;", "if (rb > cap_a) rb = cap_a;"),
    "scale_cap_ignores_recipe": (
        "float cap_a = oracle_e4m3_max(r);", "float cap_a = 448.0f;"),
    "reciprocal_forgets_gs": ("float den = S * gs;", "float den = S;"),
    "tie_prefers_amax4": ("if (eb < ea) {", "if (eb <= ea) {"),
    "mae_mse_swapped": (
        "t[i] = mse ? e * e : fabsf(e);", "t[i] = mse ? fabsf(e) : e * e;"),
    "mae_signed_error": ("t[i] = mse ? e * e : fabsf(e);", "t[i] = mse ? e * e : e;"),
    "error_sign_flipped": ("float e = fmaf(-w, gs, x[i]);", "float e = fmaf(w, gs, x[i]);"),
    "fast_math_ignored": ("if (!r->err_use_fast_math) {", "if (1) {"),
    # other plausible rounding steps of the 4over6 element error (readings R6, R7)
    "error_f32_unfused": ("float e = fmaf(-w, gs, x[i]);", "float e = x[i] - w * gs;"),
    "fast_math_decode_factor_rounded": (
        "double e = f16_round(fma(-w, gh, xh));",
        "double e = f16_round(fma(-oracle_e2m1_decode(q[i]), f16_round(S * gh), xh));"),
    "fast_math_dequant_in_f32": (
        "double e = f16_round(fma(-w, gh, xh));",
        "double e = f16_round(xh - f16_round((double)((float)w * gs)));"),
    "fast_math_unfused": (
        "double e = f16_round(fma(-w, gh, xh));", "double e = f16_round(xh - f16_round(w * gh));"),
    "fast_math_keeps_gs_exact": ("double gh = f16_round((double)gs);",
                                 "double gh = (double)gs * 3.0;"),
    "global_scale_ignores_recipe": (
        "float denom = 6.0f * oracle_e4m3_max(r);", "float denom = 6.0f * 448.0f;"),
    "global_scale_zero_tensor": ("if (amax == 0.0f) return 1.0f;", ""),
    "v_interleave_read_as_linear": (
        "return page * sf_page_stride + (h * ps + group * 4) * nb + j * 4 + lane;",
        "return page * sf_page_stride + (h * ps + group * 4 + lane) * nb + j;"),
    "v_interleave_applied_to_k": (
        "int64_t si = (kv == 1 && v_sf_layout == 1)", "int64_t si = (v_sf_layout == 1)"),
    "v_interleave_groups_span_heads": (
        "return page * sf_page_stride + (h * ps + group * 4) * nb + j * 4 + lane;",
        "return page * sf_page_stride + (group * 4 * 2 + h * 4) * nb + j * 4 + lane;"),
    "hnd_addressed_as_nhd": (
        "return layout == 0 ? slot * H + h : h * ps + slot;", "return slot * H + h;"),
    "append_slot_off_by_one": ("int64_t slot = pos % ps;", "int64_t slot = (pos + 1) % ps;"),
    "dequant_rounds_scale_product_first": (
        "  float w = (float)(oracle_e2m1_decode(code) * oracle_e4m3_decode(s));\n"
        "  float d = w * gs;",
        "  float d = (float)oracle_e2m1_decode(code) * (float)((float)oracle_e4m3_decode(s) * gs);"),
    "dequant_writes_past_length": (
        "int64_t len = seq_lens[b] < max_seq_len ? seq_lens[b] : max_seq_len;",
        "int64_t len = max_seq_len;"),
    "dequant_nibble_order": (
        "uint32_t code = (d % 2 == 0) ? (byte & 0xFu) : (byte >> 4);\n          o[d]",
        "uint32_t code = (d % 2 == 1) ? (byte & 0xFu) : (byte >> 4);\n          o[d]"),
    "materialize_page_not_shifted": ("int64_t o = base + j + 1;", "int64_t o = base + j;"),
    "materialize_page0_not_zeroed": ("  memset(out, 0, (size_t)(2 * page_elems));\n", ""),
    "materialize_padding_not_zeroed": (
        "else if (zero_tables) fp8_block_tables[b * mpps + j] = 0;",
        "else if (zero_tables) fp8_block_tables[b * mpps + j] = -1;"),
    "materialize_v_uses_k_table": (
        "int64_t col = shared ? b * max_num_pages + j : (b * 2 + kv) * max_num_pages + j;",
        "int64_t col = shared ? b * max_num_pages + j : (b * 2) * max_num_pages + j;"),
    "kv_quantize_blocks_rotated": (
        "quantize_block(xb, gs, r, codes + i * (cols / 2) + 8 * j, sf + i * (cols / 16) + j, NULL,",
        "quantize_block(xb, gs, r, codes + i * (cols / 2) + 8 * ((j + 1) % (cols / 16)),\n"
        "                     sf + i * (cols / 16) + ((j + 1) % (cols / 16)), NULL,"),
    "kv_quantize_ignores_recipe": (
        "quantize_block(xb, gs, r, codes + i * (cols / 2)", "quantize_block(xb, gs, NULL, codes + i * (cols / 2)"),
    "kv_dequantize_nibble_order": (
        "uint32_t code = (d % 2 == 0) ? (byte & 0xFu) : (byte >> 4);\n      out[i * cols + d]",
        "uint32_t code = (d % 2 == 1) ? (byte & 0xFu) : (byte >> 4);\n      out[i * cols + d]"),
    "kv_dequantize_scale_of_next_block": (
        "dequant_value(code, sf[i * (cols / 16) + d / 16], gs, out_bf16);",
        "dequant_value(code, sf[i * (cols / 16) + ((d / 16) + 1) % (cols / 16)], gs, out_bf16);"),
    "materialize_applies_nothing": (
        "double w = oracle_e2m1_decode(code) * oracle_e4m3_decode(sf[si]);",
        "double w = oracle_e2m1_decode(code);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    with open(SRC) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    so = O.compile_source(str(path), str(tmp_path / "libmutant.so"))
    O.use(O.load(so))
    try:
        caught = None
        for pin in pins.ALL_PINS:
            try:
                pin(O)
            except AssertionError:
                caught = pin.__name__
                break
        assert caught is not None, f"no pin notices mutant {name}"
    finally:
        O.use(None)
