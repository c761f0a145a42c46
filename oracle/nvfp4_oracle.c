/*
 * nvfp4_oracle.c -- plain, slow CPU oracle for the NVFP4 paged KV-cache operations.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the benchmark's CPU
 * baseline leg may load this library. The product (the CUDA library) never calls it and
 * shares no code, header, table or constant with it.
 *
 * Sources (FlashInfer documentation pages):
 *   [P1] "flashinfer.quantization.nvfp4_kv_dequantize_paged" -- description, parameters.
 *   [P2] "flashinfer.page.nvfp4_quantize_append_paged_kv_cache" -- description, parameters, note.
 *   [P3] "flashinfer.quantization.kernels.nvfp4_kv_materialize.nvfp4_kv_materialize_fp8"
 *        -- parameters, returns, note.
 *   [P4] "flashinfer.quantization" API index -- "NVFP4 4over6 Recipes" section,
 *        "Precedence" note, "NVFP4KVMaterializer" class.
 *   [P5] "flashinfer.quantization" API index -- "FP4 KV Cache Quantization" section:
 *        nvfp4_kv_quantize / nvfp4_kv_dequantize (contiguous, linear block-scale layout).
 *
 * Conventions the pages leave open, fixed here (each is one reading, stated where used):
 *   - E2M1 grid {0,0.5,1,1.5,2,3,4,6}, round-to-nearest-even, saturating at 6, sign kept
 *     (a negative value that rounds to zero gives code 0x8).
 *   - E4M3 (e4m3fn): bias 7, 3 fraction bits, subnormals down to 2^-9, largest finite 448,
 *     round-to-nearest-even, saturating at 448.
 *   - Packed byte = code of element 2k in the low nibble, element 2k+1 in the high nibble.
 *   - Floating-point arithmetic is IEEE binary32 with round-to-nearest-even per operation
 *     and no contraction (this file must be compiled with -ffp-contract=off), except where
 *     a fused multiply-add is written out explicitly with fmaf()/fma().
 *
 * Every function is a loop nest that follows the per-element definition; the only
 * parallelism is an OpenMP "parallel for" over independent rows or pages, which does not
 * change any result.
 *
 * Pinning (tests/pins.py, tests/test_oracle_mutants.py): the formats against library
 * casts and brute force; the block quantization against exact rational arithmetic; the
 * paged addressing against numpy views of the documented tensor shapes; dequant and the
 * FP8 copy against numpy binary32 arithmetic over every (code, scale) pair.
 * Parity unpinned, in part: four readings have no outside reference -- the reciprocal form
 * of the element scaling x * (1/(S*gs)), the order of the 4over6 error sum, and the
 * rounding steps of the 4over6 element error in binary32 (one fused rounding) and in
 * binary16 (operands rounded to binary16, then one fused rounding). The pins fix every
 * result whose rounding decisions are clear of a midpoint and whose candidate errors are
 * not near-tied; the outcomes inside those bands follow the readings alone. An independent
 * restatement of the readings (tests/pins.py, exact rational arithmetic) checks that this
 * file computes them as stated.
 * Parity unpinned: the 4-token-interleaved V-scale layout of the materialize input. The
 * pages name it without defining it; the reading (interleaved4_sf_offset) is pinned only
 * against a second expression of itself, the layout writer in oracle/__init__.py.
 */
#include <float.h>
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_API __attribute__((visibility("default")))

/* ------------------------------------------------------------------------------------- */
/* Number formats, written from their definitions.                                        */
/* ------------------------------------------------------------------------------------- */

/* Magnitude of a binary floating-point code with `ebits` exponent bits, `mbits` fraction
 * bits and exponent bias `bias`: exponent field 0 is the subnormal range
 * 0.m * 2^(1-bias), otherwise 1.m * 2^(e-bias). Special encodings are handled by callers. */
static double fmt_decode_mag(uint32_t bits, int ebits, int mbits, int bias) {
  uint32_t m = bits & ((1u << mbits) - 1u);
  uint32_t e = (bits >> mbits) & ((1u << ebits) - 1u);
  if (e == 0) return ldexp((double)m, 1 - bias - mbits);
  return ldexp((double)((1u << mbits) | m), (int)e - bias - mbits);
}

/* Round a >= 0 to the nearest number with `mbits` fraction bits whose exponent is at
 * least `emin` (below 2^emin the spacing stays 2^(emin-mbits): the subnormal range).
 * Ties go to the even significand. No upper limit is applied here. */
static double fmt_round_mag(double a, int mbits, int emin) {
  if (a == 0.0) return 0.0;
  int e;
  (void)frexp(a, &e);
  e -= 1; /* 2^e <= a < 2^(e+1) */
  if (e < emin) e = emin;
  double q = ldexp(1.0, e - mbits); /* spacing of representable numbers around a */
  double n = a / q;                 /* exact: q is a power of two */
  double fl = floor(n);
  double fr = n - fl;
  if (fr > 0.5 || (fr == 0.5 && fmod(fl, 2.0) == 1.0)) fl += 1.0;
  return fl * q;
}

/* Bits (without sign) of a representable finite magnitude v. */
static uint32_t fmt_encode_mag(double v, int mbits, int bias) {
  if (v == 0.0) return 0;
  int e;
  (void)frexp(v, &e);
  e -= 1;
  int emin = 1 - bias;
  if (e < emin) return (uint32_t)ldexp(v, mbits - emin); /* subnormal: v / 2^(emin-mbits) */
  double frac = ldexp(v, -e) - 1.0;                      /* in [0, 1) */
  return ((uint32_t)(e + bias) << mbits) | (uint32_t)ldexp(frac, mbits);
}

/* E2M1: 1 sign, 2 exponent, 1 fraction bit, bias 1, no special values. */
ORACLE_API double oracle_e2m1_decode(uint32_t code) {
  double mag = fmt_decode_mag(code & 7u, 2, 1, 1);
  return (code & 8u) ? -mag : mag;
}

/* Round-to-nearest-even onto the E2M1 grid, saturating at 6, keeping the sign. */
ORACLE_API uint32_t oracle_e2m1_encode(double v) {
  uint32_t s = signbit(v) ? 8u : 0u;
  double a = fmt_round_mag(fabs(v), 1, 0);
  if (a > 6.0) a = 6.0;
  return s | fmt_encode_mag(a, 1, 1);
}

/* E4M3 (e4m3fn): bias 7, 3 fraction bits; S.1111.111 is NaN, there are no infinities. */
ORACLE_API double oracle_e4m3_decode(uint32_t byte) {
  if ((byte & 0x7Fu) == 0x7Fu) return NAN;
  double mag = fmt_decode_mag(byte & 0x7Fu, 4, 3, 7);
  return (byte & 0x80u) ? -mag : mag;
}

/* Round-to-nearest-even onto E4M3, saturating at +-448; NaN stays NaN (0x7F). */
ORACLE_API uint32_t oracle_e4m3_encode(double v) {
  if (isnan(v)) return 0x7Fu;
  uint32_t s = signbit(v) ? 0x80u : 0u;
  double a = fmt_round_mag(fabs(v), 3, -6);
  if (a > 448.0) a = 448.0;
  return s | fmt_encode_mag(a, 3, 7);
}

/* IEEE binary16: 5 exponent, 10 fraction bits, bias 15. */
ORACLE_API double oracle_f16_decode(uint32_t bits) {
  uint32_t e = (bits >> 10) & 0x1Fu;
  double mag;
  if (e == 0x1Fu) mag = (bits & 0x3FFu) ? NAN : INFINITY;
  else mag = fmt_decode_mag(bits & 0x7FFFu, 5, 10, 15);
  return (bits & 0x8000u) ? -mag : mag;
}

/* Round-to-nearest-even to binary16; results above the largest finite value are Inf. */
ORACLE_API uint32_t oracle_f16_encode(double v) {
  if (isnan(v)) return 0x7E00u;
  uint32_t s = signbit(v) ? 0x8000u : 0u;
  double a = isinf(v) ? INFINITY : fmt_round_mag(fabs(v), 10, -14);
  if (a > 65504.0) return s | 0x7C00u;
  return s | fmt_encode_mag(a, 10, 15);
}

/* bfloat16: 8 exponent, 7 fraction bits, bias 127. */
ORACLE_API double oracle_bf16_decode(uint32_t bits) {
  uint32_t e = (bits >> 7) & 0xFFu;
  double mag;
  if (e == 0xFFu) mag = (bits & 0x7Fu) ? NAN : INFINITY;
  else mag = fmt_decode_mag(bits & 0x7FFFu, 8, 7, 127);
  return (bits & 0x8000u) ? -mag : mag;
}

/* Round-to-nearest-even to bfloat16; results above the largest finite value are Inf. */
ORACLE_API uint32_t oracle_bf16_encode(double v) {
  if (isnan(v)) return 0x7FC0u;
  uint32_t s = signbit(v) ? 0x8000u : 0u;
  double a = isinf(v) ? INFINITY : fmt_round_mag(fabs(v), 7, -126);
  if (a > ldexp(255.0, 120)) return s | 0x7F80u; /* (2 - 2^-7) * 2^127 */
  return s | fmt_encode_mag(a, 7, 127);
}

/* binary16 rounding of a double, returned as a double (NaN propagates). */
static double f16_round(double v) { return oracle_f16_decode(oracle_f16_encode(v)); }

/* ------------------------------------------------------------------------------------- */
/* Recipes ([P4] "NVFP4 4over6 Recipes").                                                 */
/* ------------------------------------------------------------------------------------- */

typedef struct {
  float e4m3_max;            /* top of the block-scale range ("e4m3_max" knob) */
  int32_t err_mode;          /* 0 = summed absolute error, 1 = summed squared error */
  int32_t err_use_fast_math; /* 1 = evaluate the error in binary16 */
} oracle_recipe;

/* Block-scale clamp implied by a recipe ([P4] nvfp4_e4m3_max): 448 for standard NVFP4
 * (no recipe), the recipe's e4m3_max under 4over6. */
ORACLE_API float oracle_e4m3_max(const oracle_recipe* r) { return r ? r->e4m3_max : 448.0f; }

/* Exact value of one 16-bit input element. */
static float in_value(const uint16_t* x, int64_t i, int is_bf16) {
  return is_bf16 ? (float)oracle_bf16_decode(x[i]) : (float)oracle_f16_decode(x[i]);
}

/* Global decode scale for one tensor ([P4] make_nvfp4_global_scale, per-tensor form):
 *   gs = amax(|x|) / (6 * e4m3_max), amax exact, 6*e4m3_max and the quotient each rounded
 *   to binary32. 6 is the largest E2M1 magnitude ([P4] 4over6 recipes). Reading: an
 *   all-zero tensor gets gs = 1. */
ORACLE_API float oracle_global_scale(const uint16_t* x, int is_bf16, int64_t numel,
                                     const oracle_recipe* r) {
  float amax = 0.0f;
  for (int64_t i = 0; i < numel; ++i) {
    float a = fabsf(in_value(x, i, is_bf16));
    if (a > amax) amax = a;
  }
  if (amax == 0.0f) return 1.0f;
  float denom = 6.0f * oracle_e4m3_max(r);
  return amax / denom;
}

/* ------------------------------------------------------------------------------------- */
/* One 16-element block ([P2] description; [P4] 4over6 recipes).                          */
/* ------------------------------------------------------------------------------------- */

/* Element codes of a block for block-scale byte s: each element is multiplied by the
 * reciprocal of its decode factor S*gs and rounded onto the E2M1 grid. Reading: one
 * binary32 reciprocal per block, 0 when S*gs is 0, clamped to FLT_MAX when it overflows. */
static void encode_block(const float x[16], uint32_t s, float gs, uint32_t q[16]) {
  float S = (float)oracle_e4m3_decode(s);
  float den = S * gs;
  float inv = 0.0f;
  if (den != 0.0f) {
    inv = 1.0f / den;
    if (inv > FLT_MAX) inv = FLT_MAX;
  }
  for (int i = 0; i < 16; ++i) {
    float y = x[i] * inv;
    q[i] = oracle_e2m1_encode(y);
  }
}

/* Sum of 16 terms by halving strides: t[i] += t[i+8], then t[i] += t[i+4], t[i+2], t[i+1].
 * Reading: the pages do not fix the order; this fixed balanced tree makes it exact. */
static float tree16_f32(float t[16]) {
  for (int half = 8; half >= 1; half /= 2)
    for (int i = 0; i < half; ++i) t[i] = t[i] + t[i + half];
  return t[0];
}

static double tree16_f16(double t[16]) {
  for (int half = 8; half >= 1; half /= 2)
    for (int i = 0; i < half; ++i) t[i] = f16_round(t[i] + t[i + half]);
  return t[0];
}

/* Reconstruction error of a candidate ([P4]: each candidate is quantized and then
 * dequantized, and the reconstructions are compared). One rule in both precisions: the
 * element error is the residual x - e2m1(q)*S*gs, formed from operands of the evaluation's
 * precision and rounded once to that precision (a fused multiply-add), the product taken in
 * the order the decode rule is written, (e2m1 value * block scale) * global scale ([P2] k_scale
 * / v_scale parameter: e2m1_value * block_scale * global_scale).
 *   binary32 (the default, which [P4] calls exact): e = RN32(x - (e2m1(q)*S)*gs); e2m1*S is
 *     exact in binary32, so the one rounding is that of the residual.
 *   binary16 ([P4] err_use_fast_math, the error evaluated in fp16): the operands become
 *     binary16 first, x_h = RN16(x) and g_h = RN16(gs) (e2m1*S is exact in binary16), and
 *     e = RN16(x_h - (e2m1(q)*S)*g_h).
 * The summed term is |e| (MAE) or e*e rounded to the precision (MSE); the partial sums are
 * rounded to it as well. Parity unpinned: the pages fix neither the rounding steps nor the
 * association; tests/pins.py restates this reading independently, which pins this code to
 * the reading, not the reading to the pages. */
static double block_error(const float x[16], const uint32_t q[16], uint32_t s, float gs,
                          const oracle_recipe* r) {
  double S = oracle_e4m3_decode(s);
  int mse = r->err_mode == 1;
  if (!r->err_use_fast_math) {
    float t[16];
    for (int i = 0; i < 16; ++i) {
      float w = (float)(oracle_e2m1_decode(q[i]) * S); /* exact: at most 6 significant bits */
      float e = fmaf(-w, gs, x[i]);
      t[i] = mse ? e * e : fabsf(e);
    }
    return (double)tree16_f32(t);
  }
  double t[16];
  double gh = f16_round((double)gs);
  for (int i = 0; i < 16; ++i) {
    double xh = f16_round((double)x[i]);
    double w = oracle_e2m1_decode(q[i]) * S; /* exact: at most 6 significant bits */
    double e = f16_round(fma(-w, gh, xh));   /* w*gh is exact in double; one rounding */
    t[i] = mse ? f16_round(e * e) : fabs(e);
  }
  return tree16_f16(t);
}

/* Quantize one block of 16 exact input values with global decode scale gs.
 *   Standard NVFP4: scale from amax/6 ([P4]): S_A = E4M3(min(amax / (6*gs), e4m3_max)).
 *   4over6: also S_B = E4M3(min(amax / (4*gs), 448)) -- the 1.5x tighter amax/4 scale,
 *   which the e4m3_max knob keeps representable ([P4] e4m3_max=256) -- quantize and
 *   dequantize with both and keep B only when its error is strictly smaller (reading:
 *   ties keep amax/6). Outputs 8 packed bytes and the block-scale byte. */
static int quantize_block(const float x[16], float gs, const oracle_recipe* r,
                          uint8_t codes[8], uint8_t* sf, double* err_a, double* err_b) {
  float amax = 0.0f;
  for (int i = 0; i < 16; ++i) {
    float a = fabsf(x[i]);
    if (a > amax) amax = a;
  }
  float cap_a = oracle_e4m3_max(r);
  float g6 = 6.0f * gs;
  float ra = amax / g6;
  if (ra > cap_a) ra = cap_a;
  uint32_t sa = oracle_e4m3_encode(ra);
  uint32_t qa[16];
  encode_block(x, sa, gs, qa);
  uint32_t s = sa;
  const uint32_t* q = qa;
  uint32_t qb[16];
  int chose_b = 0;
  if (r) {
    float g4 = 4.0f * gs;
    float rb = amax / g4;
    if (rb > 448.0f) rb = 448.0f;
    uint32_t sb = oracle_e4m3_encode(rb);
    encode_block(x, sb, gs, qb);
    double ea = block_error(x, qa, sa, gs, r);
    double eb = block_error(x, qb, sb, gs, r);
    if (err_a) *err_a = ea;
    if (err_b) *err_b = eb;
    if (eb < ea) {
      s = sb;
      q = qb;
      chose_b = 1;
    }
  }
  for (int k = 0; k < 8; ++k) codes[k] = (uint8_t)(q[2 * k] | (q[2 * k + 1] << 4));
  *sf = (uint8_t)s;
  return chose_b;
}

/* Block-level entry for tests: x16 holds 16 raw fp16/bf16 values. Returns 1 when the
 * amax/4 candidate was kept; err_a/err_b (nullable) receive the two candidate errors. */
ORACLE_API int oracle_quantize_block(const uint16_t* x16, int is_bf16, float gs,
                                     const oracle_recipe* r, uint8_t* codes8, uint8_t* sf,
                                     double* err_a, double* err_b) {
  float x[16];
  for (int i = 0; i < 16; ++i) x[i] = in_value(x16, i, is_bf16);
  return quantize_block(x, gs, r, codes8, sf, err_a, err_b);
}

/* ------------------------------------------------------------------------------------- */
/* Paged addressing ([P1]/[P2] parameters: NHD [pages, page_size, heads, .] and HND       */
/* [pages, heads, page_size, .]; a page may be strided more widely than it is long).      */
/* ------------------------------------------------------------------------------------- */

static int64_t row_index_in_page(int layout, int64_t slot, int64_t h, int64_t ps, int64_t H) {
  return layout == 0 ? slot * H + h : h * ps + slot;
}

/* Byte offsets of (page, slot, head) in the packed cache and in the scale cache. */
ORACLE_API void oracle_row_offsets(int layout, int64_t page, int64_t slot, int64_t h, int64_t ps,
                                   int64_t H, int64_t D, int64_t data_page_stride,
                                   int64_t sf_page_stride, int64_t* data_off, int64_t* sf_off) {
  int64_t r = row_index_in_page(layout, slot, h, ps, H);
  *data_off = page * data_page_stride + r * (D / 2);
  *sf_off = page * sf_page_stride + r * (D / 16);
}

/* ------------------------------------------------------------------------------------- */
/* Quantize-and-append ([P2]).                                                           */
/* ------------------------------------------------------------------------------------- */

/* Row i of the appended tensor goes to logical position positions[i] of request
 * batch_indices[i]; that position lives in page kv_indices[kv_indptr[b] + pos / ps] at
 * slot pos % ps. Each of the D/16 blocks of every (row, head) is quantized independently. */
static void append_one(const uint16_t* x, int is_bf16, int64_t nnz, int64_t H, int64_t D,
                       int64_t row_stride, const int32_t* batch_indices,
                       const int32_t* positions, uint8_t* data, uint8_t* sf,
                       int64_t data_page_stride, int64_t sf_page_stride, int64_t ps, int layout,
                       const int32_t* kv_indices, const int32_t* kv_indptr, float gs,
                       const oracle_recipe* r, int nthreads) {
  (void)nthreads;
#pragma omp parallel for schedule(static) num_threads(nthreads)
  for (int64_t i = 0; i < nnz; ++i) {
    int64_t b = batch_indices[i];
    int64_t pos = positions[i];
    int64_t page = kv_indices[kv_indptr[b] + pos / ps];
    int64_t slot = pos % ps;
    for (int64_t h = 0; h < H; ++h) {
      int64_t doff, soff;
      oracle_row_offsets(layout, page, slot, h, ps, H, D, data_page_stride, sf_page_stride,
                         &doff, &soff);
      for (int64_t j = 0; j < D / 16; ++j) {
        float xb[16];
        for (int k = 0; k < 16; ++k) xb[k] = in_value(x, i * row_stride + h * D + 16 * j + k, is_bf16);
        quantize_block(xb, gs, r, data + doff + 8 * j, sf + soff + j, NULL, NULL);
      }
    }
  }
}

ORACLE_API void oracle_quantize_append_paged(
    const uint16_t* k, const uint16_t* v, int is_bf16, int64_t nnz, int32_t H, int32_t D,
    int64_t k_row_stride, int64_t v_row_stride, const int32_t* batch_indices,
    const int32_t* positions, uint8_t* k_data, uint8_t* k_sf, int64_t k_data_page_stride,
    int64_t k_sf_page_stride, uint8_t* v_data, uint8_t* v_sf, int64_t v_data_page_stride,
    int64_t v_sf_page_stride, int32_t ps, int32_t layout, const int32_t* kv_indices,
    const int32_t* kv_indptr, float k_scale, float v_scale, const oracle_recipe* r,
    int32_t nthreads) {
  append_one(k, is_bf16, nnz, H, D, k_row_stride, batch_indices, positions, k_data, k_sf,
             k_data_page_stride, k_sf_page_stride, ps, layout, kv_indices, kv_indptr, k_scale,
             r, nthreads);
  append_one(v, is_bf16, nnz, H, D, v_row_stride, batch_indices, positions, v_data, v_sf,
             v_data_page_stride, v_sf_page_stride, ps, layout, kv_indices, kv_indptr, v_scale,
             r, nthreads);
}

/* ------------------------------------------------------------------------------------- */
/* Paged dequantize ([P1]).                                                              */
/* ------------------------------------------------------------------------------------- */

/* out = round_out( (e2m1(q) * S) * gs ): the first product is exact in binary32, the second
 * is rounded to binary32, then one final rounding to the output type
 * ([P2]: value = e2m1_value * block_scale * global_scale). */
static uint16_t dequant_value(uint32_t code, uint32_t s, float gs, int out_bf16) {
  float w = (float)(oracle_e2m1_decode(code) * oracle_e4m3_decode(s));
  float d = w * gs;
  return (uint16_t)(out_bf16 ? oracle_bf16_encode(d) : oracle_f16_encode(d));
}

static void dequant_one(const uint8_t* data, const uint8_t* sf, int64_t data_page_stride,
                        int64_t sf_page_stride, int64_t ps, int64_t H, int64_t D, int layout,
                        const void* block_tables, int bt_i64, int64_t max_pages,
                        const int32_t* seq_lens, int64_t B, float gs, uint16_t* out,
                        int out_bf16, int64_t max_seq_len, int nthreads) {
  (void)nthreads;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
  for (int64_t b = 0; b < B; ++b) {
    int64_t len = seq_lens[b] < max_seq_len ? seq_lens[b] : max_seq_len;
    for (int64_t t = 0; t < len; ++t) {
      int64_t col = b * max_pages + t / ps;
      int64_t page = bt_i64 ? ((const int64_t*)block_tables)[col]
                            : (int64_t)((const int32_t*)block_tables)[col];
      int64_t slot = t % ps;
      for (int64_t h = 0; h < H; ++h) {
        int64_t doff, soff;
        oracle_row_offsets(layout, page, slot, h, ps, H, D, data_page_stride, sf_page_stride,
                           &doff, &soff);
        uint16_t* o = out + ((b * max_seq_len + t) * H + h) * D;
        for (int64_t d = 0; d < D; ++d) {
          uint32_t byte = data[doff + d / 2];
          uint32_t code = (d % 2 == 0) ? (byte & 0xFu) : (byte >> 4);
          o[d] = dequant_value(code, sf[soff + d / 16], gs, out_bf16);
        }
      }
    }
  }
}

ORACLE_API void oracle_dequantize_paged(
    const uint8_t* k_data, const uint8_t* k_sf, int64_t k_data_page_stride,
    int64_t k_sf_page_stride, const uint8_t* v_data, const uint8_t* v_sf,
    int64_t v_data_page_stride, int64_t v_sf_page_stride, int32_t ps, int32_t H, int32_t D,
    int32_t layout, const void* block_tables, int32_t bt_i64, int32_t max_pages,
    const int32_t* seq_lens, int32_t B, float k_scale, float v_scale, uint16_t* out_k,
    uint16_t* out_v, int32_t out_bf16, int32_t max_seq_len, int32_t nthreads) {
  dequant_one(k_data, k_sf, k_data_page_stride, k_sf_page_stride, ps, H, D, layout,
              block_tables, bt_i64, max_pages, seq_lens, B, k_scale, out_k, out_bf16,
              max_seq_len, nthreads);
  dequant_one(v_data, v_sf, v_data_page_stride, v_sf_page_stride, ps, H, D, layout,
              block_tables, bt_i64, max_pages, seq_lens, B, v_scale, out_v, out_bf16,
              max_seq_len, nthreads);
}

/* ------------------------------------------------------------------------------------- */
/* FP8 materialize ([P3]; [P4] NVFP4KVMaterializer).                                     */
/* ------------------------------------------------------------------------------------- */

/* Byte offset of V block scale j of (page, head h, slot) when the V scales use the
 * 4-token-interleaved layout that the materialize parameters name (v_block_scales,
 * [num_pages, H, page_size, D/16]) without defining it. Reading: the tensor keeps that
 * shape; within head h's slice of a page the slots go in groups of four (page_size % 4 == 0
 * is the materializer's requirement), and a group stores block 0 of its four slots, then
 * block 1, and so on, slot-minor. Parity unpinned: the pages give no example of the
 * layout. */
static int64_t interleaved4_sf_offset(int64_t page, int64_t h, int64_t slot, int64_t j,
                                      int64_t ps, int64_t nb, int64_t sf_page_stride) {
  int64_t group = slot / 4, lane = slot % 4;
  return page * sf_page_stride + (h * ps + group * 4) * nb + j * 4 + lane;
}

/* Output shape [num_pages+1, 2, H, ps, D] float8_e4m3fn. Request b's page j goes to out page
 * o = base_b + j + 1 with base_b = kv_page_indptr[b] (or b * mpps without it); only
 * E2M1 value times E4M3 block scale is applied, rounded to E4M3 (reading: saturating at 448).
 * Page 0 is zero. fp8_block_tables[b, j] = o for the active pages; with zero_tables the other
 * entries are 0 (functional form), otherwise they are left alone (run() form). Reading: every
 * slot of an active page is converted, the copy being page-granular. Reading: a length above
 * mpps*ps is clamped to it. v_sf_layout 1: the V scales are read in the 4-token-interleaved
 * layout above (HND only; K scales stay linear), 0: linear. */
ORACLE_API void oracle_materialize_fp8(
    const uint8_t* k_data, const uint8_t* k_sf, int64_t k_data_page_stride,
    int64_t k_sf_page_stride, const uint8_t* v_data, const uint8_t* v_sf,
    int64_t v_data_page_stride, int64_t v_sf_page_stride, int32_t ps, int32_t H, int32_t D,
    int32_t layout, const int32_t* block_tables, int32_t max_num_pages, int32_t shared,
    const int32_t* seq_lens, int32_t B, int32_t max_kv_len, const int32_t* kv_page_indptr,
    uint8_t* out, int32_t* fp8_block_tables, int32_t zero_tables, int32_t v_sf_layout,
    int32_t nthreads) {
  int64_t mpps = ((int64_t)max_kv_len + ps - 1) / ps;
  int64_t page_elems = (int64_t)H * ps * D; /* one of K or V of an output page */
  memset(out, 0, (size_t)(2 * page_elems));
  (void)nthreads;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
  for (int64_t b = 0; b < B; ++b) {
    int64_t len = seq_lens[b];
    int64_t np = (len + ps - 1) / ps;
    if (np > mpps) np = mpps;
    int64_t base = kv_page_indptr ? kv_page_indptr[b] : b * mpps;
    for (int64_t j = 0; j < mpps; ++j) {
      if (j < np) fp8_block_tables[b * mpps + j] = (int32_t)(base + j + 1);
      else if (zero_tables) fp8_block_tables[b * mpps + j] = 0;
    }
    for (int64_t j = 0; j < np; ++j) {
      int64_t o = base + j + 1;
      for (int kv = 0; kv < 2; ++kv) {
        int64_t col = shared ? b * max_num_pages + j : (b * 2 + kv) * max_num_pages + j;
        int64_t page = block_tables[col];
        const uint8_t* data = kv ? v_data : k_data;
        const uint8_t* sf = kv ? v_sf : k_sf;
        int64_t dps = kv ? v_data_page_stride : k_data_page_stride;
        int64_t sps = kv ? v_sf_page_stride : k_sf_page_stride;
        uint8_t* dst = out + (o * 2 + kv) * page_elems;
        for (int64_t h = 0; h < H; ++h) {
          for (int64_t slot = 0; slot < ps; ++slot) {
            int64_t doff, soff;
            oracle_row_offsets(layout, page, slot, h, ps, H, D, dps, sps, &doff, &soff);
            for (int64_t d = 0; d < D; ++d) {
              uint32_t byte = data[doff + d / 2];
              uint32_t code = (d % 2 == 0) ? (byte & 0xFu) : (byte >> 4);
              int64_t si = (kv == 1 && v_sf_layout == 1)
                               ? interleaved4_sf_offset(page, h, slot, d / 16, ps, D / 16, sps)
                               : soff + d / 16;
              double w = oracle_e2m1_decode(code) * oracle_e4m3_decode(sf[si]);
              dst[(h * ps + slot) * D + d] = (uint8_t)oracle_e4m3_encode(w);
            }
          }
        }
      }
    }
  }
}

/* Number of OpenMP threads a parallel region would use (1 without OpenMP). */
ORACLE_API int32_t oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ------------------------------------------------------------------------------------- */
/* Contiguous quantize and dequantize ([P5]).                                            */
/* ------------------------------------------------------------------------------------- */

/* nvfp4_kv_quantize: the same per-block rule as the append, on a plain [rows, cols] tensor
 * (any leading dimensions flattened into rows). Reading: output codes [rows, cols/2] and
 * scales [rows, cols/16], both row-major, i.e. the linear block-scale layout the section
 * names; the recipe applies as for every NVFP4 entry point ([P4], "Precedence"). */
ORACLE_API void oracle_kv_quantize(const uint16_t* x, int is_bf16, int64_t rows, int64_t cols,
                                   int64_t row_stride, float gs, const oracle_recipe* r,
                                   uint8_t* codes, uint8_t* sf, int32_t nthreads) {
  (void)nthreads;
#pragma omp parallel for schedule(static) num_threads(nthreads)
  for (int64_t i = 0; i < rows; ++i) {
    for (int64_t j = 0; j < cols / 16; ++j) {
      float xb[16];
      for (int k = 0; k < 16; ++k) xb[k] = in_value(x, i * row_stride + 16 * j + k, is_bf16);
      quantize_block(xb, gs, r, codes + i * (cols / 2) + 8 * j, sf + i * (cols / 16) + j, NULL,
                     NULL);
    }
  }
}

/* nvfp4_kv_dequantize: every element of the [rows, cols] codes decodes with its block's
 * scale and the global scale, exactly as a paged dequant ([P2] decode rule). */
ORACLE_API void oracle_kv_dequantize(const uint8_t* codes, const uint8_t* sf, int64_t rows,
                                     int64_t cols, float gs, uint16_t* out, int32_t out_bf16,
                                     int32_t nthreads) {
  (void)nthreads;
#pragma omp parallel for schedule(static) num_threads(nthreads)
  for (int64_t i = 0; i < rows; ++i) {
    for (int64_t d = 0; d < cols; ++d) {
      uint32_t byte = codes[i * (cols / 2) + d / 2];
      uint32_t code = (d % 2 == 0) ? (byte & 0xFu) : (byte >> 4);
      out[i * cols + d] = dequant_value(code, sf[i * (cols / 16) + d / 16], gs, out_bf16);
    }
  }
}
