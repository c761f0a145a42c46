// append.cu -- quantize-and-append into a paged NVFP4 cache.
//
// FlashInfer "flashinfer.page.nvfp4_quantize_append_paged_kv_cache" (description,
// parameters, note) and the "NVFP4 4over6 Recipes" section of the "flashinfer.quantization"
// index (two-candidate block-scale search, e4m3_max, err_mode, err_use_fast_math).
//
// One thread quantizes one 16-element block of one (token, head) row, for K and for V: the
// two blocks share the destination lookup and give the thread two independent chains of
// work. The main kernel is fed by a TMA ring (tiles of consecutive rows in shared memory);
// the direct-load kernel, for rows too long for a stage, reads the blocks from global
// memory, a warp covering 32 consecutive blocks (1 KB of contiguous input).
//
// Per block and candidate scale byte s (S = E4M3 value, gs = global decode scale):
//   inv = 1 / (S * gs)      (binary32 reciprocal; 0 when S*gs is 0; at most FLT_MAX)
//   q_i = E2M1_RNE_satfinite(x_i * inv)
// Standard NVFP4: s = E4M3(min(amax / (6 gs), e4m3_max)); the quotient is the correctly
// rounded one, from a precomputed reciprocal of 6 gs (see div_rn_with_rcp).
// 4over6: s_B = E4M3(min(amax / (4 gs), 448)) as well; each candidate's error sums, over the
// block, |e_i| (MAE) or e_i^2 (MSE):
//   binary32 error: e_i = RN32(x_i - (e2m1(q_i) * S) * gs) (e2m1 * S is exact in binary16,
//                   the rest is one fused multiply-add);
//   binary16 error: the same residual from binary16 operands, rounded once to binary16:
//                   e_i = RN16(x_h - (e2m1(q_i) * S) * g_h), x_h = RN16(x_i), g_h = RN16(gs);
//                   squares and sums rounded to binary16.
// The sum runs over a fixed halving tree: t[i] += t[i+8], t[i+4], t[i+2], t[i+1] (the
// binary16 sums run it as packed two-lane adds, pairs (2k, 2k+1)). B is kept only when its
// error is strictly smaller.
//
// Per-CTA shared tables, indexed by scale byte: 1/(S*gs) (both tensors), and (S, S) as half2
// (the 4over6 recipes).
#include <cfloat>
#include <type_traits>

#include "internal.h"
#include "pipeline.cuh"

namespace nvfp4 {
namespace {

constexpr int kThreads = 256;

// Per-tensor constants for one block quantization.
struct TensorConsts {
  float gs;       // global decode scale
  uint32_t neg_gh2;  // -RN16(gs) in both binary16 halves (binary16 error)
  float g6, r6;   // fp32(6 gs) and its reciprocal
  float g4, r4;   // 4 gs and its reciprocal
  bool exact_rcp; // both divisors and reciprocals are normal: use div_rn_with_rcp
};

__device__ __forceinline__ TensorConsts make_consts(float gs) {
  TensorConsts c;
  c.gs = gs;
  const uint32_t gh = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(gs))) ^ 0x8000u;
  c.neg_gh2 = gh | (gh << 16);
  c.g6 = __fmul_rn(6.0f, gs);
  c.g4 = __fmul_rn(4.0f, gs);
  c.r6 = __frcp_rn(c.g6);
  c.r4 = __frcp_rn(c.g4);
  const float lo = FLT_MIN, hi = FLT_MAX;
  c.exact_rcp = c.g6 >= lo && c.g6 <= hi && c.g4 >= lo && c.r6 >= lo && c.r6 <= hi &&
                c.r4 >= lo && c.r4 <= hi;
  return c;
}

// RN(a / b). EXACT: the caller knows that b and rb are normal (div_rn_with_rcp applies).
template <bool EXACT>
__device__ __forceinline__ float quotient(float a, float b, float rb, bool exact_rcp) {
  if (EXACT) return div_rn_with_rcp(a, b, rb);
  return exact_rcp ? div_rn_with_rcp(a, b, rb) : __fdiv_rn(a, b);
}

// Exact binary32 values of the 16 elements. For bf16 the low half is widened with an
// integer multiply by 2^16 (the FMA pipe) rather than a shift (the half-rate ALU pipe,
// which the E2M1 decodes already keep busy).
template <bool BF16>
__device__ __forceinline__ void unpack16(const U32x8& in, float x[16]) {
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    if (BF16) {
      uint32_t lo;
      asm("mul.lo.u32 %0, %1, 65536;" : "=r"(lo) : "r"(in.w[k]));
      x[2 * k] = __uint_as_float(lo);
      x[2 * k + 1] = f32_from_bf16_hi(in.w[k]);
    } else {
      x[2 * k] = f32_from_f16_lo(in.w[k]);
      x[2 * k + 1] = f32_from_f16_hi(in.w[k]);
    }
  }
}

// Four element pairs (x[0..7]) with multiplier inv: the four code bytes, and the decoded
// values e2m1(q) as four half2. The decodes read the bytes of the packed word (which takes
// fewer integer instructions than decoding each conversion result).
__device__ __forceinline__ uint32_t encode8(const float* x, float inv, uint32_t v[4]) {
  uint32_t code;
  asm("{\n\t"
      ".reg .b64 ip, p0, p1, p2, p3;\n\t"
      ".reg .f32 y0, y1, y2, y3, y4, y5, y6, y7;\n\t"
      ".reg .b8 q0, q1, q2, q3, r0, r1, r2, r3;\n\t"
      "mov.b64 ip, {%5, %5};\n\t"
      "mov.b64 p0, {%6, %7};\n\t"
      "mov.b64 p1, {%8, %9};\n\t"
      "mov.b64 p2, {%10, %11};\n\t"
      "mov.b64 p3, {%12, %13};\n\t"
      "mul.rn.f32x2 p0, p0, ip;\n\t"
      "mul.rn.f32x2 p1, p1, ip;\n\t"
      "mul.rn.f32x2 p2, p2, ip;\n\t"
      "mul.rn.f32x2 p3, p3, ip;\n\t"
      "mov.b64 {y0, y1}, p0;\n\t"
      "mov.b64 {y2, y3}, p1;\n\t"
      "mov.b64 {y4, y5}, p2;\n\t"
      "mov.b64 {y6, y7}, p3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q0, y1, y0;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q1, y3, y2;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q2, y5, y4;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q3, y7, y6;\n\t"
      "mov.b32 %0, {q0, q1, q2, q3};\n\t"
      "mov.b32 {r0, r1, r2, r3}, %0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, r0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, r1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, r2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %4, r3;\n\t"
      "}"
      : "=r"(code), "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
      : "f"(inv), "f"(x[0]), "f"(x[1]), "f"(x[2]), "f"(x[3]), "f"(x[4]), "f"(x[5]), "f"(x[6]),
        "f"(x[7]));
  return code;
}

// Codes of a block without the decoded values (standard NVFP4).
__device__ __forceinline__ uint32_t codes8(const float* x, float inv) {
  uint32_t code;
  asm("{\n\t"
      ".reg .b64 ip, p0, p1, p2, p3;\n\t"
      ".reg .f32 y0, y1, y2, y3, y4, y5, y6, y7;\n\t"
      ".reg .b8 q0, q1, q2, q3;\n\t"
      "mov.b64 ip, {%1, %1};\n\t"
      "mov.b64 p0, {%2, %3};\n\t"
      "mov.b64 p1, {%4, %5};\n\t"
      "mov.b64 p2, {%6, %7};\n\t"
      "mov.b64 p3, {%8, %9};\n\t"
      "mul.rn.f32x2 p0, p0, ip;\n\t"
      "mul.rn.f32x2 p1, p1, ip;\n\t"
      "mul.rn.f32x2 p2, p2, ip;\n\t"
      "mul.rn.f32x2 p3, p3, ip;\n\t"
      "mov.b64 {y0, y1}, p0;\n\t"
      "mov.b64 {y2, y3}, p1;\n\t"
      "mov.b64 {y4, y5}, p2;\n\t"
      "mov.b64 {y6, y7}, p3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q0, y1, y0;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q1, y3, y2;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q2, y5, y4;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q3, y7, y6;\n\t"
      "mov.b32 %0, {q0, q1, q2, q3};\n\t"
      "}"
      : "=r"(code)
      : "f"(inv), "f"(x[0]), "f"(x[1]), "f"(x[2]), "f"(x[3]), "f"(x[4]), "f"(x[5]), "f"(x[6]),
        "f"(x[7]));
  return code;
}

// One candidate with the binary32 error: codes c0, c1 and the error sum. The terms and the
// tree are scalar: binary32 operations split across the two FMA pipes, which measured
// faster here than the packed two-lane forms.
template <bool MSE>
__device__ __forceinline__ float candidate_f32(const float x[16], float inv, uint32_t S2,
                                               float neg_gs, uint32_t& c0, uint32_t& c1) {
  uint32_t v[8];
  c0 = encode8(x, inv, v);
  c1 = encode8(x + 8, inv, v + 4);
  float t[16];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint32_t w = hmul2_rn(v[k], S2);  // e2m1 * S, exact
    // each element error is rounded once: a fused multiply-add
    const float e0 = __fmaf_rn(f32_from_f16_lo(w), neg_gs, x[2 * k]);
    const float e1 = __fmaf_rn(f32_from_f16_hi(w), neg_gs, x[2 * k + 1]);
    t[2 * k] = MSE ? __fmul_rn(e0, e0) : fabsf(e0);
    t[2 * k + 1] = MSE ? __fmul_rn(e1, e1) : fabsf(e1);
  }
#pragma unroll
  for (int h = 8; h >= 1; h /= 2) {
#pragma unroll
    for (int i = 0; i < h; ++i) t[i] = __fadd_rn(t[i], t[i + h]);
  }
  return t[0];
}

// One candidate with the binary16 error: codes c0, c1 and the error sum (as a float).
// S2 = (S, S) and neg_gh2 = (-g_h, -g_h) as half2.
template <bool MSE>
__device__ __forceinline__ float candidate_f16(const float x[16], const uint32_t xh[8], float inv,
                                               uint32_t S2, uint32_t neg_gh2, uint32_t nzh2,
                                               uint32_t& c0, uint32_t& c1) {
  uint32_t t[8];
  c0 = encode8(x, inv, t);
  c1 = encode8(x + 8, inv, t + 4);
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint32_t w = hmul2_rn(t[k], S2);  // e2m1 * S, exact
    const uint32_t e = hfma2_rn(w, neg_gh2, xh[k]);  // x_h - w * g_h, one rounding
    if (MSE) {
      t[k] = hsq2_rn(e, nzh2);
    } else {
      asm("abs.f16x2 %0, %1;" : "=r"(t[k]) : "r"(e));
    }
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) t[k] = hadd2_rn(t[k], t[k + 4]);
  t[0] = hadd2_rn(t[0], t[2]);
  t[1] = hadd2_rn(t[1], t[3]);
  t[0] = hadd2_rn(t[0], t[1]);
  const __half s = __hadd_rn(__ushort_as_half(static_cast<unsigned short>(t[0] & 0xFFFFu)),
                             __ushort_as_half(static_cast<unsigned short>(t[0] >> 16)));
  return __half2float(s);
}

// Per-CTA tables indexed by scale byte. The binary32-error recipes read both of a
// candidate's constants with one 8-byte shared-memory load (measured faster there; the
// other recipes measured faster with separate arrays).
union Tables {
  struct {
    float inv[2][256];         // 1 / (S * gs) per tensor
    uint32_t S2[256];          // (S, S) as half2 (binary16-error recipes)
  } split;                     // standard NVFP4 and the binary16-error recipes
  uint2 pair[2][256];          // binary32-error recipes: (bits of 1 / (S * gs), (S, S) as half2)
};

struct BlockOut {
  uint32_t c0, c1, s;
};

template <bool BF16, int MODE, bool EXACT = false>
__device__ __forceinline__ BlockOut quantize_block(const U32x8& in, const TensorConsts& tc,
                                                   const Tables& tab, int kv, float cap_a,
                                                   uint32_t nz) {
  float x[16];
  unpack16<BF16>(in, x);
  // max |x|: the standard and binary16-error recipes chain three-input maxima of
  // magnitudes (8 instead of 16, off the busy integer pipe's share); the binary32-error
  // recipes fold |x| into two-input maxima
  float amax;
  if (MODE == 0 || MODE >= 3) {
    asm("max.abs.f32 %0, %1, %2, %3;" : "=f"(amax) : "f"(x[0]), "f"(x[1]), "f"(x[2]));
#pragma unroll
    for (int i = 3; i < 15; i += 2)
      asm("max.abs.f32 %0, %0, %1, %2;" : "+f"(amax) : "f"(x[i]), "f"(x[i + 1]));
    amax = fmaxf(amax, fabsf(x[15]));
  } else {
    amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
  }
  const float ra = fminf(quotient<EXACT>(amax, tc.g6, tc.r6, tc.exact_rcp), cap_a);
  BlockOut r;
  if (MODE == 0) {
    r.s = e4m3x2_from_f32(ra, 0.0f) & 0xFFu;
    const float inv = tab.split.inv[kv][r.s];
    r.c0 = codes8(x, inv);
    r.c1 = codes8(x + 8, inv);
    return r;
  }
  const float rb = fminf(quotient<EXACT>(amax, tc.g4, tc.r4, tc.exact_rcp), 448.0f);
  const uint32_t sab = e4m3x2_from_f32(ra, rb);
  // sb = sab >> 8 and sa = sab & 0xFF as multiplies (FMA pipe)
  uint32_t sb;
  asm("mul.hi.u32 %0, %1, 16777216;" : "=r"(sb) : "r"(sab));
  const uint32_t sa = sab - sb * 256u;
  uint32_t a0, a1, b0, b1;
  float ea, eb;
  if (MODE == 1 || MODE == 2) {
    const uint2 ta = tab.pair[kv][sa], tb = tab.pair[kv][sb];
    ea = candidate_f32<MODE == 2>(x, __uint_as_float(ta.x), ta.y, -tc.gs, a0, a1);
    eb = candidate_f32<MODE == 2>(x, __uint_as_float(tb.x), tb.y, -tc.gs, b0, b1);
  } else {
    uint32_t xh[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) xh[k] = BF16 ? f16x2_from_f32(x[2 * k], x[2 * k + 1]) : in.w[k];
    const uint32_t nzh2 = (nz >> 16) | nz;  // binary16 -0 in both halves
    ea = candidate_f16<MODE == 4>(x, xh, tab.split.inv[kv][sa], tab.split.S2[sa], tc.neg_gh2,
                                  nzh2, a0, a1);
    eb = candidate_f16<MODE == 4>(x, xh, tab.split.inv[kv][sb], tab.split.S2[sb], tc.neg_gh2,
                                  nzh2, b0, b1);
  }
  const bool take_b = eb < ea;
  r.c0 = take_b ? b0 : a0;
  r.c1 = take_b ? b1 : a1;
  r.s = take_b ? sb : sa;
  return r;
}

// The two global scales: from the arguments, or from device memory when given there.
// Returns false (and reports it) when a device-held scale is not positive finite.
__device__ __forceinline__ bool load_scales(const AppendArgs& a, float gs[2]) {
  gs[0] = a.gs[0];
  gs[1] = a.gs[1];
  if (a.gs_dev[0] != nullptr) {
    gs[0] = __ldg(a.gs_dev[0]);
    gs[1] = __ldg(a.gs_dev[1]);
    const bool ok = gs[0] > 0.0f && gs[0] <= FLT_MAX && gs[1] > 0.0f && gs[1] <= FLT_MAX;
    if (!ok) {
      if (threadIdx.x == 0 && blockIdx.x == 0) flag(a.status, NVFP4_DEV_BAD_SCALE);
      return false;
    }
  }
  return true;
}

// Fill the per-CTA tables for both tensors' global scales; ends with __syncthreads().
template <int MODE>
__device__ __forceinline__ void fill_tables(Tables& tab, const float gs[2]) {
  for (int s = threadIdx.x; s < 256; s += blockDim.x) {
    const uint32_t S2 = f16x2_from_e4m3x2(static_cast<uint32_t>(s) * 0x0101u);
    const float S = f32_from_f16_lo(S2);
#pragma unroll
    for (int kv = 0; kv < 2; ++kv) {
      const float den = __fmul_rn(S, gs[kv]);
      const float inv = den == 0.0f ? 0.0f : fminf(__frcp_rn(den), FLT_MAX);
      if (MODE == 1 || MODE == 2) {
        tab.pair[kv][s] = make_uint2(__float_as_uint(inv), S2);
      } else {
        tab.split.inv[kv][s] = inv;
        if (kv == 0) tab.split.S2[s] = S2;
      }
    }
  }
  __syncthreads();
}

// Destination of appended row i: request batch_indices[i], logical position positions[i],
// page kv_indices[kv_indptr[b] + pos / page_size], slot pos % page_size. Rows outside the
// described space or with a page outside a pool are reported and marked invalid.
struct RowMeta {
  int32_t page;   // physical page (valid only with flags bit 0 / bit 1)
  int32_t slot;   // slot inside the page
  int32_t flags;  // bit 0: K page valid, bit 1: V page valid
  int32_t pad;
};

__device__ __forceinline__ RowMeta resolve_row(const AppendArgs& a, int64_t i) {
  RowMeta m{0, 0, 0, 0};
  const int32_t b = __ldg(a.batch_indices + i);
  const int32_t pos = __ldg(a.positions + i);
  if (b < 0 || b >= a.batch_size) {
    flag(a.status, NVFP4_DEV_BAD_BATCH);
    return m;
  }
  const int64_t start = __ldg(a.kv_indptr + b);
  const int64_t npages = static_cast<int64_t>(__ldg(a.kv_indptr + b + 1)) - start;
  const int64_t lp = pos >= 0 ? div_q(pos, a.div_ps) : -1;
  bool ok = pos >= 0 && lp < npages && start >= 0 && start + lp < a.num_kv_indices;
  if (ok && a.kv_last_page_len) ok = pos < (npages - 1) * a.ps + __ldg(a.kv_last_page_len + b);
  if (!ok) {
    flag(a.status, NVFP4_DEV_BAD_POSITION);
    return m;
  }
  const int64_t page = __ldg(a.kv_indices + start + lp);
  m.page = static_cast<int32_t>(page);
  m.slot = static_cast<int32_t>(pos - lp * a.ps);
  const bool kok = page >= 0 && page < a.kc.num_pages;
  const bool vok = page >= 0 && page < a.vc.num_pages;
  if (!kok || !vok) flag(a.status, NVFP4_DEV_BAD_PAGE);
  m.flags = (kok ? 1 : 0) | (vok ? 2 : 0);
  return m;
}

template <bool BF16, int MODE, bool VEC256>
__global__ void __launch_bounds__(kThreads) append_kernel(const AppendArgs a) {
  __shared__ Tables tab;
  float gs[2];
  if (!load_scales(a, gs)) return;
  fill_tables<MODE>(tab, gs);
  const TensorConsts tck = make_consts(gs[0]);
  const TensorConsts tcv = make_consts(gs[1]);

  const int64_t total = a.nnz * a.H * a.nb;
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t blk = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; blk < total;
       blk += step) {
    const int64_t row = div_q(blk, a.div_nb);
    const int32_t j = static_cast<int32_t>(blk - row * a.nb);
    const int64_t i = div_q(row, a.div_H);
    const int32_t h = static_cast<int32_t>(row - i * a.H);
    const int64_t col = (static_cast<int64_t>(h) * a.D + 16 * j) * 2;
    const uint8_t* pk = a.k + i * a.k_row_bytes + col;
    const uint8_t* pv = a.v + i * a.v_row_bytes + col;
    const U32x8 xk = VEC256 ? ld_nc_256(pk) : ld_nc_2x128(pk);
    U32x8 xv{};
    if (a.v != nullptr) xv = VEC256 ? ld_nc_256(pv) : ld_nc_2x128(pv);

    int64_t page = i, slot = 0;  // contiguous form: row i is "page" i (stride H*D/2)
    if (!a.contig) {
      const int32_t b = __ldg(a.batch_indices + i);
      const int32_t pos = __ldg(a.positions + i);
      if (b < 0 || b >= a.batch_size) {
        flag(a.status, NVFP4_DEV_BAD_BATCH);
        continue;
      }
      const int64_t start = __ldg(a.kv_indptr + b);
      const int64_t npages = static_cast<int64_t>(__ldg(a.kv_indptr + b + 1)) - start;
      const int64_t lp = pos >= 0 ? div_q(pos, a.div_ps) : -1;
      bool ok = pos >= 0 && lp < npages && start >= 0 && start + lp < a.num_kv_indices;
      if (ok && a.kv_last_page_len)
        ok = pos < (npages - 1) * a.ps + __ldg(a.kv_last_page_len + b);
      if (!ok) {
        flag(a.status, NVFP4_DEV_BAD_POSITION);
        continue;
      }
      page = __ldg(a.kv_indices + start + lp);
      slot = pos - lp * a.ps;
    }
    const int64_t r = a.layout == NVFP4_NHD ? slot * a.H + h : static_cast<int64_t>(h) * a.ps + slot;

#pragma unroll
    for (int kv = 0; kv < 2; ++kv) {
      if (kv == 1 && a.v == nullptr) continue;
      const nvfp4_paged_cache& c = kv ? a.vc : a.kc;
      if (page < 0 || page >= c.num_pages) {
        flag(a.status, NVFP4_DEV_BAD_PAGE);
        continue;
      }
      const BlockOut q =
          quantize_block<BF16, MODE>(kv ? xv : xk, kv ? tcv : tck, tab, kv, a.cap_a, a.neg_zero);
      uint8_t* dst = c.data + page * c.data_page_stride + r * (a.D / 2) + 8 * j;
      *reinterpret_cast<uint2*>(dst) = make_uint2(q.c0, q.c1);
      c.sf[page * c.sf_page_stride + r * a.nb + j] = static_cast<uint8_t>(q.s);
    }
  }
}

// ---- TMA-fed variant ------------------------------------------------------------------
//
// A tile is `rows` consecutive appended tokens, all heads, of K and of V. The producer warp
// resolves the destination page of each row (one lane per row, so the dependent index
// loads overlap), writes it into the stage, and bulk-copies the tile's K and V rows into
// shared memory. The consumer warps quantize blocks straight from shared memory: thread k
// of a tile takes block k of K and block k of V (a row's blocks are contiguous there).

// Destination of one appended row in both caches, resolved once per row by the producer:
// the addresses of (page, slot, head 0, block 0) in the K and V codes and scales; null when
// the row or its page is invalid. Head h, block j of the row is at
// base + h * head_step + {8 j | j}.
struct RowDst {
  uint8_t* kd;
  uint8_t* ks;
  uint8_t* vd;
  uint8_t* vs;
};

template <bool CONTIG>
__device__ __forceinline__ RowDst resolve_row_dst(const AppendArgs& a, int64_t i) {
  RowDst d{nullptr, nullptr, nullptr, nullptr};
  const int64_t rd = a.layout == NVFP4_NHD ? static_cast<int64_t>(a.H) * (a.D / 2) : a.D / 2;
  const int64_t rs = a.layout == NVFP4_NHD ? static_cast<int64_t>(a.H) * a.nb : a.nb;
  if (CONTIG) {
    d.kd = a.kc.data + i * rd;
    d.ks = a.kc.sf + i * rs;
    return d;
  }
  const RowMeta m = resolve_row(a, i);
  if (m.flags & 1) {
    d.kd = a.kc.data + m.page * a.kc.data_page_stride + m.slot * rd;
    d.ks = a.kc.sf + m.page * a.kc.sf_page_stride + m.slot * rs;
  }
  if (m.flags & 2) {
    d.vd = a.vc.data + m.page * a.vc.data_page_stride + m.slot * rd;
    d.vs = a.vc.sf + m.page * a.vc.sf_page_stride + m.slot * rs;
  }
  return d;
}

struct AppendTmaLayout {
  uint32_t rows;        // tokens per tile
  uint32_t row_bytes;   // H * D * 2 (one row of one tensor)
  uint32_t nkv;         // tensors per stage: 2 (K and V), 1 for the contiguous form
  uint32_t stage_bytes; // K tile [+ V tile] + row destinations
  uint32_t tables_off, stages_off, bars_off, misc_off, total;
  int ns;
};

inline AppendTmaLayout append_tma_layout(uint32_t rows, uint32_t row_bytes, uint32_t nkv, int ns) {
  AppendTmaLayout L;
  L.rows = rows;
  L.row_bytes = row_bytes;
  L.nkv = nkv;
  L.stage_bytes = round_up(nkv * rows * row_bytes + rows * sizeof(RowDst), 128);
  L.ns = ns;
  L.tables_off = 0;
  L.stages_off = round_up(sizeof(Tables), 128);
  L.bars_off = L.stages_off + static_cast<uint32_t>(ns) * L.stage_bytes;
  L.misc_off = L.bars_off + 2u * static_cast<uint32_t>(ns) * 8u;
  // misc: abort flag, per-stage issue counts, per-stage tile index
  L.total = L.misc_off + 4u * (1u + 2u * static_cast<uint32_t>(ns));
  return L;
}

// TMA ring shape (measured): two CTAs per SM with 12-row tiles; twelve consumer warps,
// except for the binary32-error recipes (more arithmetic and registers per block), which
// run eight.
__host__ __device__ constexpr int append_consumer_warps(int mode) {
  return (mode == 1 || mode == 2) ? 8 : 12;
}
__host__ __device__ constexpr int append_threads(int mode) {
  return 32 * append_consumer_warps(mode) + 32;
}
constexpr int kAppendCtasPerSm = 2;
// Tiles a producer takes from the work queue per atomic: two consecutive tiles (measured
// faster than one or a fixed share; consecutive rows land in the same pages).
constexpr int kTilesPerFetch = 2;

// NKV: tensors per stage, 2 (K and V, paged) or 1 (the contiguous form). FIXED: a row's
// blocks divide the consumer threads (chosen at launch), so each thread keeps one (head, block).
template <bool BF16, int MODE, int NKV, bool FIXED>
__global__ void __launch_bounds__(append_threads(MODE), kAppendCtasPerSm)
    append_tma_kernel(const AppendArgs a, const AppendTmaLayout L) {
  constexpr int kConsumerWarps = append_consumer_warps(MODE);
  constexpr int kConsumers = kConsumerWarps * 32;
  constexpr uint32_t nkv = NKV;
  extern __shared__ __align__(128) uint8_t smem[];
  Tables& tab = *reinterpret_cast<Tables*>(smem + L.tables_off);
  uint8_t* stages = smem + L.stages_off;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars_off);
  uint64_t* empty = full + L.ns;
  volatile int32_t* s_abort = reinterpret_cast<int32_t*>(smem + L.misc_off);
  volatile uint32_t* s_issued = reinterpret_cast<uint32_t*>(smem + L.misc_off + 4);
  const int ns = L.ns;
  // tile of each stage (-1: no more tiles)
  volatile int32_t* s_tile = reinterpret_cast<int32_t*>(smem + L.misc_off + 4 + 4 * ns);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float gs[2];
  // uniform over the grid, before any barrier, copy or work taken from the queue
  if (!load_scales(a, gs)) return;
  const WorkQueue q = work_queue(a.workspace);
  if (threadIdx.x == 0) {
    for (int s = 0; s < ns; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, kConsumerWarps);
      s_issued[s] = 0;
    }
    *s_abort = 0;
    fence_mbar_init();
  }
  fill_tables<MODE>(tab, gs);  // ends with __syncthreads()

  const int64_t tiles = (a.nnz + L.rows - 1) / L.rows;
  const uint32_t tile_bytes = L.rows * L.row_bytes;
  const bool contiguous =
      a.k_row_bytes == L.row_bytes && (nkv == 1 || a.v_row_bytes == L.row_bytes);
  if (warp == kConsumerWarps) {
    int s = 0;
    uint32_t phase = 0, round = 0;  // phase = parity of `round`, the stage's fill count
    ItemCursor cur;
    if (lane == 0) cur.init(q, kTilesPerFetch);
    for (;;) {
      long long tile = 0;
      if (lane == 0) tile = cur.next(q, tiles);
      tile = __shfl_sync(0xFFFFFFFFu, tile, 0);
      const bool end = tile >= tiles;
      // (test control: withhold the first stage so that the consumers' wait expires)
      const bool withhold = !end && a.pipe.stall && round == 0 && s == 0;
      const int64_t row0 = end ? 0 : tile * L.rows;
      const uint32_t nrows = (end || withhold) ? 0u
          : static_cast<uint32_t>(min(static_cast<int64_t>(L.rows), a.nnz - row0));
      // Resolve this tile's destinations (a chain of dependent index loads, one row per
      // lane: at most 32 rows) while the consumers still work on the stage it will use.
      RowDst d{nullptr, nullptr, nullptr, nullptr};
      if (static_cast<uint32_t>(lane) < nrows) d = resolve_row_dst<NKV == 1>(a, row0 + lane);
      bool ok = true;
      if (lane == 0) ok = mbar_wait(empty + s, phase ^ 1u, a.pipe.wait_limit) && !*s_abort;
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) {
        if (lane == 0) {
          *s_abort = 1;
          flag(a.status, NVFP4_DEV_TIMEOUT);
        }
        break;
      }
      if (end) {
        if (lane == 0) {
          s_tile[s] = -1;
          mbar_arrive(full + s);
          s_issued[s] = round + 1;
        }
        __syncwarp();
        break;
      }
      uint8_t* st = stages + static_cast<uint32_t>(s) * L.stage_bytes;
      RowDst* dst = reinterpret_cast<RowDst*>(st + nkv * tile_bytes);
      if (static_cast<uint32_t>(lane) < nrows) dst[lane] = d;
      if (lane == 0) s_tile[s] = static_cast<int32_t>(tile);
      __syncwarp();
      if (lane == 0 && !withhold) mbar_arrive_expect_tx(full + s, nkv * nrows * L.row_bytes);
      __syncwarp();
      if (contiguous) {
        if (lane == 0 && nrows > 0) {
          bulk_g2s(st, a.k + row0 * a.k_row_bytes, nrows * L.row_bytes, full + s);
          if (nkv == 2)
            bulk_g2s(st + tile_bytes, a.v + row0 * a.v_row_bytes, nrows * L.row_bytes, full + s);
        }
      } else if (static_cast<uint32_t>(lane) < nrows) {
        const uint32_t r = lane;
        bulk_g2s(st + r * L.row_bytes, a.k + (row0 + r) * a.k_row_bytes, L.row_bytes, full + s);
        if (nkv == 2)
          bulk_g2s(st + tile_bytes + r * L.row_bytes, a.v + (row0 + r) * a.v_row_bytes,
                   L.row_bytes, full + s);
      }
      if (lane == 0 && !withhold) s_issued[s] = round + 1;
      __syncwarp();
      if (++s == ns) {
        s = 0;
        phase ^= 1u;
        ++round;
      }
    }
  } else {
    const int ct = threadIdx.x;
    const TensorConsts tck = make_consts(gs[0]);
    const TensorConsts tcv = make_consts(gs[1]);
    const int32_t row_blocks = a.H * a.nb;
    // step between heads of one row: codes, scales
    const int32_t hsd = a.layout == NVFP4_NHD ? a.D / 2 : a.ps * (a.D / 2);
    const int32_t hss = a.layout == NVFP4_NHD ? a.nb : a.ps * a.nb;
    // when a row's blocks divide the consumer count, each thread keeps one (head, block)
    constexpr bool fixed = FIXED;
    const int32_t fr0 = fixed ? ct / row_blocks : 0, frs = fixed ? kConsumers / row_blocks : 0;
    const int32_t frem = fixed ? ct - fr0 * row_blocks : 0;
    const int32_t fh = fixed ? frem / a.nb : 0, fj = fixed ? frem - fh * a.nb : 0;
    const int32_t fod = fh * hsd + 8 * fj, fos = fh * hss + fj;
    // The consumer loop is compiled twice: when both tensors' scale divisors and their
    // reciprocals are normal (every realistic global scale), the quotients need no IEEE
    // division fallback; the general form keeps it.
    auto consume = [&](auto exact_tag) {
    constexpr bool kExact = decltype(exact_tag)::value;
    int s = 0;
    uint32_t phase = 0;
    for (;;) {
      if (*s_abort || !mbar_wait(full + s, phase, a.pipe.wait_limit)) {
        if (lane == 0) {
          *s_abort = 1;
          flag(a.status, NVFP4_DEV_TIMEOUT);
        }
        break;
      }
      const int64_t tile = s_tile[s];
      if (tile < 0) break;
      const uint8_t* st = stages + static_cast<uint32_t>(s) * L.stage_bytes;
      const RowDst* dst = reinterpret_cast<const RowDst*>(st + nkv * tile_bytes);
      const int32_t nrows =
          static_cast<int32_t>(min(static_cast<int64_t>(L.rows), a.nnz - tile * L.rows));
      const int32_t nblk = nrows * row_blocks;
      for (int32_t k = ct, rf = fr0; k < nblk; k += kConsumers, rf += frs) {
        int32_t r = rf, od = fod, os = fos;
        if (!fixed) {
          r = div_q32(k, a.div_row_blocks);
          const int32_t rem = k - r * row_blocks;
          const int32_t h = div_q32(rem, a.div_nb);
          const int32_t j = rem - h * a.nb;
          od = h * hsd + 8 * j;
          os = h * hss + j;
        }
        const RowDst d = dst[r];
#pragma unroll
        for (int kv = 0; kv < NKV; ++kv) {
          uint8_t* pd = kv ? d.vd : d.kd;
          if (pd == nullptr) continue;
          const U32x8 x = ld_shared_256(st + kv * tile_bytes + 32 * k);
          const BlockOut q =
              quantize_block<BF16, MODE, kExact>(x, kv ? tcv : tck, tab, kv, a.cap_a,
                                                 a.neg_zero);
          *reinterpret_cast<uint2*>(pd + od) = make_uint2(q.c0, q.c1);
          (kv ? d.vs : d.ks)[os] = static_cast<uint8_t>(q.s);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty + s);
      if (++s == ns) {
        s = 0;
        phase ^= 1u;
      }
    }
    };
    if (tck.exact_rcp && tcv.exact_rcp) consume(std::integral_constant<bool, true>{});
    else consume(std::integral_constant<bool, false>{});
  }
  // no copy may still be landing in this CTA's shared memory when it exits
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int s = 0; s < ns; ++s)
      if (s_issued[s] > 0) mbar_wait(full + s, (s_issued[s] - 1) & 1u, a.pipe.wait_limit);
    finish_queue(q);
  }
}

template <bool BF16, int MODE, bool VEC256>
nvfp4_status launch_t(const AppendArgs& a, cudaStream_t stream) {
  const auto kern = append_kernel<BF16, MODE, VEC256>;
  const int64_t total = a.nnz * a.H * a.nb;
  const int64_t need = (total + kThreads - 1) / kThreads;
  const int64_t cap = static_cast<int64_t>(sm_count()) *
                      blocks_per_sm(reinterpret_cast<const void*>(kern), kThreads, 0);
  const int grid = static_cast<int>(need < cap ? need : cap);
  if (grid <= 0) return NVFP4_OK;
  kern<<<grid, kThreads, 0, stream>>>(a);
  return check_launch("nvfp4_quantize_append_paged");
}

// TMA path: tiles of up to 32 rows (the producer gives each row one lane) and about 24 KB
// per tensor, 2 to 6 stages in 100 KB (two CTAs per SM).
template <bool BF16, int MODE>
nvfp4_status launch_tma(const AppendArgs& a, uint32_t row_bytes, uint32_t nkv,
                        cudaStream_t stream) {
  const bool fx = append_consumer_warps(MODE) * 32 % (a.H * a.nb) == 0;
  const auto kern = nkv == 2 ? (fx ? append_tma_kernel<BF16, MODE, 2, true> : append_tma_kernel<BF16, MODE, 2, false>)
                             : (fx ? append_tma_kernel<BF16, MODE, 1, true> : append_tma_kernel<BF16, MODE, 1, false>);
  uint32_t rows = 24576u * (nkv == 2 ? 1u : 2u) / row_bytes;
  rows = rows < 1 ? 1 : (rows > 32 ? 32 : rows);
  const uint32_t one = round_up(nkv * rows * row_bytes + rows * sizeof(RowDst), 128);
  int ns = static_cast<int>(100u * 1024u / one);
  ns = ns < 2 ? 2 : (ns > 6 ? 6 : ns);
  const AppendTmaLayout L = append_tma_layout(rows, row_bytes, nkv, ns);
  const nvfp4_status st = set_dynamic_smem(reinterpret_cast<const void*>(kern), L.total,
                                           "nvfp4_quantize_append_paged");
  if (st != NVFP4_OK) return st;
  const int64_t tiles = (a.nnz + rows - 1) / rows;
  if (tiles > INT32_MAX) return fail(NVFP4_ERR_UNSUPPORTED, "nvfp4_quantize_append_paged: more than 2^31 tiles");
  const int64_t cap = static_cast<int64_t>(sm_count()) *
                      blocks_per_sm(reinterpret_cast<const void*>(kern), append_threads(MODE),
                                    L.total);
  const int grid = static_cast<int>(tiles < cap ? tiles : cap);
  if (grid <= 0) return NVFP4_OK;
  kern<<<grid, append_threads(MODE), L.total, stream>>>(a, L);
  return check_launch("nvfp4_quantize_append_paged");
}

// Calls of at most this many 16-element blocks per tensor run the direct-load kernel: it
// starts work sooner than the TMA ring, whose per-CTA set-up (tables, index chain, first
// stage) is the latency of a small call. Measured with one new token per request (8 heads
// of 128): 8.8 against 10.9 us up to 1024 tokens and 15.0 against 17.0 us at 4096 (bf16,
// standard and 4over6 fp16-error), level at 8192 and slower beyond.
constexpr int64_t kDirectMaxBlocks = int64_t(1) << 18;

template <bool BF16, int MODE>
nvfp4_status launch_v(const AppendArgs& a, bool vec256, cudaStream_t s) {
  // one row of K and V (all heads) must fit a stage; bases and row strides are 16-byte
  // aligned by the entry point's checks
  const int64_t row_bytes = static_cast<int64_t>(a.H) * a.D * 2;
  const uint32_t nkv = a.v != nullptr ? 2u : 1u;
  bool ring = nkv * row_bytes <= 48 * 1024;
  if (ring && a.pipe.append_kernel == 0) ring = a.nnz * a.H * a.nb > kDirectMaxBlocks;
  if (a.pipe.append_kernel == 2) ring = false;
  if (ring)
    return launch_tma<BF16, MODE>(a, static_cast<uint32_t>(row_bytes), nkv, s);
  return vec256 ? launch_t<BF16, MODE, true>(a, s) : launch_t<BF16, MODE, false>(a, s);
}

template <bool BF16>
nvfp4_status launch_m(const AppendArgs& a, int mode, bool vec256, cudaStream_t s) {
  switch (mode) {
    case 0: return launch_v<BF16, 0>(a, vec256, s);
    case 1: return launch_v<BF16, 1>(a, vec256, s);
    case 2: return launch_v<BF16, 2>(a, vec256, s);
    case 3: return launch_v<BF16, 3>(a, vec256, s);
    default: return launch_v<BF16, 4>(a, vec256, s);
  }
}

}  // namespace

nvfp4_status launch_append(const AppendArgs& a, bool bf16, int mode, bool vec256,
                           cudaStream_t stream) {
  return bf16 ? launch_m<true>(a, mode, vec256, stream) : launch_m<false>(a, mode, vec256, stream);
}

}  // namespace nvfp4
