// append.cu -- quantize-and-append into a paged NVFP4 cache.
//
// FlashInfer "flashinfer.page.nvfp4_quantize_append_paged_kv_cache" (description,
// parameters, note) and the "NVFP4 4over6 Recipes" section of the "flashinfer.quantization"
// index (two-candidate block-scale search, e4m3_max, err_mode, err_use_fast_math).
//
// One thread quantizes one 16-element block of one (token, head) row, for K and for V: the
// two blocks share the page lookup and give each thread two independent 32-byte loads in
// flight. A warp covers 32 consecutive blocks, i.e. 1 KB of contiguous input.
//
// Per block and candidate scale byte s (S = E4M3 value, gs = global decode scale):
//   inv = 1 / (S * gs)      (binary32 reciprocal; 0 when S*gs is 0; at most FLT_MAX)
//   q_i = E2M1_RNE_satfinite(x_i * inv)
// The 256 possible `inv` per tensor are computed once per CTA into shared memory.
// Standard NVFP4: s = E4M3(min(amax / (6 gs), e4m3_max)).
// 4over6: s_B = E4M3(min(amax / (4 gs), 448)) as well; each candidate's error sums, over the
// block, |e_i| (MAE) or e_i^2 (MSE) with e_i = x_i - e2m1(q_i) * S * gs, rounded once
// (binary32 FMA) -- or, with fast math, the whole error in binary16 (x, gs rounded to
// binary16; e2m1 * S exact in binary16; fused multiply-subtract; squares and sums rounded to
// binary16). The sum runs over a fixed halving tree: t[i] += t[i+8], t[i+4], t[i+2], t[i+1].
// B is kept only when its error is strictly smaller.
#include <cfloat>

#include "internal.h"

namespace nvfp4 {
namespace {

constexpr int kThreads = 256;

template <bool BF16>
__device__ __forceinline__ void unpack16(const U32x8& in, float x[16]) {
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    if (BF16) {
      x[2 * k] = f32_from_bf16_lo(in.w[k]);
      x[2 * k + 1] = f32_from_bf16_hi(in.w[k]);
    } else {
      x[2 * k] = f32_from_f16_lo(in.w[k]);
      x[2 * k + 1] = f32_from_f16_hi(in.w[k]);
    }
  }
}

// Codes of the block for element multiplier `inv`: two words of four code bytes each.
__device__ __forceinline__ void encode16(const float x[16], float inv, uint32_t& c0,
                                         uint32_t& c1) {
  float y[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) y[i] = __fmul_rn(x[i], inv);
  c0 = e2m1x8_from_f32(y[0], y[1], y[2], y[3], y[4], y[5], y[6], y[7]);
  c1 = e2m1x8_from_f32(y[8], y[9], y[10], y[11], y[12], y[13], y[14], y[15]);
}

// e2m1(q) * S as eight half2 (exact: at most 6 significant bits, inside binary16's range).
__device__ __forceinline__ void scaled_codes(uint32_t c0, uint32_t c1, uint32_t S2,
                                             uint32_t w[8]) {
  f16x2x4_from_e2m1x8(c0, w[0], w[1], w[2], w[3]);
  f16x2x4_from_e2m1x8(c1, w[4], w[5], w[6], w[7]);
#pragma unroll
  for (int k = 0; k < 8; ++k) w[k] = hmul2_rn(w[k], S2);
}

// Binary32 reconstruction error of one candidate.
template <bool MSE>
__device__ __forceinline__ float error_f32(const float x[16], uint32_t c0, uint32_t c1,
                                           uint32_t S2, float neg_gs) {
  uint32_t w[8];
  scaled_codes(c0, c1, S2, w);
  float t[16];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float e0 = __fmaf_rn(f32_from_f16_lo(w[k]), neg_gs, x[2 * k]);
    const float e1 = __fmaf_rn(f32_from_f16_hi(w[k]), neg_gs, x[2 * k + 1]);
    t[2 * k] = MSE ? __fmul_rn(e0, e0) : fabsf(e0);
    t[2 * k + 1] = MSE ? __fmul_rn(e1, e1) : fabsf(e1);
  }
#pragma unroll
  for (int half = 8; half >= 1; half /= 2) {
#pragma unroll
    for (int i = 0; i < half; ++i) t[i] = __fadd_rn(t[i], t[i + half]);
  }
  return t[0];
}

// Binary16 ("fast math") reconstruction error of one candidate; returned widened to float.
template <bool MSE>
__device__ __forceinline__ float error_f16(const uint32_t xh[8], uint32_t c0, uint32_t c1,
                                           uint32_t S2, uint32_t neg_gh2) {
  uint32_t t[8];
  scaled_codes(c0, c1, S2, t);
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint32_t e = hfma2_rn(t[k], neg_gh2, xh[k]);
    t[k] = MSE ? hmul2_rn(e, e) : (e & 0x7FFF7FFFu);
  }
  // pairs hold elements (2k, 2k+1): pair k + pair k+4 is t[i] + t[i+8], and so on
#pragma unroll
  for (int k = 0; k < 4; ++k) t[k] = hadd2_rn(t[k], t[k + 4]);
  t[0] = hadd2_rn(t[0], t[2]);
  t[1] = hadd2_rn(t[1], t[3]);
  t[0] = hadd2_rn(t[0], t[1]);
  const __half s = __hadd_rn(__ushort_as_half(static_cast<unsigned short>(t[0] & 0xFFFFu)),
                             __ushort_as_half(static_cast<unsigned short>(t[0] >> 16)));
  return __half2float(s);
}

struct BlockOut {
  uint32_t c0, c1, s;
};

template <bool BF16, int MODE>
__device__ __forceinline__ BlockOut quantize_block(const U32x8& in, float gs,
                                                   const float* __restrict__ inv_tab,
                                                   float cap_a, uint32_t neg_gh2) {
  float x[16];
  unpack16<BF16>(in, x);
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
  const float ra = fminf(__fdiv_rn(amax, __fmul_rn(6.0f, gs)), cap_a);
  BlockOut r;
  if (MODE == 0) {
    r.s = e4m3x2_from_f32(ra, 0.0f) & 0xFFu;
    encode16(x, inv_tab[r.s], r.c0, r.c1);
    return r;
  }
  const float rb = fminf(__fdiv_rn(amax, __fmul_rn(4.0f, gs)), 448.0f);
  const uint32_t sab = e4m3x2_from_f32(ra, rb);
  const uint32_t sa = sab & 0xFFu, sb = sab >> 8;
  uint32_t a0, a1, b0, b1;
  encode16(x, inv_tab[sa], a0, a1);
  encode16(x, inv_tab[sb], b0, b1);
  const uint32_t S2 = f16x2_from_e4m3x2(sab);
  const uint32_t SA2 = __byte_perm(S2, 0, 0x1010);  // (S_A, S_A)
  const uint32_t SB2 = __byte_perm(S2, 0, 0x3232);  // (S_B, S_B)
  float ea, eb;
  if (MODE == 1 || MODE == 2) {
    const float neg_gs = -gs;
    ea = error_f32<MODE == 2>(x, a0, a1, SA2, neg_gs);
    eb = error_f32<MODE == 2>(x, b0, b1, SB2, neg_gs);
  } else {
    uint32_t xh[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) xh[k] = BF16 ? f16x2_from_f32(x[2 * k], x[2 * k + 1]) : in.w[k];
    ea = error_f16<MODE == 4>(xh, a0, a1, SA2, neg_gh2);
    eb = error_f16<MODE == 4>(xh, b0, b1, SB2, neg_gh2);
  }
  const bool take_b = eb < ea;
  r.c0 = take_b ? b0 : a0;
  r.c1 = take_b ? b1 : a1;
  r.s = take_b ? sb : sa;
  return r;
}

template <bool BF16, int MODE, bool VEC256>
__global__ void __launch_bounds__(kThreads) append_kernel(const AppendArgs a) {
  __shared__ float s_inv[2][256];
  for (int s = threadIdx.x; s < 256; s += blockDim.x) {
    const float S = f32_from_f16_lo(f16x2_from_e4m3x2(static_cast<uint32_t>(s)));
#pragma unroll
    for (int kv = 0; kv < 2; ++kv) {
      const float den = __fmul_rn(S, a.gs[kv]);
      s_inv[kv][s] = den == 0.0f ? 0.0f : fminf(__frcp_rn(den), FLT_MAX);
    }
  }
  __syncthreads();

  uint32_t neg_gh2[2];
#pragma unroll
  for (int kv = 0; kv < 2; ++kv) {
    const uint32_t gh = __half_as_ushort(__float2half_rn(a.gs[kv])) ^ 0x8000u;
    neg_gh2[kv] = gh | (gh << 16);
  }

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
    const U32x8 xv = VEC256 ? ld_nc_256(pv) : ld_nc_2x128(pv);

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
    const int64_t page = __ldg(a.kv_indices + start + lp);
    const int64_t slot = pos - lp * a.ps;
    const int64_t r = a.layout == NVFP4_NHD ? slot * a.H + h : static_cast<int64_t>(h) * a.ps + slot;

#pragma unroll
    for (int kv = 0; kv < 2; ++kv) {
      const nvfp4_paged_cache& c = kv ? a.vc : a.kc;
      if (page < 0 || page >= c.num_pages) {
        flag(a.status, NVFP4_DEV_BAD_PAGE);
        continue;
      }
      const BlockOut q =
          quantize_block<BF16, MODE>(kv ? xv : xk, a.gs[kv], s_inv[kv], a.cap_a, neg_gh2[kv]);
      uint8_t* dst = c.data + page * c.data_page_stride + r * (a.D / 2) + 8 * j;
      *reinterpret_cast<uint2*>(dst) = make_uint2(q.c0, q.c1);
      c.sf[page * c.sf_page_stride + r * a.nb + j] = static_cast<uint8_t>(q.s);
    }
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

template <bool BF16, int MODE>
nvfp4_status launch_v(const AppendArgs& a, bool vec256, cudaStream_t s) {
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
