// dequant.cu -- paged NVFP4 cache -> contiguous fp16/bf16.
//
// FlashInfer "flashinfer.quantization.nvfp4_kv_dequantize_paged" (description, parameters):
// gather pages through block_tables, write [batch, max_seq_len, heads, head_dim], leave
// positions >= seq_lens untouched. Decode (the append page's description):
//   out = round_out( (e2m1(q) * S) * gs )  -- e2m1 * S is exact (binary16 holds it), the
//   product with gs is rounded to binary32, then one rounding to the output type.
//
// Persistent CTAs walk a flat list of (request, page, K|V) work items built by a per-CTA
// scan of the request lengths in shared memory. One item is a page's tokens x all heads:
// its output is one contiguous run of ntok * H * D elements. Thread k of the item decodes
// 16-element block k (8 code bytes + 1 scale byte) into a 32-byte store, so each warp
// store covers 1 KB of contiguous output; up to eight blocks per thread are loaded before any
// is decoded to keep enough bytes in flight.
#include "internal.h"
#include "scan.cuh"

namespace nvfp4 {
namespace {

// 128-thread CTAs (about a dozen resident per SM) each load a whole 16-token page's blocks
// per thread before decoding, so many pages' loads are in flight at once.
constexpr int kThreads = 128;
constexpr int kUnroll = 8;

template <bool OUT_BF16>
__device__ __forceinline__ U32x8 decode_block(uint2 codes, uint32_t s, float gs) {
  const uint32_t S2 = f16x2_from_e4m3x2(s | (s << 8));
  uint32_t w[8];
  f16x2x4_from_e2m1x8(codes.x, w[0], w[1], w[2], w[3]);
  f16x2x4_from_e2m1x8(codes.y, w[4], w[5], w[6], w[7]);
  U32x8 o;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint32_t p = hmul2_rn(w[k], S2);  // exact
    const float d0 = __fmul_rn(f32_from_f16_lo(p), gs);
    const float d1 = __fmul_rn(f32_from_f16_hi(p), gs);
    o.w[k] = OUT_BF16 ? bf16x2_from_f32(d0, d1) : f16x2_from_f32(d0, d1);
  }
  return o;
}

template <bool OUT_BF16, bool BT64, bool VEC256>
__global__ void __launch_bounds__(kThreads) dequant_kernel(const DequantArgs a) {
  extern __shared__ int32_t s_cum[];
  const int32_t L = a.L;
  const int32_t ps = a.ps;
  // a length is clamped to the output and to what the block table reaches
  const int32_t cap = static_cast<int32_t>(min(static_cast<int64_t>(L), a.max_pages * ps));
  block_inclusive_scan(s_cum, a.B, [&](int32_t b) {
    int32_t len = __ldg(a.seq_lens + b);
    if (len > cap) {
      flag(a.status, NVFP4_DEV_LEN_CLAMPED);
      len = cap;
    }
    return len > 0 ? (len + ps - 1) / ps : 0;
  });
  const int32_t pages = s_cum[a.B - 1];
  const float gs_k = __ldg(a.k_scale);
  const float gs_v = __ldg(a.v_scale);
  const int32_t row_blocks = a.H * a.nb;
  const int64_t row_bytes = static_cast<int64_t>(a.H) * a.D * 2;

  for (int64_t item = blockIdx.x; item < 2 * static_cast<int64_t>(pages); item += gridDim.x) {
    const int kv = static_cast<int>(item & 1);
    const int32_t pi = static_cast<int32_t>(item >> 1);
    const int32_t b = scan_find(s_cum, a.B, pi);
    const int32_t j = pi - (b > 0 ? s_cum[b - 1] : 0);
    const int32_t len = min(__ldg(a.seq_lens + b), cap);
    const int32_t t0 = j * ps;
    const int32_t ntok = min(ps, len - t0);
    const int64_t tcol = static_cast<int64_t>(b) * a.max_pages + j;
    const int64_t page = BT64 ? __ldg(reinterpret_cast<const int64_t*>(a.block_tables) + tcol)
                              : __ldg(reinterpret_cast<const int32_t*>(a.block_tables) + tcol);
    const nvfp4_paged_cache& c = kv ? a.vc : a.kc;
    if (page < 0 || page >= c.num_pages) {
      if (threadIdx.x == 0) flag(a.status, NVFP4_DEV_BAD_PAGE);
      continue;
    }
    const uint8_t* __restrict__ pd = c.data + page * c.data_page_stride;
    const uint8_t* __restrict__ psf = c.sf + page * c.sf_page_stride;
    uint8_t* __restrict__ ob =
        (kv ? a.out_v : a.out_k) + (static_cast<int64_t>(b) * L + t0) * row_bytes;
    const float gs = kv ? gs_v : gs_k;
    const int32_t nblk = ntok * row_blocks;

    for (int32_t k0 = threadIdx.x; k0 < nblk; k0 += kThreads * kUnroll) {
      uint2 codes[kUnroll];
      uint32_t sc[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int32_t k = k0 + u * kThreads;
        if (k < nblk) {
          int32_t off = k;  // NHD: block index inside the page equals k
          if (a.layout == NVFP4_HND) {
            const int32_t slot = static_cast<int32_t>(div_q(k, a.div_row_blocks));
            const int32_t rem = k - slot * row_blocks;
            const int32_t h = static_cast<int32_t>(div_q(rem, a.div_nb));
            off = (h * ps + slot) * a.nb + (rem - h * a.nb);
          }
          codes[u] = __ldg(reinterpret_cast<const uint2*>(pd) + off);
          sc[u] = __ldg(psf + off);
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int32_t k = k0 + u * kThreads;
        if (k < nblk) {
          const U32x8 o = decode_block<OUT_BF16>(codes[u], sc[u], gs);
          uint8_t* dst = ob + static_cast<int64_t>(k) * 32;
          if (VEC256) {
            st_256(dst, o);
          } else {
            reinterpret_cast<uint4*>(dst)[0] = make_uint4(o.w[0], o.w[1], o.w[2], o.w[3]);
            reinterpret_cast<uint4*>(dst)[1] = make_uint4(o.w[4], o.w[5], o.w[6], o.w[7]);
          }
        }
      }
    }
  }
}

template <bool OUT_BF16, bool BT64, bool VEC256>
nvfp4_status launch_t(const DequantArgs& a, cudaStream_t stream) {
  const auto kern = dequant_kernel<OUT_BF16, BT64, VEC256>;
  const size_t smem = static_cast<size_t>(a.B) * sizeof(int32_t);
  if (smem > 48 * 1024) {
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(smem));
  }
  const int grid = sm_count() * blocks_per_sm(reinterpret_cast<const void*>(kern), kThreads, smem);
  kern<<<grid, kThreads, smem, stream>>>(a);
  return check_launch("nvfp4_dequantize_paged");
}

template <bool OUT_BF16, bool BT64>
nvfp4_status launch_v(const DequantArgs& a, bool vec256, cudaStream_t s) {
  return vec256 ? launch_t<OUT_BF16, BT64, true>(a, s) : launch_t<OUT_BF16, BT64, false>(a, s);
}

}  // namespace

nvfp4_status launch_dequant(const DequantArgs& a, bool out_bf16, bool bt64, bool vec256,
                            cudaStream_t stream) {
  if (out_bf16)
    return bt64 ? launch_v<true, true>(a, vec256, stream) : launch_v<true, false>(a, vec256, stream);
  return bt64 ? launch_v<false, true>(a, vec256, stream) : launch_v<false, false>(a, vec256, stream);
}

}  // namespace nvfp4
