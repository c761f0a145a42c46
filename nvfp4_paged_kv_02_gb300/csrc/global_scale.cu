// global_scale.cu -- per-tensor global decode scale.
//
// "flashinfer.quantization" index, make_nvfp4_global_scale and the "NVFP4 4over6 Recipes"
// warning (the scale must be built with the quantizer's recipe):
//   gs = amax(|x|) / (6 * e4m3_max)   (binary32; gs = 1 for an all-zero tensor)
// so that the block holding the tensor's amax gets the top block scale e4m3_max.
//
// The amax is exact: |x| of fp16/bf16 orders like the integer (bits & 0x7FFF), so the scan
// takes unsigned 16-bit maxima of the masked words (two per 32-bit lane op; eight 32-byte
// loads in flight per thread) and reduces over the CTA. A large tensor is scanned by many
// CTAs, which combine with an atomic max on the binary32 bit pattern of the result,
// accumulated in the output word itself (zeroed by a memset first); a one-thread kernel
// then turns the amax into gs. A small tensor is scanned by one CTA, which writes gs itself.
#include "internal.h"

namespace nvfp4 {
namespace {

constexpr int kThreads = 512;
// Tensors of at most this many elements take the one-CTA kernel: one launch instead of a
// memset, a many-CTA scan and a finalize. Measured (bf16, L2 flushed): 6.8 against 9.9 us at
// 12,928 elements, 8.8 against 9.9 us at 65,536, level at 131,072, slower from 262,144.
constexpr int64_t kOneCtaMaxNumel = int64_t(1) << 16;

template <bool BF16>
__device__ __forceinline__ uint32_t f32_bits_of_mag16(uint32_t m) {
  return BF16 ? (m << 16) : __float_as_uint(__half2float(__ushort_as_half(static_cast<unsigned short>(m))));
}

// max |x| over this CTA's share of the tensor (a grid-stride scan), as the binary32 bit
// pattern of the magnitude; valid in thread 0.
template <bool BF16>
__device__ __forceinline__ uint32_t cta_amax_bits(const uint16_t* __restrict__ x, int64_t numel) {
  __shared__ uint32_t s_red[kThreads / 32];
  uint32_t m2 = 0;  // two 16-bit maxima
  const int64_t nvec = numel / 16;
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t v = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; v + 7 * step < nvec; v += 8 * step) {
    U32x8 w[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) w[u] = ld_nc_2x128(x + (v + u * step) * 16);
#pragma unroll
    for (int u = 0; u < 8; ++u)
#pragma unroll
      for (int k = 0; k < 8; ++k) m2 = __vmaxu2(m2, w[u].w[k] & 0x7FFF7FFFu);
  }
  for (; v < nvec; v += step) {
    const U32x8 w = ld_nc_2x128(x + v * 16);
#pragma unroll
    for (int k = 0; k < 8; ++k) m2 = __vmaxu2(m2, w.w[k] & 0x7FFF7FFFu);
  }
  for (int64_t i = nvec * 16 + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
       i < numel; i += step)
    m2 = __vmaxu2(m2, static_cast<uint32_t>(x[i]) & 0x7FFFu);
  uint32_t m = f32_bits_of_mag16<BF16>(max(m2 & 0xFFFFu, m2 >> 16));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    m = threadIdx.x < (kThreads / 32) ? s_red[threadIdx.x] : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  }
  return m;
}

__device__ __forceinline__ float scale_from_amax(float amax, float denom) {
  return amax == 0.0f ? 1.0f : __fdiv_rn(amax, denom);
}

// Many CTAs: each combines its maximum into the output word (zeroed first) with an atomic
// max on the bit pattern; finalize_kernel then turns the amax into gs.
template <bool BF16>
__global__ void __launch_bounds__(kThreads) amax_kernel(const uint16_t* __restrict__ x,
                                                        int64_t numel, uint32_t* acc) {
  const uint32_t m = cta_amax_bits<BF16>(x, numel);
  if (threadIdx.x == 0 && m != 0) atomicMax(acc, m);
}

__global__ void finalize_kernel(float* out, float denom) {
  *out = scale_from_amax(__uint_as_float(*reinterpret_cast<const uint32_t*>(out)), denom);
}

// A small tensor: one CTA scans all of it and writes gs (one launch, nothing zeroed first).
template <bool BF16>
__global__ void __launch_bounds__(kThreads) amax_one_cta_kernel(const uint16_t* __restrict__ x,
                                                                int64_t numel, float denom,
                                                                float* out) {
  const uint32_t m = cta_amax_bits<BF16>(x, numel);
  if (threadIdx.x == 0) *out = scale_from_amax(__uint_as_float(m), denom);
}

}  // namespace

nvfp4_status launch_global_scale(const void* x, bool bf16, int64_t numel, float denom,
                                 float* out, cudaStream_t stream) {
  const uint16_t* xp = static_cast<const uint16_t*>(x);
  if (numel <= kOneCtaMaxNumel) {
    if (bf16) amax_one_cta_kernel<true><<<1, kThreads, 0, stream>>>(xp, numel, denom, out);
    else amax_one_cta_kernel<false><<<1, kThreads, 0, stream>>>(xp, numel, denom, out);
    return check_launch("nvfp4_make_global_scale");
  }
  cudaError_t e = cudaMemsetAsync(out, 0, sizeof(float), stream);
  if (e != cudaSuccess) return fail(NVFP4_ERR_CUDA, std::string("cudaMemsetAsync: ") + cudaGetErrorString(e));
  const void* kern = bf16 ? reinterpret_cast<const void*>(amax_kernel<true>)
                          : reinterpret_cast<const void*>(amax_kernel<false>);
  const int64_t need = (numel / 16 + kThreads - 1) / kThreads;
  const int64_t cap = static_cast<int64_t>(sm_count()) * blocks_per_sm(kern, kThreads, 0);
  const int grid = static_cast<int>(need < 1 ? 1 : (need < cap ? need : cap));
  uint32_t* acc = reinterpret_cast<uint32_t*>(out);
  if (bf16) amax_kernel<true><<<grid, kThreads, 0, stream>>>(xp, numel, acc);
  else amax_kernel<false><<<grid, kThreads, 0, stream>>>(xp, numel, acc);
  nvfp4_status st = check_launch("nvfp4_make_global_scale");
  if (st != NVFP4_OK) return st;
  finalize_kernel<<<1, 1, 0, stream>>>(out, denom);
  return check_launch("nvfp4_make_global_scale");
}

}  // namespace nvfp4
