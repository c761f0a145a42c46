// device.cuh -- sm_103a device helpers shared by the NVFP4 KV-cache kernels.
//
// Number formats (FlashInfer "nvfp4_quantize_append_paged_kv_cache" description; "NVFP4
// 4over6 Recipes"): E2M1 element codes, two per byte with element 2k in the low nibble;
// E4M3 block scales stored as bytes. Conversions use the Blackwell hardware cvt forms:
//   cvt.rn.satfinite.e2m1x2.f32  two binary32 -> one byte (RNE, saturating at +-6)
//   cvt.rn.f16x2.e2m1x2          one byte -> two exact binary16 values
//   cvt.rn.satfinite.e4m3x2.f32  two binary32 -> two E4M3 bytes (RNE, saturating at 448)
//   cvt.rn.f16x2.e4m3x2          two E4M3 bytes -> two exact binary16 values
//   cvt.rn.satfinite.e4m3x2.f16x2  two binary16 -> two E4M3 bytes
// In every packed form the first-listed (upper) source lands in the upper half of the
// destination, so the low element goes last.
//
// Arithmetic that decides a code or an output value is written with explicit IEEE
// round-to-nearest operations (".rn" PTX forms and __f*_rn intrinsics), and the
// translation units are compiled with -fmad=false, so no multiply-add is contracted
// unless it is written as a fused operation on purpose.
#pragma once

#include <cstdint>

#include <cuda_fp16.h>

namespace nvfp4 {

// ---- packed format conversions --------------------------------------------------------

// Four bytes of E2M1 codes -> four half2 (byte k -> h[k], low nibble in .x).
__device__ __forceinline__ void f16x2x4_from_e2m1x8(uint32_t w, uint32_t& h0, uint32_t& h1,
                                                    uint32_t& h2, uint32_t& h3) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
      : "r"(w));
}

// Two binary32 values -> two E4M3 bytes: `lo` in bits 7:0, `hi` in bits 15:8.
__device__ __forceinline__ uint32_t e4m3x2_from_f32(float lo, float hi) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}

// Two E4M3 bytes (bits 7:0 and 15:8 of `b`) -> half2 (.x from bits 7:0).
__device__ __forceinline__ uint32_t f16x2_from_e4m3x2(uint32_t b) {
  uint32_t r;
  uint16_t s = static_cast<uint16_t>(b);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(s));
  return r;
}

// half2 -> two E4M3 bytes (.x in bits 7:0), RNE, saturating at 448.
__device__ __forceinline__ uint32_t e4m3x2_from_f16x2(uint32_t h) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(d) : "r"(h));
  return d;
}

// Two binary32 -> half2 (RNE; overflow gives Inf), .x = lo.
__device__ __forceinline__ uint32_t f16x2_from_f32(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two binary32 -> bf16x2 (RNE), .x = lo.
__device__ __forceinline__ uint32_t bf16x2_from_f32(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float f32_from_f16_lo(uint32_t h) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h & 0xFFFFu)));
}
__device__ __forceinline__ float f32_from_f16_hi(uint32_t h) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h >> 16)));
}
// Exact binary32 value of the two bf16 halves of a word.
__device__ __forceinline__ float f32_from_bf16_hi(uint32_t w) {
  return __uint_as_float(w & 0xFFFF0000u);
}

// ---- packed binary16 arithmetic (IEEE RN, subnormals kept) ------------------------------

__device__ __forceinline__ uint32_t hmul2_rn(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t hadd2_rn(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("add.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t hfma2_rn(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

// Squares written as a fused multiply-add whose addend `nz` is -0 at run time:
// RN(a*a + -0) == RN(a*a), one rounding. The compiler cannot see that the addend is -0, so
// it can neither turn the FMA back into a multiply nor contract it into a following add.
// (ptxas was seen to fuse a packed square -- and an fma with a literal -0 addend -- into
// the next packed add despite the .rn modifier and -fmad=false, which changes the
// rounding of an error sum.)
// ---- scalar helpers -----------------------------------------------------------------------
__device__ __forceinline__ uint32_t hsq2_rn(uint32_t a, uint32_t nz) {
  uint32_t r;
  asm("fma.rn.f16x2 %0, %1, %1, %2;" : "=r"(r) : "r"(a), "r"(nz));
  return r;
}

// Correctly rounded a / b from a precomputed rb = RN(1/b): q0 = a*rb, the residual
// a - q0*b is exact in a fused multiply-add, and q0 + residual*rb rounds to RN(a/b)
// (Markstein's theorem) for normal b and normal a/b.
__device__ __forceinline__ float div_rn_with_rcp(float a, float b, float rb) {
  const float q0 = __fmul_rn(a, rb);
  const float r = __fmaf_rn(-q0, b, a);
  return __fmaf_rn(r, rb, q0);
}

// ---- memory access ----------------------------------------------------------------------

struct U32x8 {
  uint32_t w[8];
};

// 32-byte read-only load (address 32-byte aligned).
__device__ __forceinline__ U32x8 ld_nc_256(const void* p) {
  U32x8 r;
  asm volatile(
      "ld.global.nc.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
      : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3]), "=r"(r.w[4]), "=r"(r.w[5]),
        "=r"(r.w[6]), "=r"(r.w[7])
      : "l"(p));
  return r;
}

// Two 16-byte read-only loads (address 16-byte aligned).
__device__ __forceinline__ U32x8 ld_nc_2x128(const void* p) {
  U32x8 r;
  const uint4 a = __ldg(reinterpret_cast<const uint4*>(p));
  const uint4 b = __ldg(reinterpret_cast<const uint4*>(p) + 1);
  r.w[0] = a.x; r.w[1] = a.y; r.w[2] = a.z; r.w[3] = a.w;
  r.w[4] = b.x; r.w[5] = b.y; r.w[6] = b.z; r.w[7] = b.w;
  return r;
}

// 32 bytes from shared memory (address 16-byte aligned).
__device__ __forceinline__ U32x8 ld_shared_256(const void* p) {
  U32x8 r;
  const uint4 a = reinterpret_cast<const uint4*>(p)[0];
  const uint4 b = reinterpret_cast<const uint4*>(p)[1];
  r.w[0] = a.x; r.w[1] = a.y; r.w[2] = a.z; r.w[3] = a.w;
  r.w[4] = b.x; r.w[5] = b.y; r.w[6] = b.z; r.w[7] = b.w;
  return r;
}

// 32-byte store (address 32-byte aligned).
__device__ __forceinline__ void st_256(void* p, const U32x8& v) {
  asm volatile(
      "st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
      :
      : "l"(p), "r"(v.w[0]), "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3]), "r"(v.w[4]), "r"(v.w[5]),
        "r"(v.w[6]), "r"(v.w[7])
      : "memory");
}

// Record a device-side status bit (nullable status word).
__device__ __forceinline__ void flag(int32_t* status, int32_t bit) {
  if (status) atomicOr(status, bit);
}

// n / d and n % d for d > 0; `shift` >= 0 when d is a power of two (2^shift).
struct Div {
  int64_t d;
  int32_t shift;
};
__host__ __device__ inline Div make_div(int64_t d) {
  Div r{d, -1};
  if (d > 0 && (d & (d - 1)) == 0) {
    int s = 0;
    while ((int64_t(1) << s) < d) ++s;
    r.shift = s;
  }
  return r;
}
__device__ __forceinline__ int64_t div_q(int64_t n, Div d) {
  return d.shift >= 0 ? (n >> d.shift) : n / d.d;
}
// The same for non-negative 32-bit n with a divisor below 2^31.
__device__ __forceinline__ int32_t div_q32(int32_t n, Div d) {
  return d.shift >= 0 ? (n >> d.shift) : n / static_cast<int32_t>(d.d);
}

}  // namespace nvfp4
