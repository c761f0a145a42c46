// scan.cuh -- per-CTA page scan used by the persistent paged kernels.
//
// Each CTA computes, in shared memory, the inclusive prefix sum over requests of the number
// of pages each request contributes, and maps a flat page index back to (request, page)
// by binary search. Batch sizes up to kMaxScanBatch fit.
#pragma once

#include <cstdint>

namespace nvfp4 {

// s_cum[b] = sum_{b' <= b} count(b') for b < n. `count` is evaluated once per request.
// Must be called by every thread of the CTA; ends with __syncthreads().
template <typename CountFn>
__device__ __forceinline__ void block_inclusive_scan(int32_t* s_cum, int32_t n, CountFn count) {
  __shared__ int32_t s_warp[32];
  const int tid = threadIdx.x;
  const int nt = blockDim.x;
  const int per = (n + nt - 1) / nt;
  const int lo = tid * per;
  const int hi = min(n, lo + per);
  int32_t local = 0;
  for (int b = lo; b < hi; ++b) {
    local += count(b);
    s_cum[b] = local;
  }
  // inclusive scan of the per-thread totals
  const int lane = tid & 31, warp = tid >> 5;
  int32_t v = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t u = __shfl_up_sync(0xFFFFFFFFu, v, o);
    if (lane >= o) v += u;
  }
  if (lane == 31) s_warp[warp] = v;
  __syncthreads();
  if (warp == 0) {
    const int nw = (nt + 31) >> 5;
    int32_t w = lane < nw ? s_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t u = __shfl_up_sync(0xFFFFFFFFu, w, o);
      if (lane >= o) w += u;
    }
    if (lane < nw) s_warp[lane] = w;
  }
  __syncthreads();
  const int32_t offset = (v - local) + (warp > 0 ? s_warp[warp - 1] : 0);
  for (int b = lo; b < hi; ++b) s_cum[b] += offset;
  __syncthreads();
}

// Smallest b with s_cum[b] > idx (idx < s_cum[n-1]).
__device__ __forceinline__ int32_t scan_find(const int32_t* s_cum, int32_t n, int32_t idx) {
  int32_t lo = 0, hi = n - 1;
  while (lo < hi) {
    const int32_t mid = (lo + hi) >> 1;
    if (s_cum[mid] > idx) hi = mid;
    else lo = mid + 1;
  }
  return lo;
}

}  // namespace nvfp4
