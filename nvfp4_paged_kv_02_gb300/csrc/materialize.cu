// materialize.cu -- active pages of a paged NVFP4 cache -> FP8 E4M3 copy.
//
// FlashInfer "nvfp4_kv_materialize_fp8" (parameters, returns, note) and
// "NVFP4KVMaterializer.run" ("flashinfer.quantization" index): request b's page j goes to
// output page kv_page_indptr[b] + j + 1 (b * max_pages_per_seq + j + 1 by default) of a
// [num_pages + 1, 2, H, page_size, D] float8_e4m3fn copy whose page 0 is zero; only E2M1
// value x E4M3 block scale is applied (exact in binary16), rounded to E4M3 with saturation
// at 448; fp8_block_tables[b, j] holds the output page.
//
// Persistent CTAs walk a flat list of (active page, K|V) items from a shared-memory scan of
// the request lengths. An item converts H * page_size * D elements; thread k handles the
// 32-element chunk k of the output half page (16 code bytes + 2 scale bytes in, one
// 32-byte store out). With HND input, chunk k is also the k-th 16-byte chunk of the input
// page, so both streams are contiguous.
//
// V scales may also come in the 4-token-interleaved layout the materialize parameters name
// for v_block_scales (HND only). The pages do not define it; the reading taken here keeps
// the [pages, H, page_size, D/16] shape and, within each head's page slice, stores each
// group of four slots block-major and slot-minor, so block j of page row r (= h * ps + slot)
// is byte (r & ~3) * (D/16) + 4 j + (r & 3). Only the scale index changes: the page is
// still one contiguous run of scale bytes.
#include "internal.h"
#include "pipeline.cuh"
#include "scan.cuh"

namespace nvfp4 {
namespace {

// TMA ring shape: twelve consumer warps, three CTAs per SM (measured faster than eight).
constexpr int kConsumerWarps = 12;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kTmaThreads = kConsumers + 32;

// 128-thread CTAs (about a dozen resident per SM): each thread loads its four chunks of a
// 16-token page before converting, and many pages are in flight per SM.
constexpr int kThreads = 128;
constexpr int kUnroll = 4;

__device__ __forceinline__ uint32_t fp8x2(uint32_t h2, uint32_t S2) {
  return e4m3x2_from_f16x2(hmul2_rn(h2, S2));
}

// 16 code bytes (32 elements, two blocks) with scale bytes s0, s1 -> 32 E4M3 bytes.
__device__ __forceinline__ U32x8 convert_chunk(uint4 c, uint32_t s01) {
  const uint32_t s0 = s01 & 0xFFu, s1 = (s01 >> 8) & 0xFFu;
  const uint32_t S0 = f16x2_from_e4m3x2(s0 | (s0 << 8));
  const uint32_t S1 = f16x2_from_e4m3x2(s1 | (s1 << 8));
  const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
  U32x8 o;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t h0, h1, h2, h3;
    f16x2x4_from_e2m1x8(cw[q], h0, h1, h2, h3);
    const uint32_t S = q < 2 ? S0 : S1;
    o.w[2 * q] = fp8x2(h0, S) | (fp8x2(h1, S) << 16);
    o.w[2 * q + 1] = fp8x2(h2, S) | (fp8x2(h3, S) << 16);
  }
  return o;
}

// The two scale bytes of output chunk k (blocks 2c and 2c + 1 of page row r = k / (D/32)).
// Linear: the 16-bit word at chunk offset `off`. Interleaved V (HND, so off == k): bytes
// (r & ~3) * (D/16) + 8c + (r & 3) and 4 bytes after it.
__device__ __forceinline__ uint32_t interleaved4_scales(const uint8_t* sf, int32_t k,
                                                        int32_t row_chunks, Div div_row_chunks) {
  const int32_t r = static_cast<int32_t>(div_q(k, div_row_chunks));
  const int32_t c = k - r * row_chunks;
  const int32_t i0 = (r & ~3) * (2 * row_chunks) + 8 * c + (r & 3);
  return static_cast<uint32_t>(sf[i0]) | (static_cast<uint32_t>(sf[i0 + 4]) << 8);
}

template <bool VIL>
__global__ void __launch_bounds__(kThreads) materialize_kernel(const MaterializeArgs a) {
  extern __shared__ int32_t s_cum[];
  const int32_t ps = a.ps;
  const int32_t mpps = a.mpps;
  block_inclusive_scan(s_cum, a.B, [&](int32_t b) {
    const int32_t len = __ldg(a.seq_lens + b);
    int32_t n = len > 0 ? static_cast<int32_t>((static_cast<int64_t>(len) + ps - 1) / ps) : 0;
    if (n > mpps) {
      flag(a.status, NVFP4_DEV_LEN_CLAMPED);
      n = mpps;
    }
    return n;
  });
  const int32_t pages = s_cum[a.B - 1];
  const int64_t half_page = static_cast<int64_t>(a.H) * ps * a.D;  // bytes of K or V
  const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t gstep = static_cast<int64_t>(gridDim.x) * blockDim.x;

  // page 0 of the copy is zero
  for (int64_t q = gtid; q < 2 * half_page / 16; q += gstep)
    reinterpret_cast<uint4*>(a.out)[q] = make_uint4(0, 0, 0, 0);

  // page table: active entries, and zero padding in the functional form
  const int64_t entries = static_cast<int64_t>(a.B) * mpps;
  for (int64_t e = gtid; e < entries; e += gstep) {
    const int32_t b = static_cast<int32_t>(div_q(e, a.div_mpps));
    const int32_t j = static_cast<int32_t>(e - static_cast<int64_t>(b) * mpps);
    const int32_t n = s_cum[b] - (b > 0 ? s_cum[b - 1] : 0);
    if (j < n) {
      const int64_t base = a.kv_page_indptr ? __ldg(a.kv_page_indptr + b)
                                            : static_cast<int64_t>(b) * mpps;
      a.tables[e] = static_cast<int32_t>(base + j + 1);
    } else if (a.zero_tables) {
      a.tables[e] = 0;
    }
  }

  const int32_t row_chunks = a.D / 32;
  const int32_t chunks = a.H * ps * row_chunks;
  for (int64_t item = blockIdx.x; item < 2 * static_cast<int64_t>(pages); item += gridDim.x) {
    const int kv = static_cast<int>(item & 1);
    const int32_t pi = static_cast<int32_t>(item >> 1);
    const int32_t b = scan_find(s_cum, a.B, pi);
    const int32_t j = pi - (b > 0 ? s_cum[b - 1] : 0);
    const int64_t tcol = a.shared ? static_cast<int64_t>(b) * a.max_num_pages + j
                                  : (static_cast<int64_t>(b) * 2 + kv) * a.max_num_pages + j;
    const int64_t page = __ldg(a.block_tables + tcol);
    const int64_t base = a.kv_page_indptr ? __ldg(a.kv_page_indptr + b)
                                          : static_cast<int64_t>(b) * mpps;
    const int64_t o = base + j + 1;
    const nvfp4_paged_cache& c = kv ? a.vc : a.kc;
    if (page < 0 || page >= c.num_pages) {
      if (threadIdx.x == 0) flag(a.status, NVFP4_DEV_BAD_PAGE);
      continue;
    }
    if (o < 1 || o >= a.out_num_pages) {
      if (threadIdx.x == 0) flag(a.status, NVFP4_DEV_BAD_OUT_PAGE);
      continue;
    }
    const uint8_t* __restrict__ pd = c.data + page * c.data_page_stride;
    const uint8_t* __restrict__ psf = c.sf + page * c.sf_page_stride;
    uint8_t* __restrict__ dst = a.out + (o * 2 + kv) * half_page;

    for (int32_t k0 = threadIdx.x; k0 < chunks; k0 += kThreads * kUnroll) {
      uint4 cv[kUnroll];
      uint32_t sv[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int32_t k = k0 + u * kThreads;
        if (k < chunks) {
          int32_t off = k;  // HND: chunk k of the output is chunk k of the input page
          if (a.layout == NVFP4_NHD) {
            const int32_t h = static_cast<int32_t>(div_q(k, a.div_page_chunks));
            const int32_t rem = k - h * (ps * row_chunks);
            const int32_t slot = static_cast<int32_t>(div_q(rem, a.div_row_chunks));
            off = (slot * a.H + h) * row_chunks + (rem - slot * row_chunks);
          }
          cv[u] = __ldg(reinterpret_cast<const uint4*>(pd) + off);
          if (VIL && kv)
            sv[u] = interleaved4_scales(psf, k, row_chunks, a.div_row_chunks);
          else
            sv[u] = __ldg(reinterpret_cast<const uint16_t*>(psf) + off);
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int32_t k = k0 + u * kThreads;
        if (k < chunks) st_256(dst + static_cast<int64_t>(k) * 32, convert_chunk(cv[u], sv[u]));
      }
    }
  }
}

// Items the producers take from the work queue per atomic: consecutive items are the K and
// V halves of neighbouring output pages, so about 128 KB of output per batch (measured: 8
// items of 16-slot pages on the large pool, 1120 against 1180 us with 2), but at least 8
// batches per CTA so that the last wave stays even (decode workload: 4, not 8). Every CTA
// computes the same value from the same item count.
__device__ __forceinline__ int items_per_fetch(int64_t items, int64_t item_bytes) {
  int k = static_cast<int>(min(static_cast<int64_t>(8),
                               max(static_cast<int64_t>(1), (int64_t(128) << 10) / item_bytes)));
  while (k > 1 && items < static_cast<int64_t>(gridDim.x) * k * 8) k >>= 1;
  return k;
}

// ---- TMA-fed variant ------------------------------------------------------------------
//
// The producer warp resolves each (active page, K|V) item -- source page, output page --
// and bulk-copies the source page's codes and scales into the next free shared-memory
// stage; the consumer warps convert from shared memory and stream the 32-byte stores.

template <bool VIL>
__global__ void __launch_bounds__(kTmaThreads, 3) materialize_tma_kernel(const MaterializeArgs a,
                                                                       const TmaLayout L) {
  extern __shared__ __align__(128) uint8_t smem[];
  int32_t* s_cum = reinterpret_cast<int32_t*>(smem);
  uint8_t* stages = smem + L.stages_off;
  StageMeta* meta = reinterpret_cast<StageMeta*>(smem + L.meta_off);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars_off);
  uint64_t* empty = full + L.ns;
  volatile int32_t* s_abort = reinterpret_cast<int32_t*>(smem + L.misc_off);
  volatile uint32_t* s_issued = reinterpret_cast<uint32_t*>(smem + L.misc_off + 4);
  const int ns = L.ns;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < ns; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, kConsumerWarps);
      s_issued[s] = 0;
    }
    *s_abort = 0;
    fence_mbar_init();
  }
  const int32_t ps = a.ps;
  const int32_t mpps = a.mpps;
  block_inclusive_scan(s_cum, a.B, [&](int32_t b) {  // ends with __syncthreads()
    const int32_t len = __ldg(a.seq_lens + b);
    int32_t n = len > 0 ? static_cast<int32_t>((static_cast<int64_t>(len) + ps - 1) / ps) : 0;
    if (n > mpps) {
      flag(a.status, NVFP4_DEV_LEN_CLAMPED);
      n = mpps;
    }
    return n;
  });
  const int64_t half_page = static_cast<int64_t>(a.H) * ps * a.D;
  const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t gstep = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t q = gtid; q < 2 * half_page / 16; q += gstep)
    reinterpret_cast<uint4*>(a.out)[q] = make_uint4(0, 0, 0, 0);
  const int64_t entries = static_cast<int64_t>(a.B) * mpps;
  for (int64_t e = gtid; e < entries; e += gstep) {
    const int32_t b = static_cast<int32_t>(div_q(e, a.div_mpps));
    const int32_t j = static_cast<int32_t>(e - static_cast<int64_t>(b) * mpps);
    const int32_t n = s_cum[b] - (b > 0 ? s_cum[b - 1] : 0);
    if (j < n) {
      const int64_t base = a.kv_page_indptr ? __ldg(a.kv_page_indptr + b)
                                            : static_cast<int64_t>(b) * mpps;
      a.tables[e] = static_cast<int32_t>(base + j + 1);
    } else if (a.zero_tables) {
      a.tables[e] = 0;
    }
  }
  const int64_t items = 2 * static_cast<int64_t>(s_cum[a.B - 1]);

  const WorkQueue q = work_queue(a.workspace);
  if (warp == kConsumerWarps) {
    int s = 0;
    uint32_t round = 0;  // how many times stage s has been used before
    ItemCursor cur;
    if (lane == 0) {
      // the last two batches' worth of items per CTA are taken one at a time
      const int per = items_per_fetch(items, half_page);
      cur.init(q, per, items - 2ll * per * gridDim.x);
    }
    for (;; s = (s + 1 == ns) ? 0 : s + 1, round += (s == 0)) {
      // the next item, its source page and output page, resolved while the consumers still
      // work on the stage it will use
      long long item = 0;
      if (lane == 0) item = cur.next(q, items);
      item = __shfl_sync(0xFFFFFFFFu, item, 0);
      const bool end = item >= items;
      StageMeta m{0, 0, 0, kStageEnd};
      int64_t page = 0;
      if (lane == 0 && !end) {
        const int kv = static_cast<int>(item & 1);
        const int32_t pi = static_cast<int32_t>(item >> 1);
        const int32_t b = scan_find(s_cum, a.B, pi);
        const int32_t j = pi - (b > 0 ? s_cum[b - 1] : 0);
        const int64_t tcol = a.shared ? static_cast<int64_t>(b) * a.max_num_pages + j
                                      : (static_cast<int64_t>(b) * 2 + kv) * a.max_num_pages + j;
        page = __ldg(a.block_tables + tcol);
        const int64_t base = a.kv_page_indptr ? __ldg(a.kv_page_indptr + b)
                                              : static_cast<int64_t>(b) * mpps;
        const int64_t o = base + j + 1;
        const bool page_ok = page >= 0 && page < (kv ? a.vc.num_pages : a.kc.num_pages);
        const bool out_ok = o >= 1 && o < a.out_num_pages;
        if (!page_ok) flag(a.status, NVFP4_DEV_BAD_PAGE);
        else if (!out_ok) flag(a.status, NVFP4_DEV_BAD_OUT_PAGE);
        const bool valid = page_ok && out_ok;
        m.f0 = static_cast<int32_t>(valid ? o : 0);
        m.f1 = kv;
        m.f2 = 0;
        m.flags = valid ? 2 : 0;
      }
      bool ok = true;
      if (lane == 0) ok = mbar_wait(empty + s, (round & 1u) ^ 1u, a.pipe.wait_limit) && !*s_abort;
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) {
        if (lane == 0) {
          *s_abort = 1;
          flag(a.status, NVFP4_DEV_TIMEOUT);
        }
        break;
      }
      // (test control: withhold the first stage so that the consumers' wait expires)
      if (lane == 0 && (end || !(a.pipe.stall && round == 0 && s == 0))) {
        meta[s] = m;
        uint8_t* st = stages + static_cast<uint32_t>(s) * L.stage_bytes;
        if (m.flags & 2) {
          const int kv = m.f1;
          const uint8_t* data = kv ? a.vc.data : a.kc.data;
          const uint8_t* sf = kv ? a.vc.sf : a.kc.sf;
          const int64_t dps = kv ? a.vc.data_page_stride : a.kc.data_page_stride;
          const int64_t sps = kv ? a.vc.sf_page_stride : a.kc.sf_page_stride;
          mbar_arrive_expect_tx(full + s, L.codes_bytes + L.sf_bytes);
          bulk_g2s(st, data + page * dps, L.codes_bytes, full + s);
          bulk_g2s(st + L.sf_off, sf + page * sps, L.sf_bytes, full + s);
        } else {
          mbar_arrive(full + s);
        }
        s_issued[s] = round + 1;
      }
      __syncwarp();
      if (end) break;
    }
  } else {
    const int ct = threadIdx.x;
    const int32_t row_chunks = a.D / 32;
    const int32_t chunks = a.H * ps * row_chunks;
    int s = 0;
    uint32_t round = 0;  // how many times stage s has been used before
    for (;; s = (s + 1 == ns) ? 0 : s + 1, round += (s == 0)) {
      if (*s_abort || !mbar_wait(full + s, round & 1u, a.pipe.wait_limit)) {
        if (lane == 0) {
          *s_abort = 1;
          flag(a.status, NVFP4_DEV_TIMEOUT);
        }
        break;
      }
      const StageMeta m = meta[s];
      if (m.flags & kStageEnd) break;
      if (m.flags & 2) {
        const uint8_t* st = stages + static_cast<uint32_t>(s) * L.stage_bytes;
        const uint8_t* sfp = st + L.sf_off;
        uint8_t* dst = a.out + (static_cast<int64_t>(m.f0) * 2 + m.f1) * half_page;
        if (VIL && m.f1) {  // interleaved V scales (HND pages only)
#pragma unroll 4
          for (int32_t k = ct; k < chunks; k += kConsumers) {
            const uint4 c = *reinterpret_cast<const uint4*>(st + 16 * k);
            const uint32_t s01 = interleaved4_scales(sfp, k, row_chunks, a.div_row_chunks);
            st_256(dst + static_cast<int64_t>(k) * 32, convert_chunk(c, s01));
          }
        } else {
#pragma unroll 4
          for (int32_t k = ct; k < chunks; k += kConsumers) {
            int32_t off = k;  // HND: chunk k of the output is chunk k of the input page
            if (a.layout == NVFP4_NHD) {
              const int32_t h = static_cast<int32_t>(div_q(k, a.div_page_chunks));
              const int32_t rem = k - h * (ps * row_chunks);
              const int32_t slot = static_cast<int32_t>(div_q(rem, a.div_row_chunks));
              off = (slot * a.H + h) * row_chunks + (rem - slot * row_chunks);
            }
            const uint4 c = *reinterpret_cast<const uint4*>(st + 16 * off);
            const uint32_t s01 = *reinterpret_cast<const uint16_t*>(sfp + 2 * off);
            st_256(dst + static_cast<int64_t>(k) * 32, convert_chunk(c, s01));
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty + s);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int s = 0; s < ns; ++s)
      if (s_issued[s] > 0) mbar_wait(full + s, (s_issued[s] - 1) & 1u, a.pipe.wait_limit);
    finish_queue(q);
  }
}

const void* materialize_kernel_ptr(bool bulk, bool v_interleaved) {
  if (bulk)
    return v_interleaved ? reinterpret_cast<const void*>(materialize_tma_kernel<true>)
                         : reinterpret_cast<const void*>(materialize_tma_kernel<false>);
  return v_interleaved ? reinterpret_cast<const void*>(materialize_kernel<true>)
                       : reinterpret_cast<const void*>(materialize_kernel<false>);
}

// Dynamic shared memory of a launch for up to max_B requests.
size_t materialize_smem(bool bulk, int max_B, int64_t cb, int64_t sb) {
  if (!bulk) return static_cast<size_t>(max_B) * sizeof(int32_t);
  return tma_layout(max_B, static_cast<uint32_t>(cb), static_cast<uint32_t>(sb),
                    stages_for(static_cast<uint32_t>(cb), static_cast<uint32_t>(sb)))
      .total;
}

}  // namespace

nvfp4_status prepare_materialize(bool bulk, bool v_interleaved, int max_B, int64_t cb,
                                 int64_t sb, MaterializeLaunch* out) {
  const void* kern = materialize_kernel_ptr(bulk, v_interleaved);
  const size_t smem = materialize_smem(bulk, max_B, cb, sb);
  if (bulk || smem > 48 * 1024) {
    const nvfp4_status st = set_dynamic_smem(kern, smem, "nvfp4_materializer_prepare");
    if (st != NVFP4_OK) return st;
  }
  const int threads = bulk ? kTmaThreads : kThreads;
  out->bulk = bulk ? 1 : 0;
  out->max_B = max_B;
  out->smem = static_cast<int32_t>(smem);
  out->grid = sm_count() * blocks_per_sm(kern, threads, smem);
  return NVFP4_OK;
}

nvfp4_status launch_materialize_prepared(const MaterializeArgs& a, const MaterializeLaunch& c,
                                         cudaStream_t stream) {
  if (c.bulk) {
    const int64_t cb = static_cast<int64_t>(a.ps) * a.H * (a.D / 2);
    const int64_t sb = static_cast<int64_t>(a.ps) * a.H * (a.D / 16);
    const TmaLayout L = tma_layout(c.max_B, static_cast<uint32_t>(cb), static_cast<uint32_t>(sb),
                                   stages_for(static_cast<uint32_t>(cb), static_cast<uint32_t>(sb)));
    if (a.v_interleaved) materialize_tma_kernel<true><<<c.grid, kTmaThreads, c.smem, stream>>>(a, L);
    else materialize_tma_kernel<false><<<c.grid, kTmaThreads, c.smem, stream>>>(a, L);
  } else {
    if (a.v_interleaved) materialize_kernel<true><<<c.grid, kThreads, c.smem, stream>>>(a);
    else materialize_kernel<false><<<c.grid, kThreads, c.smem, stream>>>(a);
  }
  return check_launch("nvfp4_materializer_run");
}

nvfp4_status launch_materialize(const MaterializeArgs& a, cudaStream_t stream) {
  const int64_t cb = static_cast<int64_t>(a.ps) * a.H * (a.D / 2);
  const int64_t sb = static_cast<int64_t>(a.ps) * a.H * (a.D / 16);
  if (pages_bulk_copyable(a.kc, a.vc, cb, sb)) {
    const auto kern = a.v_interleaved ? materialize_tma_kernel<true> : materialize_tma_kernel<false>;
    const TmaLayout L = tma_layout(a.B, static_cast<uint32_t>(cb), static_cast<uint32_t>(sb),
                                   stages_for(static_cast<uint32_t>(cb), static_cast<uint32_t>(sb)));
    const nvfp4_status st =
        set_dynamic_smem(reinterpret_cast<const void*>(kern), L.total, "nvfp4_materialize_fp8");
    if (st != NVFP4_OK) return st;
    const int grid =
        sm_count() * blocks_per_sm(reinterpret_cast<const void*>(kern), kTmaThreads, L.total);
    kern<<<grid, kTmaThreads, L.total, stream>>>(a, L);
    return check_launch("nvfp4_materialize_fp8");
  }
  const auto kern = a.v_interleaved ? materialize_kernel<true> : materialize_kernel<false>;
  const size_t smem = static_cast<size_t>(a.B) * sizeof(int32_t);
  if (smem > 48 * 1024) {
    const nvfp4_status st =
        set_dynamic_smem(reinterpret_cast<const void*>(kern), smem, "nvfp4_materialize_fp8");
    if (st != NVFP4_OK) return st;
  }
  const int grid = sm_count() * blocks_per_sm(reinterpret_cast<const void*>(kern), kThreads, smem);
  kern<<<grid, kThreads, smem, stream>>>(a);
  return check_launch("nvfp4_materialize_fp8");
}

}  // namespace nvfp4
