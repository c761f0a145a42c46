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
#include <mutex>
#include <string>

#include "internal.h"
#include "pipeline.cuh"
#include "scan.cuh"

namespace nvfp4 {
namespace {

// TMA ring shape: eight consumer warps, four CTAs per SM (48 KB of stages each; measured
// against three CTAs and against twelve warps).
constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kTmaThreads = kConsumers + 32;
// Items a producer takes from the work queue per atomic (a page of K or V is one item;
// one at a time measured best: the output of one item is already a long contiguous run).
constexpr int kItemsPerFetch = 1;

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

// ---- TMA-fed variant ------------------------------------------------------------------
//
// Warp kConsumerWarps (the producer) walks the item list: it resolves the page index and
// bulk-copies the page's codes and scales into the next free stage of a shared-memory
// ring, with the item's geometry alongside. The consumer warps decode from shared memory
// and stream the 32-byte output stores, so no warp waits on HBM latency while it could be
// decoding.

template <bool OUT_BF16, bool BT64>
__global__ void __launch_bounds__(kTmaThreads, 4) dequant_tma_kernel(const DequantArgs a,
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
  const int32_t L_out = a.L;
  const int32_t ps = a.ps;
  const int32_t cap = static_cast<int32_t>(min(static_cast<int64_t>(L_out), a.max_pages * ps));
  block_inclusive_scan(s_cum, a.B, [&](int32_t b) {  // ends with __syncthreads()
    int32_t len = __ldg(a.seq_lens + b);
    if (len > cap) {
      flag(a.status, NVFP4_DEV_LEN_CLAMPED);
      len = cap;
    }
    return len > 0 ? (len + ps - 1) / ps : 0;
  });
  const int64_t items = 2 * static_cast<int64_t>(s_cum[a.B - 1]);

  const WorkQueue q = work_queue(a.workspace);
  // With the work queue the last items (at most two per CTA) are handed out as two halves
  // each -- heads [0, H/2) and [H/2, H) of an HND page, slots [0, ps/2) and [ps/2, ps) of an
  // NHD one -- so that the last wave ends more evenly. Units below full_items are whole
  // pages; each item after them is two units.
  const int64_t full_items =
      (q.next && a.split) ? max(static_cast<int64_t>(0), items - 2 * static_cast<int64_t>(gridDim.x))
                          : items;
  const int64_t units = full_items + 2 * (items - full_items);
  if (warp == kConsumerWarps) {
    // producer: lane 0 takes the items and issues, the warp stays converged
    int s = 0;
    uint32_t round = 0;  // how many times stage s has been used before
    ItemCursor cur;
    if (lane == 0) cur.init(q, kItemsPerFetch);
    for (;; s = (s + 1 == ns) ? 0 : s + 1, round += (s == 0)) {
      // the next item and its source page, resolved while the consumers still work on the
      // stage it will use
      long long unit = 0;
      if (lane == 0) unit = cur.next(q, units);
      unit = __shfl_sync(0xFFFFFFFFu, unit, 0);
      const bool end = unit >= units;
      long long item = unit;
      int part = 0;  // 0: the whole page; 1, 2: its first or second half
      if (unit >= full_items) {
        item = full_items + ((unit - full_items) >> 1);
        part = 1 + static_cast<int>((unit - full_items) & 1);
      }
      StageMeta m{0, 0, 0, kStageEnd};
      int64_t page = 0;
      if (lane == 0 && !end) {
        const int kv = static_cast<int>(item & 1);
        const int32_t pi = static_cast<int32_t>(item >> 1);
        const int32_t b = scan_find(s_cum, a.B, pi);
        const int32_t j = pi - (b > 0 ? s_cum[b - 1] : 0);
        const int32_t len = min(__ldg(a.seq_lens + b), cap);
        const int32_t t0 = j * ps;
        const int64_t tcol = static_cast<int64_t>(b) * a.max_pages + j;
        page = BT64 ? __ldg(reinterpret_cast<const int64_t*>(a.block_tables) + tcol)
                    : __ldg(reinterpret_cast<const int32_t*>(a.block_tables) + tcol);
        const bool valid = page >= 0 && page < (kv ? a.vc.num_pages : a.kc.num_pages);
        m.f0 = b;
        m.f1 = t0;
        m.f2 = min(ps, len - t0);
        m.flags = kv | (valid ? 2 : 0) | (part << 3);
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
          const int kv = m.flags & 1;
          const uint8_t* data = kv ? a.vc.data : a.kc.data;
          const uint8_t* sf = kv ? a.vc.sf : a.kc.sf;
          const int64_t dps = kv ? a.vc.data_page_stride : a.kc.data_page_stride;
          const int64_t sps = kv ? a.vc.sf_page_stride : a.kc.sf_page_stride;
          // a half page is the first or second half of the page's codes and of its scales
          const uint32_t cb = part ? L.codes_bytes / 2 : L.codes_bytes;
          const uint32_t sb = part ? L.sf_bytes / 2 : L.sf_bytes;
          const int64_t off_c = part == 2 ? cb : 0, off_s = part == 2 ? sb : 0;
          mbar_arrive_expect_tx(full + s, cb + sb);
          bulk_g2s(st, data + page * dps + off_c, cb, full + s);
          bulk_g2s(st + L.sf_off, sf + page * sps + off_s, sb, full + s);
        } else {
          if (!end) flag(a.status, NVFP4_DEV_BAD_PAGE);
          mbar_arrive(full + s);
        }
        s_issued[s] = round + 1;
      }
      __syncwarp();
      if (end) break;
    }
  } else {
    const int ct = threadIdx.x;  // 0 .. kConsumers-1
    const int32_t row_blocks = a.H * a.nb;
    const int64_t row_bytes = static_cast<int64_t>(a.H) * a.D * 2;
    const float gs_k = __ldg(a.k_scale);
    const float gs_v = __ldg(a.v_scale);
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
        uint8_t* ob = ((m.flags & 1) ? a.out_v : a.out_k) +
                      (static_cast<int64_t>(m.f0) * L_out + m.f1) * row_bytes;
        const float gs = (m.flags & 1) ? gs_v : gs_k;
        const int32_t ntok = m.f2;
        const int part = (m.flags >> 3) & 3;
        if (a.layout == NVFP4_NHD) {
          // the page holds [slot, head, block]: the same order as the output run (a half page:
          // slots [lo, lo + ps/2))
          const int32_t lo = part == 2 ? ps / 2 : 0;
          const int32_t n = max(0, min(ntok - lo, part ? ps / 2 : ps));
          const int32_t nblk = n * row_blocks;
          uint8_t* ob_h = ob + static_cast<int64_t>(lo) * row_bytes;
#pragma unroll 4
          for (int32_t k = ct; k < nblk; k += kConsumers) {
            const uint2 codes = *reinterpret_cast<const uint2*>(st + 8 * k);
            st_256(ob_h + static_cast<int64_t>(k) * 32, decode_block<OUT_BF16>(codes, sfp[k], gs));
          }
        } else {
          // the page holds [head, slot, block]: read it in that order (no shared-memory
          // bank conflicts); each group of nb lanes still writes a contiguous output row (a half
          // page: heads [h0, h0 + H/2))
          const int32_t h0 = part == 2 ? a.H / 2 : 0;
          const int32_t page_blocks = (part ? a.H / 2 : a.H) * ps * a.nb;
#pragma unroll 4
          for (int32_t k = ct; k < page_blocks; k += kConsumers) {
            const int32_t hs = div_q32(k, a.div_nb);  // (h - h0) * ps + slot
            const int32_t blk = k - hs * a.nb;
            const int32_t h = div_q32(hs, a.div_ps);
            const int32_t slot = hs - h * ps;
            if (slot >= ntok) continue;
            const uint2 codes = *reinterpret_cast<const uint2*>(st + 8 * k);
            const int32_t o = (slot * a.H + h0 + h) * a.nb + blk;
            st_256(ob + static_cast<int64_t>(o) * 32, decode_block<OUT_BF16>(codes, sfp[k], gs));
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty + s);
    }
  }
  // no copy may still be landing in this CTA's shared memory when it exits
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int s = 0; s < ns; ++s)
      if (s_issued[s] > 0) mbar_wait(full + s, (s_issued[s] - 1) & 1u, a.pipe.wait_limit);
    finish_queue(q);
  }
}

// ---- contiguous form ----------------------------------------------------------------
//
// FlashInfer "flashinfer.quantization" index, "FP4 KV Cache Quantization":
// nvfp4_kv_dequantize on a contiguous code tensor with linear block scales. A grid-stride
// loop over 16-element blocks; each thread loads four blocks (8 code bytes + 1 scale byte
// each, a warp's loads being contiguous runs) before it decodes them into 32-byte stores.
constexpr int kKvThreads = 256;

template <bool OUT_BF16, bool VEC256>
__global__ void __launch_bounds__(kKvThreads) kv_dequant_kernel(const KvDequantArgs a) {
  const float gs = __ldg(a.gs);
  const int64_t T = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const uint2* codes = reinterpret_cast<const uint2*>(a.codes);
  for (int64_t b0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; b0 < a.blocks;
       b0 += 4 * T) {
    uint2 c[4];
    uint32_t sc[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t b = b0 + u * T;
      if (b < a.blocks) {
        c[u] = __ldg(codes + b);
        sc[u] = __ldg(a.sf + b);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t b = b0 + u * T;
      if (b < a.blocks) {
        const U32x8 o = decode_block<OUT_BF16>(c[u], sc[u], gs);
        uint8_t* dst = a.out + b * 32;
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

// The contiguous form through the same kind of ring as the paged one: a work item is a
// chunk of kKvChunk consecutive blocks (8 KB of codes and 1 KB of scales, one bulk copy each;
// 32 KB of 16-bit output), so that the reads reach HBM as long runs instead of each warp's
// 256-byte load. The blocks after the last whole chunk (fewer than kKvChunk) are decoded
// straight from global memory by the consumer threads, one block each, before the ring.
// Needs 16-byte aligned codes and scales and a 32-byte aligned output.
constexpr int32_t kKvChunk = 1024;

template <bool OUT_BF16>
__global__ void __launch_bounds__(kTmaThreads, 4) kv_dequant_tma_kernel(const KvDequantArgs a,
                                                                     const TmaLayout L) {
  extern __shared__ __align__(128) uint8_t smem[];
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
  __syncthreads();
  const int64_t chunks = a.blocks / kKvChunk;
  const WorkQueue q = work_queue(a.workspace);
  if (warp == kConsumerWarps) {
    // producer: lane 0 takes the chunks and issues, the warp stays converged
    int s = 0;
    uint32_t round = 0;  // how many times stage s has been used before
    ItemCursor cur;
    if (lane == 0) cur.init(q, 1);
    for (;; s = (s + 1 == ns) ? 0 : s + 1, round += (s == 0)) {
      long long item = 0;
      if (lane == 0) item = cur.next(q, chunks);
      item = __shfl_sync(0xFFFFFFFFu, item, 0);
      const bool end = item >= chunks;
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
        // the chunk index in two halves (f0 low, f1 high)
        meta[s] = StageMeta{static_cast<int32_t>(item & 0xFFFFFFFFll),
                            static_cast<int32_t>(item >> 32), 0, end ? kStageEnd : 2};
        if (!end) {
          uint8_t* st = stages + static_cast<uint32_t>(s) * L.stage_bytes;
          mbar_arrive_expect_tx(full + s, 9u * kKvChunk);
          bulk_g2s(st, a.codes + item * (8 * kKvChunk), 8u * kKvChunk, full + s);
          bulk_g2s(st + L.sf_off, a.sf + item * kKvChunk, static_cast<uint32_t>(kKvChunk), full + s);
        } else {
          mbar_arrive(full + s);
        }
        s_issued[s] = round + 1;
      }
      __syncwarp();
      if (end) break;
    }
  } else {
    const int ct = threadIdx.x;  // 0 .. kConsumers-1
    const float gs = __ldg(a.gs);
    // the blocks after the last whole chunk
    for (int64_t b = chunks * kKvChunk + static_cast<int64_t>(blockIdx.x) * kConsumers + ct;
         b < a.blocks; b += static_cast<int64_t>(gridDim.x) * kConsumers) {
      const uint2 codes = __ldg(reinterpret_cast<const uint2*>(a.codes) + b);
      st_256(a.out + b * 32, decode_block<OUT_BF16>(codes, __ldg(a.sf + b), gs));
    }
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
      const int64_t item = static_cast<int64_t>(static_cast<uint32_t>(m.f0)) |
                           (static_cast<int64_t>(m.f1) << 32);
      const uint8_t* st = stages + static_cast<uint32_t>(s) * L.stage_bytes;
      uint8_t* ob = a.out + item * (32 * kKvChunk);
#pragma unroll
      for (int32_t k = ct; k < kKvChunk; k += kConsumers) {
        const uint2 codes = *reinterpret_cast<const uint2*>(st + 8 * k);
        st_256(ob + static_cast<int64_t>(k) * 32,
               decode_block<OUT_BF16>(codes, st[L.sf_off + k], gs));
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty + s);
    }
  }
  // no copy may still be landing in this CTA's shared memory when it exits
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int s = 0; s < ns; ++s)
      if (s_issued[s] > 0) mbar_wait(full + s, (s_issued[s] - 1) & 1u, a.pipe.wait_limit);
    finish_queue(q);
  }
}

template <bool OUT_BF16>
nvfp4_status launch_kv_tma(const KvDequantArgs& a, cudaStream_t stream) {
  const auto kern = kv_dequant_tma_kernel<OUT_BF16>;
  const uint32_t cb = 8u * kKvChunk, sb = static_cast<uint32_t>(kKvChunk);
  const TmaLayout L = tma_layout(0, cb, sb, stages_for(cb, sb, 48u * 1024u));
  const nvfp4_status st =
      set_dynamic_smem(reinterpret_cast<const void*>(kern), L.total, "nvfp4_kv_dequantize");
  if (st != NVFP4_OK) return st;
  const int64_t chunks = a.blocks / kKvChunk;
  const int64_t cap = static_cast<int64_t>(sm_count()) *
                      blocks_per_sm(reinterpret_cast<const void*>(kern), kTmaThreads, L.total);
  const int grid = static_cast<int>(chunks < cap ? chunks : cap);
  kern<<<grid, kTmaThreads, L.total, stream>>>(a, L);
  return check_launch("nvfp4_kv_dequantize");
}

template <bool OUT_BF16, bool VEC256>
nvfp4_status launch_kv(const KvDequantArgs& a, cudaStream_t stream) {
  const auto kern = kv_dequant_kernel<OUT_BF16, VEC256>;
  const int64_t need = (a.blocks + 4 * kKvThreads - 1) / (4 * kKvThreads);
  const int64_t cap = static_cast<int64_t>(sm_count()) *
                      blocks_per_sm(reinterpret_cast<const void*>(kern), kKvThreads, 0);
  const int grid = static_cast<int>(need < cap ? need : cap);
  if (grid <= 0) return NVFP4_OK;
  kern<<<grid, kKvThreads, 0, stream>>>(a);
  return check_launch("nvfp4_kv_dequantize");
}

template <bool OUT_BF16, bool BT64, bool VEC256>
nvfp4_status launch_t(const DequantArgs& a, cudaStream_t stream) {
  const auto kern = dequant_kernel<OUT_BF16, BT64, VEC256>;
  const size_t smem = static_cast<size_t>(a.B) * sizeof(int32_t);
  if (smem > 48 * 1024) {
    const nvfp4_status st =
        set_dynamic_smem(reinterpret_cast<const void*>(kern), smem, "nvfp4_dequantize_paged");
    if (st != NVFP4_OK) return st;
  }
  const int grid = sm_count() * blocks_per_sm(reinterpret_cast<const void*>(kern), kThreads, smem);
  kern<<<grid, kThreads, smem, stream>>>(a);
  return check_launch("nvfp4_dequantize_paged");
}

// The TMA path needs bulk-copyable pages and a 32-byte aligned output.
bool tma_eligible(const DequantArgs& a, bool vec256, uint32_t& codes_bytes, uint32_t& sf_bytes) {
  const int64_t cb = static_cast<int64_t>(a.ps) * a.H * (a.D / 2);
  const int64_t sb = static_cast<int64_t>(a.ps) * a.H * (a.D / 16);
  codes_bytes = static_cast<uint32_t>(cb);
  sf_bytes = static_cast<uint32_t>(sb);
  return vec256 && pages_bulk_copyable(a.kc, a.vc, cb, sb);
}

template <bool OUT_BF16, bool BT64>
nvfp4_status launch_tma(const DequantArgs& a, uint32_t codes_bytes, uint32_t sf_bytes,
                        cudaStream_t stream) {
  const auto kern = dequant_tma_kernel<OUT_BF16, BT64>;
  const TmaLayout L = tma_layout(a.B, codes_bytes, sf_bytes, stages_for(codes_bytes, sf_bytes, 48u * 1024u));
  // halves of a page can be bulk-copied when the split dimension is even and each half of
  // the codes and of the scales is a whole number of 16-byte units
  DequantArgs b = a;
  const int32_t split_dim = a.layout == NVFP4_NHD ? a.ps : a.H;
  b.split = split_dim % 2 == 0 && (codes_bytes / 2) % 16 == 0 && (sf_bytes / 2) % 16 == 0;
  const nvfp4_status st =
      set_dynamic_smem(reinterpret_cast<const void*>(kern), L.total, "nvfp4_dequantize_paged");
  if (st != NVFP4_OK) return st;
  const int grid =
      sm_count() * blocks_per_sm(reinterpret_cast<const void*>(kern), kTmaThreads, L.total);
  kern<<<grid, kTmaThreads, L.total, stream>>>(b, L);
  return check_launch("nvfp4_dequantize_paged");
}

template <bool OUT_BF16, bool BT64>
nvfp4_status launch_v(const DequantArgs& a, bool vec256, cudaStream_t s) {
  uint32_t cb, sb;
  if (tma_eligible(a, vec256, cb, sb)) return launch_tma<OUT_BF16, BT64>(a, cb, sb, s);
  return vec256 ? launch_t<OUT_BF16, BT64, true>(a, s) : launch_t<OUT_BF16, BT64, false>(a, s);
}

}  // namespace

nvfp4_status launch_kv_dequant(const KvDequantArgs& a, bool out_bf16, bool vec256,
                               cudaStream_t stream) {
  const auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  if (vec256 && al16(a.codes) && al16(a.sf) && a.blocks >= kKvChunk)
    return out_bf16 ? launch_kv_tma<true>(a, stream) : launch_kv_tma<false>(a, stream);
  if (out_bf16) return vec256 ? launch_kv<true, true>(a, stream) : launch_kv<true, false>(a, stream);
  return vec256 ? launch_kv<false, true>(a, stream) : launch_kv<false, false>(a, stream);
}

nvfp4_status launch_dequant(const DequantArgs& a, bool out_bf16, bool bt64, bool vec256,
                            cudaStream_t stream) {
  if (out_bf16)
    return bt64 ? launch_v<true, true>(a, vec256, stream) : launch_v<true, false>(a, vec256, stream);
  return bt64 ? launch_v<false, true>(a, vec256, stream) : launch_v<false, false>(a, vec256, stream);
}

// ---- scratch of nvfp4_dequantize_paged_no_alloc ------------------------------------------
//
// That entry point keeps the work queue of its launches here instead of in a workspace from
// the caller: one NVFP4_WORKSPACE_BYTES block, which every device that loads the library
// holds until the process exits, and which every call of that entry point shares. Host code
// must not pass the array's name to a kernel (on the host it is only a stand-in for the
// device variable); no_alloc_scratch() looks up its device address once per device.
static __device__ __align__(256) unsigned char g_no_alloc_scratch[NVFP4_WORKSPACE_BYTES];

nvfp4_status no_alloc_scratch(void** out) {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return fail(NVFP4_ERR_CUDA, std::string("nvfp4_dequantize_paged_no_alloc: cudaGetDevice: ") +
                                    cudaGetErrorString(e));
  }
  if (dev < 0 || dev >= kMaxDevices)
    return fail(NVFP4_ERR_UNSUPPORTED, "nvfp4_dequantize_paged_no_alloc: device ordinal above 63");
  std::lock_guard<std::mutex> lk(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    // the device is current here, so this is the address on that device
    e = cudaGetSymbolAddress(&p, g_no_alloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      (void)cudaGetLastError();
      return fail(NVFP4_ERR_CUDA,
                  std::string("nvfp4_dequantize_paged_no_alloc: cudaGetSymbolAddress: ") +
                      cudaGetErrorString(e));
    }
    addr[dev] = p;
  }
  *out = addr[dev];
  return NVFP4_OK;
}

}  // namespace nvfp4
