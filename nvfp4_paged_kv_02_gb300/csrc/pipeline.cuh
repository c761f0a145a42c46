// pipeline.cuh -- shared-memory stage ring fed by TMA bulk copies (sm_90+ forms, used on
// sm_103a): mbarrier init / arrive / transaction counts / bounded waits and the
// global -> shared cp.async.bulk.
//
// Every wait is bounded: mbar_wait() gives up after kWaitLimit polls and returns false, so
// a kernel can record an error, stop issuing copies, wait (again bounded) for its own
// copies in flight and return, instead of spinning forever.
#pragma once

#include <cstdint>

#include "../../include/nvfp4kv.h"

namespace nvfp4 {

// Polls of mbarrier.try_wait before a wait is abandoned (each poll may itself suspend the
// thread for a short, hardware-defined time).
constexpr uint32_t kWaitLimit = 1u << 22;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Make initialized barriers visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Arrive and announce `bytes` of TMA traffic that will complete on this barrier.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase of parity `parity` to complete; false after `limit` polls.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          uint32_t limit = kWaitLimit) {
  for (uint32_t i = 0; i < limit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// Test control of a pipelined launch: `stall` makes the producer withhold the first stage
// of each CTA (so the consumers' wait expires), with a short `wait_limit`. `append_kernel`
// overrides the append's size-based kernel choice: 0 by size, 1 the TMA ring, 2 the
// direct-load kernel (so that tests cover both at any size).
struct PipeTest {
  uint32_t wait_limit;
  int32_t stall;
  int32_t append_kernel;
};

// Bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned) from global to
// this CTA's shared memory, completing as transaction bytes on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// ---- work distribution among the persistent CTAs ----------------------------------------
//
// Without a workspace each CTA's producer takes the items blockIdx.x, blockIdx.x + gridDim.x,
// ... (a fixed share). With one (NVFP4_WORKSPACE_BYTES of device memory, zero when the
// launch starts), the producers take the next item from a counter there as their stages
// free up, so CTAs on SMs that run ahead take more items and the last wave ends together.
// The last CTA to finish sets the workspace back to zero for the next launch on its stream.
struct WorkQueue {
  unsigned long long* next;  // item counter (null: fixed shares)
  unsigned int* done;        // CTAs that have finished taking items
};

__host__ __device__ inline WorkQueue work_queue(void* workspace) {
  WorkQueue q;
  q.next = static_cast<unsigned long long*>(workspace);
  q.done = workspace ? reinterpret_cast<unsigned int*>(static_cast<unsigned char*>(workspace) + 8)
                     : nullptr;
  return q;
}

// The items of one CTA's producer (one thread calls it). From the queue they come `per`
// at a time, consecutive (one atomic per batch: a single counter takes a few hundred
// million atomics a second, which small items would otherwise reach, and consecutive items
// of one CTA write neighbouring output); in fixed shares one at a time. The next batch is
// requested when the current one is started, so the atomic's latency overlaps the work on
// the current items. Batches requested from item `tail` on are single items, so that the
// last wave ends more evenly.
struct ItemCursor {
  long long mine, base, next_base, tail;
  int i, per, n, next_n;

  __device__ __forceinline__ long long take(const WorkQueue& q, int count) {
    if (q.next) return static_cast<long long>(atomicAdd(q.next, static_cast<unsigned long long>(count)));
    const long long it = mine;
    mine += gridDim.x;
    return it;
  }
  __device__ __forceinline__ void init(const WorkQueue& q, int items_per_fetch,
                                       long long tail_from = 0x7FFFFFFFFFFFFFFFll) {
    mine = blockIdx.x;
    i = 0;
    per = q.next ? (items_per_fetch > 0 ? items_per_fetch : 1) : 1;
    tail = tail_from;
    n = next_n = per;
    next_base = 0;
    base = take(q, n);
  }
  // The next item; one at or past `limit` means there is no more work.
  __device__ __forceinline__ long long next(const WorkQueue& q, long long limit) {
    const long long item = base + i;
    if (i == 0 && item < limit) {
      next_n = item >= tail ? 1 : per;
      next_base = take(q, next_n);
    }
    if (++i == n) {
      base = next_base;
      n = next_n;
      i = 0;
    }
    return item;
  }
};

// Called by one thread of every CTA once the CTA takes no more items.
__device__ __forceinline__ void finish_queue(const WorkQueue& q) {
  if (!q.next) return;
  __threadfence();
  if (atomicAdd(q.done, 1u) == gridDim.x - 1) {
    *q.next = 0;
    *q.done = 0;
    __threadfence();
  }
}

// ---- page-stage ring layout shared by the TMA-fed paged kernels ------------------------
//
// Dynamic shared memory: [per-request scan: B int32][ns stages: codes | scales]
// [ns StageMeta][ns full + ns empty mbarriers][abort flag][ns issue counters].
// Each kernel file sets its ring's shape: warps 0..W-1 consume, warp W produces (bulk
// copies), so a CTA has 32 * W + 32 threads.

struct StageMeta {
  int32_t f0, f1, f2, flags;  // item fields chosen by the kernel; flags bit 1 = page valid
};
// flags bit 2: no more items (the consumers leave their loop)
constexpr int32_t kStageEnd = 4;

struct TmaLayout {
  uint32_t codes_bytes, sf_bytes;  // one page of one tensor
  uint32_t sf_off, stage_bytes;    // inside a stage
  uint32_t stages_off, meta_off, bars_off, misc_off, total;
  int ns;
};

__host__ __device__ inline uint32_t round_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline TmaLayout tma_layout(int B, uint32_t codes_bytes, uint32_t sf_bytes,
                                                int ns) {
  TmaLayout L;
  L.codes_bytes = codes_bytes;
  L.sf_bytes = sf_bytes;
  L.sf_off = round_up(codes_bytes, 128);
  L.stage_bytes = L.sf_off + round_up(sf_bytes, 128);
  L.ns = ns;
  L.stages_off = round_up(static_cast<uint32_t>(B) * 4u, 128);
  L.meta_off = L.stages_off + static_cast<uint32_t>(ns) * L.stage_bytes;
  L.bars_off = L.meta_off + static_cast<uint32_t>(ns) * sizeof(StageMeta);
  L.misc_off = L.bars_off + 2u * static_cast<uint32_t>(ns) * 8u;
  L.total = L.misc_off + 4u * (1u + static_cast<uint32_t>(ns));
  return L;
}

// Stages that fit in `budget` bytes, between 2 and 8 (64 KB leaves room for three CTAs
// per SM).
inline int stages_for(uint32_t codes_bytes, uint32_t sf_bytes, uint32_t budget = 64u * 1024u) {
  const uint32_t one = round_up(codes_bytes, 128) + round_up(sf_bytes, 128);
  int ns = static_cast<int>(budget / one);
  return ns < 2 ? 2 : (ns > 8 ? 8 : ns);
}

// Whether one page of each cache can be bulk-copied: 16-byte aligned bases and strides,
// copy sizes a multiple of 16, and a stage small enough for two per CTA.
inline bool pages_bulk_copyable(const nvfp4_paged_cache& k, const nvfp4_paged_cache& v,
                                int64_t codes_bytes, int64_t sf_bytes) {
  auto al = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  return codes_bytes % 16 == 0 && sf_bytes % 16 == 0 && codes_bytes + sf_bytes <= 48 * 1024 &&
         al(k.data) && al(k.sf) && al(v.data) && al(v.sf) && k.data_page_stride % 16 == 0 &&
         v.data_page_stride % 16 == 0 && k.sf_page_stride % 16 == 0 && v.sf_page_stride % 16 == 0;
}

}  // namespace nvfp4
