/*
 * nvfp4kv.h -- C ABI of the GB300 (sm_103a) NVFP4 paged KV-cache library.
 *
 * Operations, as the FlashInfer documentation pages define them:
 *   - quantize-and-append into a paged NVFP4 cache
 *       ("flashinfer.page.nvfp4_quantize_append_paged_kv_cache": description, parameters, note)
 *   - paged dequantize into contiguous fp16/bf16
 *       ("flashinfer.quantization.nvfp4_kv_dequantize_paged": description, parameters)
 *   - materialize the active pages as an FP8 E4M3 copy
 *       ("flashinfer.quantization.kernels.nvfp4_kv_materialize.nvfp4_kv_materialize_fp8":
 *        parameters, returns, note; "NVFP4KVMaterializer" class on the
 *        "flashinfer.quantization" index page)
 *   - the per-tensor global decode scale and the recipe's block-scale clamp
 *       ("flashinfer.quantization" index: "NVFP4 4over6 Recipes", make_nvfp4_global_scale,
 *        nvfp4_e4m3_max)
 *   - contiguous quantize / dequantize with the same block rule
 *       ("flashinfer.quantization" index: "FP4 KV Cache Quantization", nvfp4_kv_quantize,
 *        nvfp4_kv_dequantize)
 *
 * Number formats: E2M1 codes (grid {0,0.5,1,1.5,2,3,4,6}, 4 bits, two per byte, element
 * 2k in the low nibble); E4M3 (e4m3fn) block scales stored as bytes, one per 16
 * consecutive elements of head_dim ("linear" layout); a positive fp32 global decode scale
 * gs per tensor. A value decodes as e2m1 * block_scale * gs.
 *
 * Conventions shared by every entry point:
 *   - Ownership: every pointer is caller-owned. Device pointers must point to memory of the
 *     current device. The library never allocates, never frees and never synchronizes with
 *     the host; all work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream), so the calls may be captured into CUDA graphs.
 *   - Validation: arguments that the host can check (sizes, enums, alignment, the scale
 *     values passed by value, extents shared between arguments) are checked before any
 *     launch; a failure returns a status other than NVFP4_OK, enqueues nothing and sets the
 *     text returned by nvfp4_last_error_string(). Values held in device memory (indices,
 *     lengths, page numbers) are not read on the host.
 *   - Device-side bounds: kernels never read or write outside the extents passed in. A row
 *     or page whose device-held index falls outside them is skipped; if `dev_status` is not
 *     NULL the kernel ORs the matching NVFP4_DEV_* bit into *dev_status (device memory,
 *     one int32 the caller zeroes).
 *   - Work distribution (`workspace`, the last-but-one argument of the append, dequantize,
 *     materialize and contiguous quantize and dequantize calls): NULL, or NVFP4_WORKSPACE_BYTES of device
 *     memory, 8-byte aligned, that is zero before its first use. With it, the persistent
 *     CTAs of the bulk-copy kernels take work items from a counter there as they free up
 *     (CTAs on SMs that run ahead take more); the kernel sets it back to zero before it
 *     finishes, so the same workspace serves the next call. Without it each CTA takes a
 *     fixed share. The results are the same either way. One workspace serves one call at a
 *     time: calls that may run at the same time on the device (different streams, or a
 *     graph replayed beside direct calls) need different workspaces.
 *   - Launch errors are returned as NVFP4_ERR_CUDA with the CUDA error text.
 *   - Thread safety: entry points may be called from several host threads; the error text
 *     is per thread.
 */
#ifndef NVFP4KV_H_
#define NVFP4KV_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define NVFP4KV_ABI_VERSION 5

/* Bytes of the optional `workspace` of the bulk-copy kernels (see the conventions). */
#define NVFP4_WORKSPACE_BYTES 16

/* Return codes. */
typedef int32_t nvfp4_status;
#define NVFP4_OK 0
#define NVFP4_ERR_INVALID_ARG 1 /* a size, enum, scale or extent is out of range */
#define NVFP4_ERR_UNSUPPORTED 2 /* a valid request this library does not implement */
#define NVFP4_ERR_ALIGNMENT 3   /* a pointer or stride breaks the stated alignment */
#define NVFP4_ERR_CUDA 4        /* the CUDA runtime reported an error at launch */

/* Element types of fp16/bf16 tensors. */
#define NVFP4_F16 0
#define NVFP4_BF16 1

/* Paged layouts: NHD = [pages, page_size, heads, .], HND = [pages, heads, page_size, .]. */
#define NVFP4_NHD 0
#define NVFP4_HND 1

/* Integer type of a dequantize block table. */
#define NVFP4_I32 0
#define NVFP4_I64 1

/* Layouts of a materialize V block-scale cache. LINEAR: [pages, H, page_size, D/16] row
 * after row (the K layout). INTERLEAVED4: the "4-token-interleaved" layout the materialize
 * parameters name for v_block_scales without defining it; this library's reading keeps the
 * shape and, within each head's page slice, stores each group of four slots block-major and
 * slot-minor: block j of slot t of head h sits at byte
 * (h * page_size + (t & ~3)) * (D/16) + 4 j + (t & 3) of the page. */
#define NVFP4_SF_LINEAR 0
#define NVFP4_SF_INTERLEAVED4 1

/* 4over6 error metrics ("NVFP44Over6ErrMode"): summed absolute or summed squared error. */
#define NVFP4_ERR_MAE 0
#define NVFP4_ERR_MSE 1

/* Device-side status bits (see dev_status above). */
#define NVFP4_DEV_BAD_BATCH 1     /* append: batch_indices[i] outside [0, batch_size) */
#define NVFP4_DEV_BAD_POSITION 2  /* append: position outside the request's described space,
                                     or its page entry outside kv_indices */
#define NVFP4_DEV_BAD_PAGE 4      /* a physical page index outside [0, num_pages) */
#define NVFP4_DEV_LEN_CLAMPED 8   /* a sequence length beyond the output extent, clamped */
#define NVFP4_DEV_BAD_OUT_PAGE 16 /* materialize: output page index outside the workspace */
#define NVFP4_DEV_TIMEOUT 32      /* a pipeline wait gave up (the kernel stopped early) */
#define NVFP4_DEV_BAD_SCALE 64    /* a device-held global scale is not positive finite */

/* A 4over6 recipe ("NVFP44Over6Config"; "NVFP4 4over6 Recipes" section). A NULL recipe
 * pointer means standard NVFP4 (4over6 off), as None does in the pages' kernel drivers.
 *   e4m3_max          top of the block-scale range, in (0, 448]; 256 keeps the amax/4
 *                     candidate representable ("e4m3_max=256" knob).
 *   err_mode          NVFP4_ERR_MAE or NVFP4_ERR_MSE ("err_mode" knob).
 *   err_use_fast_math 0 = error in fp32, 1 = error in fp16 (a distinct recipe). */
typedef struct {
  float e4m3_max;
  int32_t err_mode;
  int32_t err_use_fast_math;
} nvfp4_4over6_config;

/* One paged NVFP4 cache: K or V ("paged_kv_cache" / "kv_cache_sf" parameters). A stacked
 * 5-D cache with K/V on the second dimension is two of these: V's pointers offset by one
 * K/V slice and both page strides covering the pair.
 *   data             packed E2M1 codes; page p starts at data + p * data_page_stride and
 *                    holds [page_size, H, D/2] (NHD) or [H, page_size, D/2] (HND) bytes.
 *   sf               E4M3 block scales; page p at sf + p * sf_page_stride, holding
 *                    [page_size, H, D/16] (NHD) or [H, page_size, D/16] (HND) bytes.
 *   data_page_stride bytes between pages (>= page_size*H*D/2; a multiple of 16); the page
 *                    stride may exceed a compact page.
 *   sf_page_stride   bytes between scale pages (>= page_size*H*D/16).
 *   num_pages        pages in the pool; page indices outside [0, num_pages) are skipped.
 * `data` must be 16-byte aligned. */
typedef struct {
  uint8_t* data;
  uint8_t* sf;
  int64_t data_page_stride;
  int64_t sf_page_stride;
  int64_t num_pages;
} nvfp4_paged_cache;

/* ABI version of the loaded library (NVFP4KV_ABI_VERSION). */
int32_t nvfp4_abi_version(void);

/* Text of the last failure on this host thread ("" after success). */
const char* nvfp4_last_error_string(void);

/* E4M3 block-scale clamp implied by a recipe ("nvfp4_e4m3_max"): 448 for standard NVFP4
 * (recipe NULL), recipe->e4m3_max under 4over6. Host-only, no device work. */
float nvfp4_e4m3_max(const nvfp4_4over6_config* recipe);

/* Global decode scale of one fp16/bf16 tensor ("make_nvfp4_global_scale", per-tensor form;
 * "NVFP4 4over6 Recipes": the scale must come from the same recipe as the quantizer):
 *   gs = amax(|x|) / (6 * nvfp4_e4m3_max(recipe))   (binary32, one rounding per operation),
 *   gs = 1 when the tensor is all zeros.
 * 6 is the largest E2M1 magnitude. The block holding the tensor's amax then gets the top
 * block scale.
 *   x          device, numel contiguous elements of `dtype`, 16-byte aligned.
 *   numel      >= 0.
 *   scale_out  device, one float, overwritten (it is also the reduction's accumulator, so
 *              it must not alias x).
 * A tensor of at most 65,536 elements is one kernel launch (one CTA scans it and writes gs);
 * a larger one enqueues a 4-byte memset and two kernels (a many-CTA scan, then gs). */
nvfp4_status nvfp4_make_global_scale(const void* x, int32_t dtype, int64_t numel,
                                     const nvfp4_4over6_config* recipe, float* scale_out,
                                     void* stream);

/* Quantize K/V rows and write them into the paged NVFP4 caches
 * ("flashinfer.page.nvfp4_quantize_append_paged_kv_cache").
 * Row i (token i, all heads) of append_key/append_value goes to logical position
 * positions[i] of request batch_indices[i]: page kv_indices[kv_indptr[b] + pos / page_size],
 * slot pos % page_size. Every 16-element block of a (row, head) gets one E4M3 block scale:
 *   standard NVFP4: S = E4M3(min(amax / (6*gs), e4m3_max))           (amax = block max |x|)
 *   4over6 (recipe != NULL): also S_B = E4M3(min(amax / (4*gs), 448)); both candidates are
 *     quantized and dequantized and S_B is kept only if its error is strictly smaller.
 * Elements: q = E2M1_RNE_satfinite(x * (1 / (S*gs))), element 2k in the low nibble.
 *   append_key/_value  device, [nnz, H, D] of `dtype`; a token row is `*_row_stride`
 *                      elements after the previous one, heads and elements contiguous;
 *                      16-byte aligned base, row stride a multiple of 8 elements.
 *   batch_indices, positions  device int32 [nnz].
 *   k_cache, v_cache   the two paged caches (written in place).
 *   kv_indices         device int32 [kv_indptr[batch_size]]: physical pages by request.
 *   num_kv_indices     entries in kv_indices; reads past it are skipped and reported.
 *   kv_indptr          device int32 [batch_size + 1].
 *   kv_last_page_len   device int32 [batch_size] or NULL. Positions at or past
 *                      (pages_b - 1)*page_size + kv_last_page_len[b] are skipped (the
 *                      pages say the space must already be described by these tables).
 *   k_scale, v_scale   global decode scales, positive finite.
 *   recipe             NULL = standard NVFP4; otherwise the 4over6 recipe.
 * Requirements: head_dim % 16 == 0, num_kv_heads >= 1, page_size >= 1, nnz >= 0.
 * Kernels: a call of at most 2^18 blocks per tensor (nnz * H * D / 16; a decode step of up
 * to 4096 tokens at 8 heads of 128) runs a direct-load kernel, which starts sooner; larger
 * calls run a shared-memory ring fed by bulk copies. Both write the same bytes. The
 * environment variable NVFP4KV_TEST_APPEND_KERNEL=ring|direct, read on every call, overrides
 * the choice (for tests). nvfp4_kv_quantize makes the same choice. */
nvfp4_status nvfp4_quantize_append_paged(
    const void* append_key, const void* append_value, int32_t dtype, int64_t nnz,
    int32_t num_kv_heads, int32_t head_dim, int64_t key_row_stride, int64_t value_row_stride,
    const int32_t* batch_indices, const int32_t* positions, nvfp4_paged_cache k_cache,
    nvfp4_paged_cache v_cache, int32_t page_size, int32_t kv_layout,
    const int32_t* kv_indices, int64_t num_kv_indices, const int32_t* kv_indptr,
    const int32_t* kv_last_page_len, int32_t batch_size, float k_scale, float v_scale,
    const nvfp4_4over6_config* recipe, int32_t* dev_status, void* workspace, void* stream);

/* nvfp4_quantize_append_paged with the two global decode scales read from device memory
 * (k_scale, v_scale: one float each, for example the outputs of nvfp4_make_global_scale),
 * so a step needs no host round trip between computing the scales and using them. Same
 * arguments and behaviour otherwise. A scale that is not positive finite is reported as
 * NVFP4_DEV_BAD_SCALE and nothing is written. */
nvfp4_status nvfp4_quantize_append_paged_dev_scale(
    const void* append_key, const void* append_value, int32_t dtype, int64_t nnz,
    int32_t num_kv_heads, int32_t head_dim, int64_t key_row_stride, int64_t value_row_stride,
    const int32_t* batch_indices, const int32_t* positions, nvfp4_paged_cache k_cache,
    nvfp4_paged_cache v_cache, int32_t page_size, int32_t kv_layout,
    const int32_t* kv_indices, int64_t num_kv_indices, const int32_t* kv_indptr,
    const int32_t* kv_last_page_len, int32_t batch_size, const float* k_scale,
    const float* v_scale, const nvfp4_4over6_config* recipe, int32_t* dev_status,
    void* workspace, void* stream);

/* Dequantize a paged NVFP4 cache into contiguous outputs
 * ("flashinfer.quantization.nvfp4_kv_dequantize_paged").
 * For b < batch_size, t < min(seq_lens[b], max_seq_len), h < H, d < D (a length past
 * max_seq_len or past max_pages_per_request * page_size is clamped and reported):
 *   page = block_tables[b, t / page_size], slot = t % page_size,
 *   out[b, t, h, d] = round_out( (e2m1(q) * S) * gs )   in binary32, one final rounding.
 * Positions t >= seq_lens[b] are left unchanged.
 *   block_tables   device [batch_size, max_pages_per_request], int32 or int64 (table_dtype);
 *                  only the first ceil(len/page_size) columns of each row are read.
 *   seq_lens       device int32 [batch_size].
 *   k_scale, v_scale  device float[1] each: the global decode scales.
 *   output_k/_v    device, contiguous [batch_size, max_seq_len, H, D] of out_dtype,
 *                  16-byte aligned.
 * Requirements: head_dim % 16 == 0. */
nvfp4_status nvfp4_dequantize_paged(
    nvfp4_paged_cache k_cache, nvfp4_paged_cache v_cache, int32_t page_size,
    int32_t num_kv_heads, int32_t head_dim, int32_t kv_layout, const void* block_tables,
    int32_t table_dtype, int32_t max_pages_per_request, const int32_t* seq_lens,
    int32_t batch_size, const float* k_scale, const float* v_scale, void* output_k,
    void* output_v, int32_t out_dtype, int32_t max_seq_len, int32_t* dev_status,
    void* workspace, void* stream);

/* Shape of the FP8 copy ("nvfp4_kv_materialize_fp8", returns): max_pages_per_seq =
 * ceil(max_kv_len / page_size); the copy has num_pages + 1 pages, where num_pages is the
 * given value (from kv_page_indptr) or, when num_pages < 0, batch_size*max_pages_per_seq. */
nvfp4_status nvfp4_materialize_fp8_out_pages(int32_t batch_size, int32_t max_kv_len,
                                             int32_t page_size, int64_t num_pages,
                                             int64_t* out_num_pages,
                                             int32_t* max_pages_per_seq);

/* nvfp4_dequantize_paged for callers that cannot hand the library any device memory. This
 * entry point has no counterpart on the pages; it is an addition of this library.
 * The dequantize runs fastest with a work-distribution workspace (NVFP4_WORKSPACE_BYTES).
 * Some callers cannot provide one: an engine whose memory planner owns every byte of device
 * memory and hands out no buffers beyond a call's inputs and outputs, and code that must
 * not call cudaMalloc at all (it runs while the allocator is locked, or must not add
 * allocations that a memory budget did not plan for). With NULL they would get fixed
 * shares, about 13 percent slower on a large batch. This variant instead uses a 16-byte
 * array that the library itself holds in device memory (a file-scope __device__ array:
 * every GPU that loads the library keeps it until the process exits). It allocates
 * nothing: no cudaMalloc, no cudaFree, no allocating library routine.
 *   Arguments, results and requirements: those of nvfp4_dequantize_paged, without
 *   `workspace`. The scratch this call needs is those 16 bytes whatever the sizes passed,
 *   so no size can exceed it; sizes are otherwise checked as for nvfp4_dequantize_paged.
 *   Set-up: the first call on a device looks up the array's device address on that device
 *   (cudaGetSymbolAddress, with the device current) and keeps it. Make that first call
 *   before any stream capture on the device.
 *   Each call clears the array on `stream` (a 16-byte cudaMemsetAsync) and then launches;
 *   the kernel leaves it zero again. Every call shares the one array: calls that may
 *   overlap on the device (other streams, other host threads) race on it and must not be
 *   issued that way. A call rejected by the argument checks still enqueues the clearing. */
nvfp4_status nvfp4_dequantize_paged_no_alloc(
    nvfp4_paged_cache k_cache, nvfp4_paged_cache v_cache, int32_t page_size,
    int32_t num_kv_heads, int32_t head_dim, int32_t kv_layout, const void* block_tables,
    int32_t table_dtype, int32_t max_pages_per_request, const int32_t* seq_lens,
    int32_t batch_size, const float* k_scale, const float* v_scale, void* output_k,
    void* output_v, int32_t out_dtype, int32_t max_seq_len, int32_t* dev_status, void* stream);

/* Write the active pages of a paged NVFP4 cache as FP8 E4M3
 * ("nvfp4_kv_materialize_fp8"; "NVFP4KVMaterializer.run").
 * Request b's page j (j < ceil(seq_lens[b] / page_size)) goes to output page
 *   o = kv_page_indptr[b] + j + 1   (b * max_pages_per_seq + j + 1 when kv_page_indptr is
 *   NULL),
 * out[o, 0|1, h, slot, d] = E4M3_RNE_satfinite(e2m1(q) * S) for every slot of the page
 * (K at 0, V at 1; no global scale), page 0 is set to zero, fp8_block_tables[b, j] = o.
 * Nothing is written for columns j >= ceil(seq_lens[b] / page_size) of request b, nor to
 * output pages above kv_page_indptr[batch_size] ("nvfp4_kv_materialize_fp8": returns).
 *   block_tables   device int32 [batch_size, max_num_pages] when uses_shared_paged_kv_idx,
 *                  else [batch_size, 2, max_num_pages] (K row then V row);
 *                  max_num_pages >= max_pages_per_seq.
 *   seq_lens       device int32 [batch_size]; a length above max_pages_per_seq*page_size
 *                  is clamped to it.
 *   kv_page_indptr device int32 [batch_size + 1] prefix sum starting at 0, or NULL.
 *   num_pages      host copy of kv_page_indptr[batch_size] (required with kv_page_indptr,
 *                  ignored without it).
 *   out            device float8_e4m3fn bytes, contiguous [out_num_pages, 2, H, page_size,
 *                  D], out_num_pages >= num_pages + 1, 32-byte aligned.
 *   fp8_block_tables  device int32 [batch_size, max_pages_per_seq], contiguous.
 *   zero_fp8_block_tables  1: entries past each request's pages are set to 0 (the
 *                  functional API's padding); 0: they are left alone (run(), where the
 *                  caller zeroes the table once per step).
 *   v_scale_layout NVFP4_SF_LINEAR, or NVFP4_SF_INTERLEAVED4 for V scales in the
 *                  4-token-interleaved layout (HND only; K scales are always linear).
 * Requirements (the materializer's): head_dim % 64 == 0, page_size % 4 == 0. Layout HND
 * is the pages' input layout; NHD input is also accepted with linear scales. */
nvfp4_status nvfp4_materialize_fp8(
    nvfp4_paged_cache k_cache, nvfp4_paged_cache v_cache, int32_t page_size,
    int32_t num_kv_heads, int32_t head_dim, int32_t kv_layout, const int32_t* block_tables,
    int32_t max_num_pages, int32_t uses_shared_paged_kv_idx, const int32_t* seq_lens,
    int32_t batch_size, int32_t max_kv_len, const int32_t* kv_page_indptr, int64_t num_pages,
    uint8_t* out, int64_t out_num_pages, int32_t* fp8_block_tables,
    int32_t zero_fp8_block_tables, int32_t v_scale_layout, int32_t* dev_status,
    void* workspace, void* stream);

/* A materialize launch prepared once ("flashinfer.quantization" index, NVFP4KVMaterializer:
 * the static layout is checked when the materializer is built, so that each run() costs
 * the host little more than the launch). Caller-owned plain data: filled by
 * nvfp4_materializer_prepare and only read afterwards. It holds no device memory and needs
 * no release; copies are valid. */
typedef struct {
  int32_t page_size, num_kv_heads, head_dim, kv_layout;
  int32_t uses_shared_paged_kv_idx, v_scale_layout;
  int32_t max_batch_size;  /* the largest batch_size a run may pass */
  int32_t device;          /* CUDA device current at prepare; runs must use it */
  int64_t data_page_stride, sf_page_stride;  /* bytes between pages of both caches */
  int32_t bulk, grid, smem_bytes;            /* launch shape chosen at prepare */
  int32_t stall_test;                        /* NVFP4KV_TEST_STALL_PIPELINE at prepare */
  uint32_t magic;                            /* set by a successful prepare */
  int32_t reserved[3];
} nvfp4_materializer;

/* Check the static layout of a materialize loop once and choose its launch shape.
 *   m                 caller-owned, written here (and on no other call).
 *   page_size, num_kv_heads, head_dim, kv_layout, uses_shared_paged_kv_idx, v_scale_layout
 *                     as for nvfp4_materialize_fp8, with the same requirements.
 *   data_page_stride, sf_page_stride  page strides (bytes) that every run's K and V caches
 *                     will have; at least one page each, data strides a multiple of 16,
 *                     scale strides even.
 *   max_batch_size    1..16384; each run's batch_size must not exceed it (the launch
 *                     reserves shared memory for this many request lengths).
 * Runs on the current device and opts the kernel in to its shared memory (no device
 * memory is allocated and nothing is launched). Errors return the usual status codes and
 * leave m unusable. The pipeline test switch NVFP4KV_TEST_STALL_PIPELINE is read here. */
nvfp4_status nvfp4_materializer_prepare(nvfp4_materializer* m, int32_t page_size,
                                        int32_t num_kv_heads, int32_t head_dim,
                                        int32_t kv_layout, int32_t uses_shared_paged_kv_idx,
                                        int32_t v_scale_layout, int64_t data_page_stride,
                                        int64_t sf_page_stride, int32_t max_batch_size);

/* One materialize with a prepared layout (NVFP4KVMaterializer.run): the arguments and
 * results of nvfp4_materialize_fp8 with zero_fp8_block_tables = 0 (only the active
 * entries of fp8_block_tables are written; the caller zeroes the table once per step),
 * and max_kv_len given as max_pages_per_seq (the table's columns). Per call it checks only
 * what can change between calls: that m was prepared on the current device, the caches'
 * strides and base alignment, batch_size <= m->max_batch_size, the table widths, the
 * output extent and null pointers. One kernel launch on `stream` (batch_size 0: a memset
 * of the zero page); nothing allocated, no host synchronization. */
nvfp4_status nvfp4_materializer_run(const nvfp4_materializer* m, nvfp4_paged_cache k_cache,
                                    nvfp4_paged_cache v_cache, const int32_t* block_tables,
                                    int32_t max_num_pages, const int32_t* seq_lens,
                                    int32_t batch_size, int32_t max_pages_per_seq,
                                    const int32_t* kv_page_indptr, int64_t num_pages,
                                    uint8_t* out, int64_t out_num_pages,
                                    int32_t* fp8_block_tables, int32_t* dev_status,
                                    void* workspace, void* stream);

/* Quantize a contiguous fp16/bf16 tensor to NVFP4 with linear block scales
 * ("flashinfer.quantization" index, "FP4 KV Cache Quantization": nvfp4_kv_quantize).
 * The tensor is `rows` rows of `cols` elements (all leading dimensions flattened); row i
 * starts `row_stride` elements after row i-1. Every 16-element block gets the rule of
 * nvfp4_quantize_append_paged (standard NVFP4, or 4over6 with `recipe`):
 *   input        device, 16-byte aligned, row_stride a multiple of 8 elements, >= cols.
 *   dtype        NVFP4_F16 or NVFP4_BF16.
 *   global_scale device float: the global decode scale (for example from
 *                nvfp4_make_global_scale with the same recipe). Not positive finite:
 *                NVFP4_DEV_BAD_SCALE is reported and nothing is written.
 *   fp4_out      device uint8 [rows, cols/2], contiguous, 8-byte aligned: element 2k of a
 *                row in the low nibble of byte k.
 *   sf_out       device uint8 [rows, cols/16], contiguous: the E4M3 scale of block j.
 * Requirements: cols % 16 == 0, cols > 0, rows >= 0. */
nvfp4_status nvfp4_kv_quantize(const void* input, int32_t dtype, int64_t rows, int32_t cols,
                               int64_t row_stride, const float* global_scale,
                               const nvfp4_4over6_config* recipe, uint8_t* fp4_out,
                               uint8_t* sf_out, int32_t* dev_status, void* workspace,
                               void* stream);

/* Dequantize a contiguous NVFP4 tensor with linear block scales
 * ("flashinfer.quantization" index, "FP4 KV Cache Quantization": nvfp4_kv_dequantize):
 *   out[i, d] = round_out( (e2m1(q[i, d]) * S[i, d/16]) * gs )
 * with the same rounding as nvfp4_dequantize_paged.
 *   fp4          device uint8 [rows, cols/2], contiguous, 8-byte aligned.
 *   sf           device uint8 [rows, cols/16], contiguous.
 *   global_scale device float.
 *   out          device [rows, cols] of out_dtype (NVFP4_F16 or NVFP4_BF16), contiguous,
 *                16-byte aligned.
 *   dev_status   NULL or a device int32: NVFP4_DEV_TIMEOUT if a wait of the bulk-copy
 *                kernel for a shared-memory stage ran out.
 *   workspace    NULL or the work-distribution workspace (see the conventions).
 * Requirements: cols % 16 == 0, cols > 0, rows >= 0. With fp4 and sf 16-byte aligned, out
 * 32-byte aligned and at least 16384 elements, the codes and scales are read in bulk copies
 * of 1024 blocks; otherwise each thread loads its blocks directly. */
nvfp4_status nvfp4_kv_dequantize(const uint8_t* fp4, const uint8_t* sf, int64_t rows,
                                 int32_t cols, const float* global_scale, void* out,
                                 int32_t out_dtype, int32_t* dev_status, void* workspace,
                                 void* stream);

/* Pack a resolved recipe into one int64, for logs and repro tooling
 * ("flashinfer.quantization" index, "NVFP4 4over6 Recipes": nvfp4_4over6_code and its
 * inverse nvfp4_4over6_from_code). The pages do not give the bit layout; this library's is
 *   0            recipe NULL: standard NVFP4 (4over6 off)
 *   bit 0        1: 4over6 on
 *   bit 1        err_mode (0 MAE, 1 MSE)
 *   bit 2        err_use_fast_math
 *   bits 3..31   zero
 *   bits 32..63  the binary32 bit pattern of e4m3_max
 * Host only (no device work, no stream). An invalid recipe (the check every entry point
 * makes) or a NULL `code` returns NVFP4_ERR_INVALID_ARG. */
nvfp4_status nvfp4_4over6_code(const nvfp4_4over6_config* recipe, int64_t* code);

/* Inverse of nvfp4_4over6_code: code 0 gives *is_4over6 = 0 (and leaves *recipe alone);
 * otherwise *is_4over6 = 1 and *recipe is the packed recipe. A code outside the layout, or
 * one that packs an invalid recipe, returns NVFP4_ERR_INVALID_ARG. */
nvfp4_status nvfp4_4over6_from_code(int64_t code, int32_t* is_4over6,
                                    nvfp4_4over6_config* recipe);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4KV_H_ */
