// internal.h -- host-side declarations shared by the translation units of libnvfp4kv.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <string>

#include "../../include/nvfp4kv.h"
#include "device.cuh"
#include "pipeline.cuh"

#define NVFP4_EXPORT __attribute__((visibility("default")))

namespace nvfp4 {

// Per-thread error text behind nvfp4_last_error_string().
void set_error(const std::string& msg);
void clear_error();
nvfp4_status fail(nvfp4_status code, const std::string& msg);
// Check the launch that was just enqueued.
nvfp4_status check_launch(const char* what);
// Opt `kernel` in to `bytes` of dynamic shared memory; a refusal is reported as
// NVFP4_ERR_CUDA with the byte count (the launch would otherwise fail without the cause).
nvfp4_status set_dynamic_smem(const void* kernel, size_t bytes, const char* what);

// Streaming multiprocessors of the current device.
int sm_count();
// Resident CTAs per SM for `kernel` at `threads` threads and `smem` dynamic bytes
// (cached per kernel and device).
int blocks_per_sm(const void* kernel, int threads, size_t smem);

// Pipeline test control from the environment (NVFP4KV_TEST_STALL_PIPELINE=1).
PipeTest pipe_test_from_env();

// Largest batch the page-scan kernels keep in shared memory (one int32 per request).
constexpr int kMaxScanBatch = 16384;

// ---- append ------------------------------------------------------------------------------
struct AppendArgs {
  const uint8_t* k;
  const uint8_t* v;
  int64_t k_row_bytes;
  int64_t v_row_bytes;
  int64_t nnz;
  int32_t H, D, nb;
  Div div_nb, div_H, div_ps, div_row_blocks;
  const int32_t* batch_indices;
  const int32_t* positions;
  nvfp4_paged_cache kc, vc;
  int32_t ps;
  int32_t layout;
  const int32_t* kv_indices;
  int64_t num_kv_indices;
  const int32_t* kv_indptr;
  const int32_t* kv_last_page_len;
  int32_t batch_size;
  float gs[2];
  const float* gs_dev[2];  // when set, the scales are read from device memory instead
  float cap_a;
  uint32_t neg_zero;  // 0x80000000 (-0.0f), passed at run time for hsq2_rn
  PipeTest pipe;
  int32_t* status;
  void* workspace;  // NVFP4_WORKSPACE_BYTES (dynamic schedule of the ring kernel) or null
  // Contiguous form (nvfp4_kv_quantize): row i goes to kc.data + i * H*D/2 and
  // kc.sf + i * H*D/16; no index arrays are read, and v is null.
  int32_t contig;
};
// mode: 0 standard NVFP4; 1/2 4over6 binary32 MAE/MSE; 3/4 4over6 binary16 MAE/MSE.
nvfp4_status launch_append(const AppendArgs& a, bool bf16, int mode, bool vec256,
                           cudaStream_t stream);

// ---- dequantize --------------------------------------------------------------------------
struct DequantArgs {
  nvfp4_paged_cache kc, vc;
  int32_t ps, H, D, nb, layout;
  Div div_row_blocks, div_nb, div_ps;
  const void* block_tables;
  int64_t max_pages;
  const int32_t* seq_lens;
  int32_t B;
  const float* k_scale;
  const float* v_scale;
  uint8_t* out_k;
  uint8_t* out_v;
  int32_t L;
  PipeTest pipe;
  int32_t* status;
  void* workspace;  // NVFP4_WORKSPACE_BYTES (dynamic schedule of the ring kernel) or null
  int32_t split;    // the ring kernel may hand out halves of a page (set at launch)
};
// Contiguous dequantize (nvfp4_kv_dequantize): block k of the flattened [rows, cols] codes
// (8 bytes at codes + 8k, scale byte sf[k]) becomes 16 outputs at out + 32k bytes.
struct KvDequantArgs {
  const uint8_t* codes;
  const uint8_t* sf;
  int64_t blocks;  // rows * cols / 16
  const float* gs;
  uint8_t* out;
  int32_t* status;  // may be null
  PipeTest pipe;
  void* workspace;  // null: fixed shares
};
nvfp4_status launch_kv_dequant(const KvDequantArgs& a, bool out_bf16, bool vec256,
                               cudaStream_t stream);

nvfp4_status launch_dequant(const DequantArgs& a, bool out_bf16, bool bt64, bool vec256,
                            cudaStream_t stream);
// Device address (on the current device) of the library-held scratch that
// nvfp4_dequantize_paged_no_alloc uses as its workspace; looked up once per device.
nvfp4_status no_alloc_scratch(void** out);

// ---- materialize -------------------------------------------------------------------------
struct MaterializeArgs {
  nvfp4_paged_cache kc, vc;
  int32_t ps, H, D, layout;
  Div div_page_chunks, div_row_chunks, div_mpps;
  const int32_t* block_tables;
  int64_t max_num_pages;
  int32_t shared;
  const int32_t* seq_lens;
  int32_t B;
  int32_t mpps;
  const int32_t* kv_page_indptr;
  uint8_t* out;
  int64_t out_num_pages;
  int32_t* tables;
  int32_t zero_tables;
  int32_t v_interleaved;  // V scales in the 4-token-interleaved layout (HND pages)
  PipeTest pipe;
  int32_t* status;
  void* workspace;  // NVFP4_WORKSPACE_BYTES (dynamic schedule of the ring kernel) or null
};
nvfp4_status launch_materialize(const MaterializeArgs& a, cudaStream_t stream);

// A materialize launch configuration chosen once (the prepared form).
struct MaterializeLaunch {
  int32_t bulk;   // 1: the bulk-copy ring, 0: the direct-load kernel
  int32_t max_B;  // requests the shared-memory scan has room for
  int32_t smem;   // dynamic shared memory bytes
  int32_t grid;   // CTAs
};
// Choose the kernel and its launch shape for pages of cb code bytes and sb scale bytes and
// up to max_B requests; opts the kernel in to its shared memory.
nvfp4_status prepare_materialize(bool bulk, bool v_interleaved, int max_B, int64_t cb,
                                 int64_t sb, MaterializeLaunch* out);
nvfp4_status launch_materialize_prepared(const MaterializeArgs& a, const MaterializeLaunch& c,
                                         cudaStream_t stream);

// ---- global scale ------------------------------------------------------------------------
nvfp4_status launch_global_scale(const void* x, bool bf16, int64_t numel, float denom,
                                 float* out, cudaStream_t stream);

}  // namespace nvfp4
