// abi.cu -- the extern "C" entry points of libnvfp4kv: host-side validation (the checks the
// FlashInfer materializer's launcher makes -- dtypes, ranks, inner strides, 16-byte
// alignment and shared extents -- plus the scale values passed by value), then one
// launch sequence on the caller's stream.
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <sstream>
#include <unordered_map>

#include "internal.h"

namespace nvfp4 {

namespace {
thread_local std::string t_error;
}

void set_error(const std::string& msg) { t_error = msg; }
void clear_error() { t_error.clear(); }
nvfp4_status fail(nvfp4_status code, const std::string& msg) {
  t_error = msg;
  return code;
}

nvfp4_status check_launch(const char* what) {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(NVFP4_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
  return NVFP4_OK;
}

nvfp4_status set_dynamic_smem(const void* kernel, size_t bytes, const char* what) {
  const cudaError_t e =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e == cudaSuccess) return NVFP4_OK;
  (void)cudaGetLastError();  // the refusal must not surface as a later launch's error
  return fail(NVFP4_ERR_CUDA, std::string(what) + ": cannot opt in to " + std::to_string(bytes) +
                                  " bytes of dynamic shared memory: " + cudaGetErrorString(e));
}

namespace {
std::mutex g_mu;
std::unordered_map<int, int> g_sms;
std::unordered_map<std::string, int> g_occ;

int current_device() {
  int dev = 0;
  cudaGetDevice(&dev);
  return dev;
}
}  // namespace

PipeTest pipe_test_from_env() {
  const char* v = std::getenv("NVFP4KV_TEST_STALL_PIPELINE");
  PipeTest t = (v != nullptr && v[0] == '1') ? PipeTest{1u << 12, 1, 0} : PipeTest{kWaitLimit, 0, 0};
  const char* k = std::getenv("NVFP4KV_TEST_APPEND_KERNEL");
  if (k != nullptr && std::strcmp(k, "ring") == 0) t.append_kernel = 1;
  if (k != nullptr && std::strcmp(k, "direct") == 0) t.append_kernel = 2;
  return t;
}

int sm_count() {
  const int dev = current_device();
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_sms.find(dev);
  if (it != g_sms.end()) return it->second;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
  g_sms[dev] = n;
  return n;
}

int blocks_per_sm(const void* kernel, int threads, size_t smem) {
  const int dev = current_device();
  std::ostringstream key;
  key << dev << ':' << kernel << ':' << threads << ':' << smem;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_occ.find(key.str());
    if (it != g_occ.end()) return it->second;
  }
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = 1;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  g_occ[key.str()] = n;
  return n;
}

}  // namespace nvfp4

using namespace nvfp4;

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

nvfp4_status check_workspace(const char* fn, const void* workspace) {
  if (workspace && !aligned(workspace, 8))
    return fail(NVFP4_ERR_ALIGNMENT, std::string(fn) + ": workspace must be 8-byte aligned");
  return NVFP4_OK;
}

nvfp4_status check_recipe(const nvfp4_4over6_config* r) {
  if (!r) return NVFP4_OK;
  if (!(std::isfinite(r->e4m3_max) && r->e4m3_max > 0.0f && r->e4m3_max <= 448.0f))
    return fail(NVFP4_ERR_INVALID_ARG, "recipe.e4m3_max must be in (0, 448]");
  if (r->err_mode != NVFP4_ERR_MAE && r->err_mode != NVFP4_ERR_MSE)
    return fail(NVFP4_ERR_INVALID_ARG, "recipe.err_mode must be NVFP4_ERR_MAE or NVFP4_ERR_MSE");
  if (r->err_use_fast_math != 0 && r->err_use_fast_math != 1)
    return fail(NVFP4_ERR_INVALID_ARG, "recipe.err_use_fast_math must be 0 or 1");
  return NVFP4_OK;
}

nvfp4_status check_geometry(const char* fn, int32_t page_size, int32_t H, int32_t D,
                            int32_t layout) {
  std::string f(fn);
  if (page_size < 1) return fail(NVFP4_ERR_INVALID_ARG, f + ": page_size must be >= 1");
  if (H < 1) return fail(NVFP4_ERR_INVALID_ARG, f + ": num_kv_heads must be >= 1");
  if (D < 16 || D % 16 != 0) return fail(NVFP4_ERR_INVALID_ARG, f + ": head_dim must be a positive multiple of 16");
  if (layout != NVFP4_NHD && layout != NVFP4_HND)
    return fail(NVFP4_ERR_INVALID_ARG, f + ": kv_layout must be NVFP4_NHD or NVFP4_HND");
  const int64_t page_elems = static_cast<int64_t>(page_size) * H * D;
  if (page_elems > (int64_t(1) << 30))
    return fail(NVFP4_ERR_UNSUPPORTED, f + ": page_size * num_kv_heads * head_dim above 2^30");
  return NVFP4_OK;
}

nvfp4_status check_cache(const char* fn, const char* name, const nvfp4_paged_cache& c,
                         int32_t page_size, int32_t H, int32_t D) {
  std::string f = std::string(fn) + ": " + name;
  const int64_t data_bytes = static_cast<int64_t>(page_size) * H * (D / 2);
  const int64_t sf_bytes = static_cast<int64_t>(page_size) * H * (D / 16);
  if (c.num_pages < 0) return fail(NVFP4_ERR_INVALID_ARG, f + ".num_pages must be >= 0");
  if (c.num_pages > 0 && (!c.data || !c.sf)) return fail(NVFP4_ERR_INVALID_ARG, f + ": null data or sf pointer");
  if (c.data_page_stride < data_bytes)
    return fail(NVFP4_ERR_INVALID_ARG, f + ".data_page_stride is smaller than a page");
  if (c.sf_page_stride < sf_bytes)
    return fail(NVFP4_ERR_INVALID_ARG, f + ".sf_page_stride is smaller than a page");
  if (!aligned(c.data, 16) || c.data_page_stride % 16 != 0)
    return fail(NVFP4_ERR_ALIGNMENT, f + ": data must be 16-byte aligned with a page stride that is a multiple of 16");
  return NVFP4_OK;
}

}  // namespace

extern "C" {

NVFP4_EXPORT int32_t nvfp4_abi_version(void) { return NVFP4KV_ABI_VERSION; }

NVFP4_EXPORT const char* nvfp4_last_error_string(void) { return t_error.c_str(); }

NVFP4_EXPORT float nvfp4_e4m3_max(const nvfp4_4over6_config* recipe) {
  return recipe ? recipe->e4m3_max : 448.0f;
}

NVFP4_EXPORT nvfp4_status nvfp4_make_global_scale(const void* x, int32_t dtype, int64_t numel,
                                                  const nvfp4_4over6_config* recipe,
                                                  float* scale_out, void* stream) {
  clear_error();
  if (nvfp4_status st = check_recipe(recipe)) return st;
  if (dtype != NVFP4_F16 && dtype != NVFP4_BF16)
    return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_make_global_scale: dtype must be NVFP4_F16 or NVFP4_BF16");
  if (numel < 0) return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_make_global_scale: numel must be >= 0");
  if (!scale_out) return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_make_global_scale: scale_out is null");
  if (numel > 0 && !x) return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_make_global_scale: x is null");
  if (!aligned(x, 16) || !aligned(scale_out, 4))
    return fail(NVFP4_ERR_ALIGNMENT, "nvfp4_make_global_scale: x must be 16-byte aligned");
  const float denom = 6.0f * nvfp4_e4m3_max(recipe);
  return launch_global_scale(x, dtype == NVFP4_BF16, numel, denom, scale_out,
                             static_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace {

// Shared body of the two append entry points: scales by value (k_dev == nullptr) or in
// device memory.
nvfp4_status append_impl(
    const char* fn, const void* append_key, const void* append_value, int32_t dtype,
    int64_t nnz, int32_t num_kv_heads, int32_t head_dim, int64_t key_row_stride,
    int64_t value_row_stride, const int32_t* batch_indices, const int32_t* positions,
    nvfp4_paged_cache k_cache, nvfp4_paged_cache v_cache, int32_t page_size, int32_t kv_layout,
    const int32_t* kv_indices, int64_t num_kv_indices, const int32_t* kv_indptr,
    const int32_t* kv_last_page_len, int32_t batch_size, float k_scale, float v_scale,
    const float* k_dev, const float* v_dev, const nvfp4_4over6_config* recipe,
    int32_t* dev_status, void* workspace, void* stream) {
  clear_error();
  if (nvfp4_status st = check_recipe(recipe)) return st;
  if (nvfp4_status st = check_workspace(fn, workspace)) return st;
  if (nvfp4_status st = check_geometry(fn, page_size, num_kv_heads, head_dim, kv_layout)) return st;
  if (dtype != NVFP4_F16 && dtype != NVFP4_BF16)
    return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_quantize_append_paged: dtype must be NVFP4_F16 or NVFP4_BF16");
  if (nnz < 0) return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_quantize_append_paged: nnz must be >= 0");
  if (batch_size < 0) return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_quantize_append_paged: batch_size must be >= 0");
  if (k_dev == nullptr &&
      (!(std::isfinite(k_scale) && k_scale > 0.0f) || !(std::isfinite(v_scale) && v_scale > 0.0f)))
    return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_quantize_append_paged: k_scale and v_scale must be positive finite");
  if (k_dev != nullptr && (v_dev == nullptr || !aligned(k_dev, 4) || !aligned(v_dev, 4)))
    return fail(NVFP4_ERR_INVALID_ARG, std::string(fn) + ": k_scale and v_scale must be 4-byte aligned device pointers");
  if (nvfp4_status st = check_cache(fn, "k_cache", k_cache, page_size, num_kv_heads, head_dim)) return st;
  if (nvfp4_status st = check_cache(fn, "v_cache", v_cache, page_size, num_kv_heads, head_dim)) return st;
  if (nnz == 0) return NVFP4_OK;
  const int64_t row_elems = static_cast<int64_t>(num_kv_heads) * head_dim;
  if (key_row_stride < row_elems || value_row_stride < row_elems)
    return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_quantize_append_paged: row strides must cover num_kv_heads * head_dim elements");
  if (!append_key || !append_value || !batch_indices || !positions || !kv_indptr ||
      (!kv_indices && num_kv_indices > 0))
    return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_quantize_append_paged: null device pointer");
  if (!aligned(append_key, 16) || !aligned(append_value, 16) || key_row_stride % 8 != 0 ||
      value_row_stride % 8 != 0)
    return fail(NVFP4_ERR_ALIGNMENT, "nvfp4_quantize_append_paged: inputs must be 16-byte aligned with row strides a multiple of 8 elements");
  if (batch_size == 0) return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_quantize_append_paged: rows given but batch_size is 0");
  if (num_kv_indices < 0) return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_quantize_append_paged: num_kv_indices must be >= 0");

  AppendArgs a{};
  a.k = static_cast<const uint8_t*>(append_key);
  a.v = static_cast<const uint8_t*>(append_value);
  a.k_row_bytes = key_row_stride * 2;
  a.v_row_bytes = value_row_stride * 2;
  a.nnz = nnz;
  a.H = num_kv_heads;
  a.D = head_dim;
  a.nb = head_dim / 16;
  a.div_nb = make_div(a.nb);
  a.div_H = make_div(num_kv_heads);
  a.div_ps = make_div(page_size);
  a.div_row_blocks = make_div(static_cast<int64_t>(num_kv_heads) * a.nb);
  a.batch_indices = batch_indices;
  a.positions = positions;
  a.kc = k_cache;
  a.vc = v_cache;
  a.ps = page_size;
  a.layout = kv_layout;
  a.kv_indices = kv_indices;
  a.num_kv_indices = num_kv_indices;
  a.kv_indptr = kv_indptr;
  a.kv_last_page_len = kv_last_page_len;
  a.batch_size = batch_size;
  a.gs[0] = k_scale;
  a.gs[1] = v_scale;
  a.gs_dev[0] = k_dev;
  a.gs_dev[1] = v_dev;
  a.cap_a = nvfp4_e4m3_max(recipe);
  a.neg_zero = 0x80000000u;
  a.pipe = pipe_test_from_env();
  a.status = dev_status;
  a.workspace = workspace;
  int mode = 0;
  if (recipe) mode = 1 + (recipe->err_mode == NVFP4_ERR_MSE ? 1 : 0) + (recipe->err_use_fast_math ? 2 : 0);
  const bool vec256 = aligned(append_key, 32) && aligned(append_value, 32) &&
                      key_row_stride % 16 == 0 && value_row_stride % 16 == 0;
  return launch_append(a, dtype == NVFP4_BF16, mode, vec256, static_cast<cudaStream_t>(stream));
}

}  // namespace

extern "C" {

NVFP4_EXPORT nvfp4_status nvfp4_quantize_append_paged(
    const void* append_key, const void* append_value, int32_t dtype, int64_t nnz,
    int32_t num_kv_heads, int32_t head_dim, int64_t key_row_stride, int64_t value_row_stride,
    const int32_t* batch_indices, const int32_t* positions, nvfp4_paged_cache k_cache,
    nvfp4_paged_cache v_cache, int32_t page_size, int32_t kv_layout,
    const int32_t* kv_indices, int64_t num_kv_indices, const int32_t* kv_indptr,
    const int32_t* kv_last_page_len, int32_t batch_size, float k_scale, float v_scale,
    const nvfp4_4over6_config* recipe, int32_t* dev_status, void* workspace, void* stream) {
  return append_impl("nvfp4_quantize_append_paged", append_key, append_value, dtype, nnz,
                     num_kv_heads, head_dim, key_row_stride, value_row_stride, batch_indices,
                     positions, k_cache, v_cache, page_size, kv_layout, kv_indices,
                     num_kv_indices, kv_indptr, kv_last_page_len, batch_size, k_scale, v_scale,
                     nullptr, nullptr, recipe, dev_status, workspace, stream);
}

NVFP4_EXPORT nvfp4_status nvfp4_quantize_append_paged_dev_scale(
    const void* append_key, const void* append_value, int32_t dtype, int64_t nnz,
    int32_t num_kv_heads, int32_t head_dim, int64_t key_row_stride, int64_t value_row_stride,
    const int32_t* batch_indices, const int32_t* positions, nvfp4_paged_cache k_cache,
    nvfp4_paged_cache v_cache, int32_t page_size, int32_t kv_layout,
    const int32_t* kv_indices, int64_t num_kv_indices, const int32_t* kv_indptr,
    const int32_t* kv_last_page_len, int32_t batch_size, const float* k_scale,
    const float* v_scale, const nvfp4_4over6_config* recipe, int32_t* dev_status,
    void* workspace, void* stream) {
  if (k_scale == nullptr || v_scale == nullptr)
    return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_quantize_append_paged_dev_scale: null scale pointer");
  return append_impl("nvfp4_quantize_append_paged_dev_scale", append_key, append_value, dtype,
                     nnz, num_kv_heads, head_dim, key_row_stride, value_row_stride,
                     batch_indices, positions, k_cache, v_cache, page_size, kv_layout,
                     kv_indices, num_kv_indices, kv_indptr, kv_last_page_len, batch_size, 1.0f,
                     1.0f, k_scale, v_scale, recipe, dev_status, workspace, stream);
}

NVFP4_EXPORT nvfp4_status nvfp4_4over6_code(const nvfp4_4over6_config* recipe, int64_t* code) {
  clear_error();
  if (!code) return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_4over6_code: code is null");
  if (!recipe) {
    *code = 0;
    return NVFP4_OK;
  }
  if (nvfp4_status st = check_recipe(recipe)) return st;
  uint32_t bits;
  std::memcpy(&bits, &recipe->e4m3_max, sizeof(bits));
  const uint64_t c = (static_cast<uint64_t>(bits) << 32) | 1u |
                     (recipe->err_mode == NVFP4_ERR_MSE ? 2u : 0u) |
                     (recipe->err_use_fast_math ? 4u : 0u);
  *code = static_cast<int64_t>(c);
  return NVFP4_OK;
}

NVFP4_EXPORT nvfp4_status nvfp4_4over6_from_code(int64_t code, int32_t* is_4over6,
                                                 nvfp4_4over6_config* recipe) {
  clear_error();
  if (!is_4over6 || !recipe)
    return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_4over6_from_code: null output pointer");
  if (code == 0) {
    *is_4over6 = 0;
    return NVFP4_OK;
  }
  const uint64_t c = static_cast<uint64_t>(code);
  if ((c & 1u) == 0 || (c & 0xFFFFFFF8u) != 0)
    return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_4over6_from_code: not a recipe code");
  nvfp4_4over6_config r;
  const uint32_t bits = static_cast<uint32_t>(c >> 32);
  std::memcpy(&r.e4m3_max, &bits, sizeof(bits));
  r.err_mode = (c & 2u) ? NVFP4_ERR_MSE : NVFP4_ERR_MAE;
  r.err_use_fast_math = (c & 4u) ? 1 : 0;
  if (nvfp4_status st = check_recipe(&r)) return st;
  *recipe = r;
  *is_4over6 = 1;
  return NVFP4_OK;
}

NVFP4_EXPORT nvfp4_status nvfp4_kv_quantize(const void* input, int32_t dtype, int64_t rows,
                                            int32_t cols, int64_t row_stride,
                                            const float* global_scale,
                                            const nvfp4_4over6_config* recipe,
                                            uint8_t* fp4_out, uint8_t* sf_out,
                                            int32_t* dev_status, void* workspace,
                                            void* stream) {
  clear_error();
  const char* fn = "nvfp4_kv_quantize";
  if (nvfp4_status st = check_recipe(recipe)) return st;
  if (nvfp4_status st = check_workspace(fn, workspace)) return st;
  if (dtype != NVFP4_F16 && dtype != NVFP4_BF16)
    return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_kv_quantize: dtype must be NVFP4_F16 or NVFP4_BF16");
  if (cols <= 0 || cols % 16 != 0)
    return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_kv_quantize: cols must be a positive multiple of 16");
  if (rows < 0) return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_kv_quantize: rows must be >= 0");
  if (rows == 0) return NVFP4_OK;
  if (row_stride < cols)
    return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_kv_quantize: row_stride must be >= cols");
  if (!input || !global_scale || !fp4_out || !sf_out)
    return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_kv_quantize: null device pointer");
  if (!aligned(input, 16) || row_stride % 8 != 0 || !aligned(fp4_out, 8) || !aligned(global_scale, 4))
    return fail(NVFP4_ERR_ALIGNMENT, std::string(fn) + ": input must be 16-byte aligned with a row stride a multiple of 8 elements, fp4_out 8-byte aligned");
  AppendArgs a{};
  a.k = static_cast<const uint8_t*>(input);
  a.v = nullptr;
  a.k_row_bytes = row_stride * 2;
  a.nnz = rows;
  a.H = 1;
  a.D = cols;
  a.nb = cols / 16;
  a.div_nb = make_div(a.nb);
  a.div_H = make_div(1);
  a.div_ps = make_div(1);
  a.div_row_blocks = make_div(a.nb);
  a.kc = nvfp4_paged_cache{fp4_out, sf_out, cols / 2, cols / 16, rows};
  a.ps = 1;
  a.layout = NVFP4_NHD;
  a.gs[0] = a.gs[1] = 1.0f;
  a.gs_dev[0] = a.gs_dev[1] = global_scale;
  a.cap_a = nvfp4_e4m3_max(recipe);
  a.neg_zero = 0x80000000u;
  a.pipe = pipe_test_from_env();
  a.status = dev_status;
  a.workspace = workspace;
  a.contig = 1;
  int mode = 0;
  if (recipe) mode = 1 + (recipe->err_mode == NVFP4_ERR_MSE ? 1 : 0) + (recipe->err_use_fast_math ? 2 : 0);
  const bool vec256 = aligned(input, 32) && row_stride % 16 == 0;
  return launch_append(a, dtype == NVFP4_BF16, mode, vec256, static_cast<cudaStream_t>(stream));
}

NVFP4_EXPORT nvfp4_status nvfp4_kv_dequantize(const uint8_t* fp4, const uint8_t* sf,
                                              int64_t rows, int32_t cols,
                                              const float* global_scale, void* out,
                                              int32_t out_dtype, int32_t* dev_status,
                                              void* workspace, void* stream) {
  clear_error();
  if (nvfp4_status st = check_workspace("nvfp4_kv_dequantize", workspace)) return st;
  if (out_dtype != NVFP4_F16 && out_dtype != NVFP4_BF16)
    return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_kv_dequantize: out_dtype must be NVFP4_F16 or NVFP4_BF16");
  if (cols <= 0 || cols % 16 != 0)
    return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_kv_dequantize: cols must be a positive multiple of 16");
  if (rows < 0) return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_kv_dequantize: rows must be >= 0");
  if (rows == 0) return NVFP4_OK;
  if (!fp4 || !sf || !global_scale || !out)
    return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_kv_dequantize: null device pointer");
  if (!aligned(fp4, 8) || !aligned(out, 16) || !aligned(global_scale, 4))
    return fail(NVFP4_ERR_ALIGNMENT, "nvfp4_kv_dequantize: fp4 must be 8-byte aligned and out 16-byte aligned");
  KvDequantArgs a{};
  a.codes = fp4;
  a.sf = sf;
  a.blocks = rows * (cols / 16);
  a.gs = global_scale;
  a.out = static_cast<uint8_t*>(out);
  a.status = dev_status;
  a.pipe = pipe_test_from_env();
  a.workspace = workspace;
  return launch_kv_dequant(a, out_dtype == NVFP4_BF16, aligned(out, 32),
                           static_cast<cudaStream_t>(stream));
}

NVFP4_EXPORT nvfp4_status nvfp4_dequantize_paged(
    nvfp4_paged_cache k_cache, nvfp4_paged_cache v_cache, int32_t page_size,
    int32_t num_kv_heads, int32_t head_dim, int32_t kv_layout, const void* block_tables,
    int32_t table_dtype, int32_t max_pages_per_request, const int32_t* seq_lens,
    int32_t batch_size, const float* k_scale, const float* v_scale, void* output_k,
    void* output_v, int32_t out_dtype, int32_t max_seq_len, int32_t* dev_status,
    void* workspace, void* stream) {
  clear_error();
  const char* fn = "nvfp4_dequantize_paged";
  if (nvfp4_status st = check_workspace(fn, workspace)) return st;
  if (nvfp4_status st = check_geometry(fn, page_size, num_kv_heads, head_dim, kv_layout)) return st;
  if (out_dtype != NVFP4_F16 && out_dtype != NVFP4_BF16)
    return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_dequantize_paged: out_dtype must be NVFP4_F16 or NVFP4_BF16");
  if (table_dtype != NVFP4_I32 && table_dtype != NVFP4_I64)
    return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_dequantize_paged: table_dtype must be NVFP4_I32 or NVFP4_I64");
  if (batch_size < 0 || max_seq_len < 0 || max_pages_per_request < 0)
    return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_dequantize_paged: negative size");
  if (nvfp4_status st = check_cache(fn, "k_cache", k_cache, page_size, num_kv_heads, head_dim)) return st;
  if (nvfp4_status st = check_cache(fn, "v_cache", v_cache, page_size, num_kv_heads, head_dim)) return st;
  if (batch_size == 0 || max_seq_len == 0) return NVFP4_OK;
  if (batch_size > kMaxScanBatch)
    return fail(NVFP4_ERR_UNSUPPORTED, "nvfp4_dequantize_paged: batch_size above 16384");
  if (!block_tables || !seq_lens || !k_scale || !v_scale || !output_k || !output_v)
    return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_dequantize_paged: null device pointer");
  if (!aligned(output_k, 16) || !aligned(output_v, 16) || !aligned(k_scale, 4) || !aligned(v_scale, 4))
    return fail(NVFP4_ERR_ALIGNMENT, "nvfp4_dequantize_paged: outputs must be 16-byte aligned");
  DequantArgs a{};
  a.kc = k_cache;
  a.vc = v_cache;
  a.ps = page_size;
  a.H = num_kv_heads;
  a.D = head_dim;
  a.nb = head_dim / 16;
  a.layout = kv_layout;
  a.div_row_blocks = make_div(static_cast<int64_t>(num_kv_heads) * a.nb);
  a.div_nb = make_div(a.nb);
  a.div_ps = make_div(page_size);
  a.block_tables = block_tables;
  a.max_pages = max_pages_per_request;
  a.seq_lens = seq_lens;
  a.B = batch_size;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.out_k = static_cast<uint8_t*>(output_k);
  a.out_v = static_cast<uint8_t*>(output_v);
  a.L = max_seq_len;
  a.pipe = pipe_test_from_env();
  a.status = dev_status;
  a.workspace = workspace;
  const bool vec256 = aligned(output_k, 32) && aligned(output_v, 32);
  return launch_dequant(a, out_dtype == NVFP4_BF16, table_dtype == NVFP4_I64, vec256,
                        static_cast<cudaStream_t>(stream));
}

NVFP4_EXPORT nvfp4_status nvfp4_materialize_fp8_out_pages(int32_t batch_size, int32_t max_kv_len,
                                                          int32_t page_size, int64_t num_pages,
                                                          int64_t* out_num_pages,
                                                          int32_t* max_pages_per_seq) {
  clear_error();
  if (batch_size < 0 || max_kv_len < 0 || page_size < 1)
    return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_materialize_fp8_out_pages: bad size");
  const int64_t mpps = (static_cast<int64_t>(max_kv_len) + page_size - 1) / page_size;
  const int64_t n = num_pages >= 0 ? num_pages : static_cast<int64_t>(batch_size) * mpps;
  if (out_num_pages) *out_num_pages = n + 1;
  if (max_pages_per_seq) *max_pages_per_seq = static_cast<int32_t>(mpps);
  return NVFP4_OK;
}

NVFP4_EXPORT nvfp4_status nvfp4_materialize_fp8(
    nvfp4_paged_cache k_cache, nvfp4_paged_cache v_cache, int32_t page_size,
    int32_t num_kv_heads, int32_t head_dim, int32_t kv_layout, const int32_t* block_tables,
    int32_t max_num_pages, int32_t uses_shared_paged_kv_idx, const int32_t* seq_lens,
    int32_t batch_size, int32_t max_kv_len, const int32_t* kv_page_indptr, int64_t num_pages,
    uint8_t* out, int64_t out_num_pages, int32_t* fp8_block_tables,
    int32_t zero_fp8_block_tables, int32_t v_scale_layout, int32_t* dev_status,
    void* workspace, void* stream) {
  clear_error();
  const char* fn = "nvfp4_materialize_fp8";
  if (nvfp4_status st = check_workspace(fn, workspace)) return st;
  if (v_scale_layout != NVFP4_SF_LINEAR && v_scale_layout != NVFP4_SF_INTERLEAVED4)
    return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_materialize_fp8: v_scale_layout must be NVFP4_SF_LINEAR or NVFP4_SF_INTERLEAVED4");
  if (nvfp4_status st = check_geometry(fn, page_size, num_kv_heads, head_dim, kv_layout)) return st;
  if (head_dim % 64 != 0) return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_materialize_fp8: head_dim must be divisible by 64");
  if (page_size % 4 != 0) return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_materialize_fp8: page_size must be divisible by 4");
  if (batch_size < 0 || max_kv_len < 0 || max_num_pages < 0)
    return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_materialize_fp8: negative size");
  if (nvfp4_status st = check_cache(fn, "k_cache", k_cache, page_size, num_kv_heads, head_dim)) return st;
  if (nvfp4_status st = check_cache(fn, "v_cache", v_cache, page_size, num_kv_heads, head_dim)) return st;
  if (v_scale_layout == NVFP4_SF_INTERLEAVED4 && kv_layout != NVFP4_HND)
    return fail(NVFP4_ERR_UNSUPPORTED, "nvfp4_materialize_fp8: 4-token-interleaved V scales are defined for HND pages only");
  if (!aligned(k_cache.sf, 2) || !aligned(v_cache.sf, 2) || k_cache.sf_page_stride % 2 != 0 ||
      v_cache.sf_page_stride % 2 != 0)
    return fail(NVFP4_ERR_ALIGNMENT, "nvfp4_materialize_fp8: scale caches must be 2-byte aligned with even page strides");
  const int64_t mpps = (static_cast<int64_t>(max_kv_len) + page_size - 1) / page_size;
  if (max_num_pages < mpps)
    return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_materialize_fp8: block_tables needs at least ceil(max_kv_len / page_size) columns");
  int64_t n = static_cast<int64_t>(batch_size) * mpps;
  if (kv_page_indptr) {
    if (num_pages < 0) return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_materialize_fp8: kv_page_indptr requires num_pages");
    n = num_pages;
  }
  if (out_num_pages < n + 1)
    return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_materialize_fp8: out needs at least num_pages + 1 pages");
  if (!out) return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_materialize_fp8: out is null");
  if (!aligned(out, 32)) return fail(NVFP4_ERR_ALIGNMENT, "nvfp4_materialize_fp8: out must be 32-byte aligned");
  if (batch_size > kMaxScanBatch)
    return fail(NVFP4_ERR_UNSUPPORTED, "nvfp4_materialize_fp8: batch_size above 16384");
  if (batch_size > 0 && (!block_tables || !seq_lens || !fp8_block_tables))
    return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_materialize_fp8: null device pointer");
  if (mpps > INT32_MAX || n + 1 > (int64_t(1) << 31))
    return fail(NVFP4_ERR_UNSUPPORTED, "nvfp4_materialize_fp8: page counts above 2^31");
  MaterializeArgs a{};
  a.kc = k_cache;
  a.vc = v_cache;
  a.ps = page_size;
  a.H = num_kv_heads;
  a.D = head_dim;
  a.layout = kv_layout;
  a.div_page_chunks = make_div(static_cast<int64_t>(page_size) * (head_dim / 32));
  a.div_row_chunks = make_div(head_dim / 32);
  a.div_mpps = make_div(mpps > 0 ? mpps : 1);
  a.block_tables = block_tables;
  a.max_num_pages = max_num_pages;
  a.shared = uses_shared_paged_kv_idx ? 1 : 0;
  a.seq_lens = seq_lens;
  a.B = batch_size;
  a.mpps = static_cast<int32_t>(mpps);
  a.kv_page_indptr = kv_page_indptr;
  a.out = out;
  a.out_num_pages = out_num_pages;
  a.tables = fp8_block_tables;
  a.zero_tables = zero_fp8_block_tables ? 1 : 0;
  a.v_interleaved = v_scale_layout == NVFP4_SF_INTERLEAVED4 ? 1 : 0;
  a.pipe = pipe_test_from_env();
  a.status = dev_status;
  a.workspace = workspace;
  if (batch_size == 0) {
    // nothing active: the copy is just its zero page
    const size_t bytes = static_cast<size_t>(2) * num_kv_heads * page_size * head_dim;
    const cudaError_t e = cudaMemsetAsync(out, 0, bytes, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(NVFP4_ERR_CUDA, std::string("cudaMemsetAsync: ") + cudaGetErrorString(e));
    return NVFP4_OK;
  }
  return launch_materialize(a, static_cast<cudaStream_t>(stream));
}

NVFP4_EXPORT nvfp4_status nvfp4_dequantize_paged_no_alloc(
    nvfp4_paged_cache k_cache, nvfp4_paged_cache v_cache, int32_t page_size,
    int32_t num_kv_heads, int32_t head_dim, int32_t kv_layout, const void* block_tables,
    int32_t table_dtype, int32_t max_pages_per_request, const int32_t* seq_lens,
    int32_t batch_size, const float* k_scale, const float* v_scale, void* output_k,
    void* output_v, int32_t out_dtype, int32_t max_seq_len, int32_t* dev_status, void* stream) {
  clear_error();
  void* scratch = nullptr;
  if (nvfp4_status st = no_alloc_scratch(&scratch)) return st;
  // the work queue must start at zero: clear it on the stream before the launch
  const cudaError_t e =
      cudaMemsetAsync(scratch, 0, NVFP4_WORKSPACE_BYTES, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess)
    return fail(NVFP4_ERR_CUDA, std::string("nvfp4_dequantize_paged_no_alloc: cudaMemsetAsync: ") +
                                    cudaGetErrorString(e));
  return nvfp4_dequantize_paged(k_cache, v_cache, page_size, num_kv_heads, head_dim, kv_layout,
                                block_tables, table_dtype, max_pages_per_request, seq_lens,
                                batch_size, k_scale, v_scale, output_k, output_v, out_dtype,
                                max_seq_len, dev_status, scratch, stream);
}

constexpr uint32_t kMaterializerMagic = 0x4E564D31u;  // "NVM1"

NVFP4_EXPORT nvfp4_status nvfp4_materializer_prepare(
    nvfp4_materializer* m, int32_t page_size, int32_t num_kv_heads, int32_t head_dim,
    int32_t kv_layout, int32_t uses_shared_paged_kv_idx, int32_t v_scale_layout,
    int64_t data_page_stride, int64_t sf_page_stride, int32_t max_batch_size) {
  clear_error();
  const char* fn = "nvfp4_materializer_prepare";
  if (!m) return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_materializer_prepare: m is null");
  m->magic = 0;
  if (v_scale_layout != NVFP4_SF_LINEAR && v_scale_layout != NVFP4_SF_INTERLEAVED4)
    return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_materializer_prepare: v_scale_layout must be NVFP4_SF_LINEAR or NVFP4_SF_INTERLEAVED4");
  if (nvfp4_status st = check_geometry(fn, page_size, num_kv_heads, head_dim, kv_layout)) return st;
  if (head_dim % 64 != 0) return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_materializer_prepare: head_dim must be divisible by 64");
  if (page_size % 4 != 0) return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_materializer_prepare: page_size must be divisible by 4");
  if (v_scale_layout == NVFP4_SF_INTERLEAVED4 && kv_layout != NVFP4_HND)
    return fail(NVFP4_ERR_UNSUPPORTED, "nvfp4_materializer_prepare: 4-token-interleaved V scales are defined for HND pages only");
  if (max_batch_size < 1 || max_batch_size > kMaxScanBatch)
    return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_materializer_prepare: max_batch_size must be in [1, 16384]");
  const int64_t cb = static_cast<int64_t>(page_size) * num_kv_heads * (head_dim / 2);
  const int64_t sb = static_cast<int64_t>(page_size) * num_kv_heads * (head_dim / 16);
  if (data_page_stride < cb || sf_page_stride < sb)
    return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_materializer_prepare: a page stride is smaller than a page");
  if (data_page_stride % 16 != 0 || sf_page_stride % 2 != 0)
    return fail(NVFP4_ERR_ALIGNMENT, "nvfp4_materializer_prepare: data page stride must be a multiple of 16 and scale page stride even");
  // bulk copies also need 16-byte scale strides and a page that fits a stage (bases are
  // checked per run)
  const bool bulk = cb % 16 == 0 && sb % 16 == 0 && cb + sb <= 48 * 1024 && sf_page_stride % 16 == 0;
  MaterializeLaunch c{};
  if (nvfp4_status st = prepare_materialize(bulk, v_scale_layout == NVFP4_SF_INTERLEAVED4,
                                            max_batch_size, cb, sb, &c))
    return st;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return fail(NVFP4_ERR_CUDA, "nvfp4_materializer_prepare: no current CUDA device");
  }
  const char* stall = std::getenv("NVFP4KV_TEST_STALL_PIPELINE");
  *m = nvfp4_materializer{};
  m->page_size = page_size;
  m->num_kv_heads = num_kv_heads;
  m->head_dim = head_dim;
  m->kv_layout = kv_layout;
  m->uses_shared_paged_kv_idx = uses_shared_paged_kv_idx ? 1 : 0;
  m->v_scale_layout = v_scale_layout;
  m->max_batch_size = max_batch_size;
  m->device = dev;
  m->data_page_stride = data_page_stride;
  m->sf_page_stride = sf_page_stride;
  m->bulk = c.bulk;
  m->grid = c.grid;
  m->smem_bytes = c.smem;
  m->stall_test = (stall != nullptr && stall[0] == '1') ? 1 : 0;
  m->magic = kMaterializerMagic;
  return NVFP4_OK;
}

NVFP4_EXPORT nvfp4_status nvfp4_materializer_run(
    const nvfp4_materializer* m, nvfp4_paged_cache k_cache, nvfp4_paged_cache v_cache,
    const int32_t* block_tables, int32_t max_num_pages, const int32_t* seq_lens,
    int32_t batch_size, int32_t max_pages_per_seq, const int32_t* kv_page_indptr,
    int64_t num_pages, uint8_t* out, int64_t out_num_pages, int32_t* fp8_block_tables,
    int32_t* dev_status, void* workspace, void* stream) {
  clear_error();
  if (nvfp4_status st = check_workspace("nvfp4_materializer_run", workspace)) return st;
  if (!m || m->magic != kMaterializerMagic)
    return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_materializer_run: m was not prepared");
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != m->device)
    return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_materializer_run: the current device is not the one m was prepared on");
  if (batch_size < 0 || batch_size > m->max_batch_size)
    return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_materializer_run: batch_size must be in [0, max_batch_size]");
  if (max_pages_per_seq < 0 || max_num_pages < max_pages_per_seq)
    return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_materializer_run: block_tables needs at least max_pages_per_seq columns");
  const nvfp4_paged_cache* cs[2] = {&k_cache, &v_cache};
  for (const nvfp4_paged_cache* c : cs) {
    if (c->data_page_stride != m->data_page_stride || c->sf_page_stride != m->sf_page_stride)
      return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_materializer_run: cache page strides differ from the prepared ones");
    if (c->num_pages < 0 || (c->num_pages > 0 && (!c->data || !c->sf)))
      return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_materializer_run: bad cache pointers or num_pages");
    if (!aligned(c->data, 16) || !aligned(c->sf, m->bulk ? 16 : 2))
      return fail(NVFP4_ERR_ALIGNMENT, "nvfp4_materializer_run: cache data must be 16-byte aligned (scales too for this page shape)");
  }
  int64_t n = static_cast<int64_t>(batch_size) * max_pages_per_seq;
  if (kv_page_indptr) {
    if (num_pages < 0) return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_materializer_run: kv_page_indptr requires num_pages");
    n = num_pages;
  }
  if (!out || !aligned(out, 32) || out_num_pages < n + 1 || n + 1 > (int64_t(1) << 31))
    return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_materializer_run: out must be 32-byte aligned with num_pages + 1 (< 2^31) pages");
  if (batch_size > 0 && (!block_tables || !seq_lens || !fp8_block_tables))
    return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_materializer_run: null device pointer");
  const int32_t ps = m->page_size, H = m->num_kv_heads, D = m->head_dim;
  if (batch_size == 0) {
    const size_t bytes = static_cast<size_t>(2) * H * ps * D;
    const cudaError_t e = cudaMemsetAsync(out, 0, bytes, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(NVFP4_ERR_CUDA, std::string("cudaMemsetAsync: ") + cudaGetErrorString(e));
    return NVFP4_OK;
  }
  MaterializeArgs a{};
  a.kc = k_cache;
  a.vc = v_cache;
  a.ps = ps;
  a.H = H;
  a.D = D;
  a.layout = m->kv_layout;
  a.div_page_chunks = make_div(static_cast<int64_t>(ps) * (D / 32));
  a.div_row_chunks = make_div(D / 32);
  a.div_mpps = make_div(max_pages_per_seq > 0 ? max_pages_per_seq : 1);
  a.block_tables = block_tables;
  a.max_num_pages = max_num_pages;
  a.shared = m->uses_shared_paged_kv_idx;
  a.seq_lens = seq_lens;
  a.B = batch_size;
  a.mpps = max_pages_per_seq;
  a.kv_page_indptr = kv_page_indptr;
  a.out = out;
  a.out_num_pages = out_num_pages;
  a.tables = fp8_block_tables;
  a.zero_tables = 0;
  a.v_interleaved = m->v_scale_layout == NVFP4_SF_INTERLEAVED4 ? 1 : 0;
  a.pipe = m->stall_test ? PipeTest{1u << 12, 1, 0} : PipeTest{kWaitLimit, 0, 0};
  a.status = dev_status;
  a.workspace = workspace;
  const MaterializeLaunch c{m->bulk, m->max_batch_size, m->smem_bytes, m->grid};
  return launch_materialize_prepared(a, c, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
