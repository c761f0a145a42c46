"""GB300 (sm_103a) NVFP4 paged KV-cache operations.

A thin ctypes binding over ``libnvfp4kv.so`` (C ABI in ``include/nvfp4kv.h``): it only
turns torch tensors into pointers, strides and the current CUDA stream. Every step of the
work runs in the library's CUDA kernels; there is no fallback of any kind, and using an op
without the built library raises.

Operations (FlashInfer documentation pages):
  nvfp4_quantize_append_paged  "flashinfer.page.nvfp4_quantize_append_paged_kv_cache"
  nvfp4_dequantize_paged       "flashinfer.quantization.nvfp4_kv_dequantize_paged"
  nvfp4_materialize_fp8        "...kernels.nvfp4_kv_materialize.nvfp4_kv_materialize_fp8"
  NVFP4KVMaterializer          "flashinfer.quantization" index, NVFP4KVMaterializer
  nvfp4_make_global_scale      "flashinfer.quantization" index, make_nvfp4_global_scale
  nvfp4_e4m3_max               "flashinfer.quantization" index, nvfp4_e4m3_max
  nvfp4_kv_quantize,           "flashinfer.quantization" index, FP4 KV Cache Quantization
  nvfp4_kv_dequantize            (contiguous tensors, linear block scales)
  nvfp4_4over6_code,           "flashinfer.quantization" index, NVFP4 4over6 Recipes
  nvfp4_4over6_from_code         (the recipe as one int64)
"""

from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass
from typing import Optional, Sequence, Tuple, Union

import torch

from . import _build

__all__ = [
    "NVFP44Over6Config", "NVFP4KVError", "PagedCache", "load", "nvfp4_e4m3_max",
    "nvfp4_make_global_scale", "nvfp4_quantize_append_paged", "nvfp4_dequantize_paged",
    "nvfp4_materialize_fp8", "nvfp4_materialize_fp8_out_pages", "NVFP4KVMaterializer",
    "paged_caches", "LIB_PATH", "nvfp4_kv_quantize", "nvfp4_kv_dequantize",
    "nvfp4_4over6_code", "nvfp4_4over6_from_code",
]

LIB_PATH = _build.LIB_PATH

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_ALIGNMENT, ERR_CUDA = 0, 1, 2, 3, 4
F16, BF16 = 0, 1
NHD, HND = 0, 1
SF_LINEAR, SF_INTERLEAVED4 = 0, 1  # materialize V block-scale layouts
I32, I64 = 0, 1
DEV_BAD_BATCH, DEV_BAD_POSITION, DEV_BAD_PAGE, DEV_LEN_CLAMPED, DEV_BAD_OUT_PAGE = 1, 2, 4, 8, 16
DEV_TIMEOUT, DEV_BAD_SCALE = 32, 64


class NVFP4KVError(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn} failed with status {code}: {msg}")
        self.code = code


class _Cache(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("sf", ctypes.c_void_p),
                ("data_page_stride", ctypes.c_int64), ("sf_page_stride", ctypes.c_int64),
                ("num_pages", ctypes.c_int64)]


class _Materializer(ctypes.Structure):
    """nvfp4_materializer: a materialize launch prepared once (plain data)."""
    _fields_ = [("page_size", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("kv_layout", ctypes.c_int32),
                ("uses_shared_paged_kv_idx", ctypes.c_int32), ("v_scale_layout", ctypes.c_int32),
                ("max_batch_size", ctypes.c_int32), ("device", ctypes.c_int32),
                ("data_page_stride", ctypes.c_int64), ("sf_page_stride", ctypes.c_int64),
                ("bulk", ctypes.c_int32), ("grid", ctypes.c_int32), ("smem_bytes", ctypes.c_int32),
                ("stall_test", ctypes.c_int32), ("magic", ctypes.c_uint32),
                ("reserved", ctypes.c_int32 * 3)]


class _Config(ctypes.Structure):
    _fields_ = [("e4m3_max", ctypes.c_float), ("err_mode", ctypes.c_int32),
                ("err_use_fast_math", ctypes.c_int32)]


@dataclass(frozen=True)
class NVFP44Over6Config:
    """A 4over6 recipe. Defaults: the full E4M3 range and summed absolute error, evaluated
    in fp32 (the pages name e4m3_max=256 and err_mode="MSE" as the knobs to turn)."""
    e4m3_max: float = 448.0
    err_mode: str = "MAE"
    err_use_fast_math: bool = False

    def _c(self) -> _Config:
        mode = {"MAE": 0, "MSE": 1}[self.err_mode.upper()]
        return _Config(float(self.e4m3_max), mode, int(bool(self.err_use_fast_math)))


_lock = threading.Lock()
_lib = None


def load() -> ctypes.CDLL:
    """Build (if stale) and load libnvfp4kv.so. Raises if it cannot be built or loaded."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.build()
        L = ctypes.CDLL(path)
        vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
        L.nvfp4_abi_version.restype = i32
        L.nvfp4_last_error_string.restype = ctypes.c_char_p
        L.nvfp4_e4m3_max.restype = f32
        L.nvfp4_e4m3_max.argtypes = [vp]
        L.nvfp4_make_global_scale.restype = i32
        L.nvfp4_make_global_scale.argtypes = [vp, i32, i64, vp, vp, vp]
        L.nvfp4_quantize_append_paged.restype = i32
        L.nvfp4_quantize_append_paged.argtypes = [
            vp, vp, i32, i64, i32, i32, i64, i64, vp, vp, _Cache, _Cache, i32, i32, vp, i64, vp,
            vp, i32, f32, f32, vp, vp, vp, vp]
        L.nvfp4_quantize_append_paged_dev_scale.restype = i32
        L.nvfp4_quantize_append_paged_dev_scale.argtypes = [
            vp, vp, i32, i64, i32, i32, i64, i64, vp, vp, _Cache, _Cache, i32, i32, vp, i64, vp,
            vp, i32, vp, vp, vp, vp, vp, vp]
        L.nvfp4_dequantize_paged.restype = i32
        L.nvfp4_dequantize_paged.argtypes = [
            _Cache, _Cache, i32, i32, i32, i32, vp, i32, i32, vp, i32, vp, vp, vp, vp, i32, i32,
            vp, vp, vp]
        L.nvfp4_dequantize_paged_no_alloc.restype = i32
        L.nvfp4_dequantize_paged_no_alloc.argtypes = [
            _Cache, _Cache, i32, i32, i32, i32, vp, i32, i32, vp, i32, vp, vp, vp, vp, i32, i32,
            vp, vp]
        L.nvfp4_materialize_fp8_out_pages.restype = i32
        L.nvfp4_materialize_fp8_out_pages.argtypes = [i32, i32, i32, i64, vp, vp]
        L.nvfp4_materialize_fp8.restype = i32
        L.nvfp4_materialize_fp8.argtypes = [
            _Cache, _Cache, i32, i32, i32, i32, vp, i32, i32, vp, i32, i32, vp, i64, vp, i64, vp,
            i32, i32, vp, vp, vp]
        L.nvfp4_materializer_prepare.restype = i32
        L.nvfp4_materializer_prepare.argtypes = [vp, i32, i32, i32, i32, i32, i32, i64, i64, i32]
        L.nvfp4_materializer_run.restype = i32
        L.nvfp4_materializer_run.argtypes = [
            vp, _Cache, _Cache, vp, i32, vp, i32, i32, vp, i64, vp, i64, vp, vp, vp, vp]
        L.nvfp4_4over6_code.restype = i32
        L.nvfp4_4over6_code.argtypes = [vp, vp]
        L.nvfp4_4over6_from_code.restype = i32
        L.nvfp4_4over6_from_code.argtypes = [i64, vp, vp]
        L.nvfp4_kv_quantize.restype = i32
        L.nvfp4_kv_quantize.argtypes = [vp, i32, i64, i32, i64, vp, vp, vp, vp, vp, vp, vp]
        L.nvfp4_kv_dequantize.restype = i32
        L.nvfp4_kv_dequantize.argtypes = [vp, vp, i64, i32, vp, vp, i32, vp, vp, vp]
        _lib = L
        return L


def _check(fn: str, code: int) -> None:
    if code != OK:
        msg = load().nvfp4_last_error_string().decode(errors="replace")
        raise NVFP4KVError(fn, code, msg)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("nvfp4 ops take CUDA tensors only")
    return ctypes.c_void_p(t.data_ptr())


def _stream(device: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


# Work-distribution workspaces (NVFP4_WORKSPACE_BYTES of device memory, zero on first use
# and left zero by every kernel), one per (device, stream): calls on one stream run one at
# a time, so they can share one; calls on different streams may overlap and get their own.
_workspaces = {}
_dynamic_schedule = True


def set_dynamic_schedule(enabled: bool) -> None:
    """Whether the bulk-copy kernels take work items from a shared counter (the default)
    or give each CTA a fixed share. The results are the same either way."""
    global _dynamic_schedule
    _dynamic_schedule = bool(enabled)


def _ws_stream(device: torch.device):
    """(workspace, stream) arguments for a call on the current stream of `device`."""
    stream = torch.cuda.current_stream(device)
    handle = stream.cuda_stream
    ws = None
    if _dynamic_schedule:
        key = (device.index, handle)
        ws = _workspaces.get(key)
        if ws is None and not torch.cuda.is_current_stream_capturing():
            ws = torch.zeros(2, dtype=torch.int64, device=device)  # 16 bytes, on this stream
            _workspaces[key] = ws
    return (None if ws is None else ctypes.c_void_p(ws.data_ptr())), ctypes.c_void_p(handle)


def _layout(kv_layout: Union[str, int]) -> int:
    if isinstance(kv_layout, int):
        return kv_layout
    return {"NHD": NHD, "HND": HND}[kv_layout.upper()]


def _sf_layout(v_block_scales_layout: Union[str, int]) -> int:
    """'linear' or 'interleaved4' (the 4-token-interleaved V-scale layout, HND only)."""
    if isinstance(v_block_scales_layout, int):
        return v_block_scales_layout
    return {"linear": SF_LINEAR, "interleaved4": SF_INTERLEAVED4}[v_block_scales_layout.lower()]


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.float16:
        return F16
    if dt == torch.bfloat16:
        return BF16
    raise ValueError(f"expected float16 or bfloat16, got {dt}")


def _recipe(r: Optional[NVFP44Over6Config]):
    return None if r is None else ctypes.pointer(r._c())


@dataclass
class PagedCache:
    """One paged NVFP4 cache (K or V): codes and scales with their page strides (bytes)."""
    data: torch.Tensor
    sf: torch.Tensor
    data_page_stride: int
    sf_page_stride: int
    num_pages: int

    def _c(self) -> _Cache:
        return _Cache(self.data.data_ptr(), self.sf.data_ptr(), self.data_page_stride,
                      self.sf_page_stride, self.num_pages)


def _one_cache(data: torch.Tensor, sf: torch.Tensor) -> PagedCache:
    if data.dtype != torch.uint8 or sf.dtype not in (torch.uint8, torch.float8_e4m3fn):
        raise ValueError("paged caches are uint8 codes and uint8 / float8_e4m3fn scales")
    if data.dim() != 4 or sf.dim() != 4:
        raise ValueError("a paged cache tensor is 4-D [pages, ., ., head_dim // 2|16]")
    for t in (data, sf):
        if t.stride(3) != 1 or t.stride(2) != t.shape[3] or t.stride(1) != t.shape[2] * t.shape[3]:
            raise ValueError("paged cache pages must be contiguous inside (page stride may be larger)")
    return PagedCache(data, sf, data.stride(0) * data.element_size(), sf.stride(0) * sf.element_size(),
                      data.shape[0])


def paged_caches(paged_kv_cache, kv_cache_sf) -> Tuple[PagedCache, PagedCache]:
    """(K, V) caches from the pages' tuple form (two 4-D tensors each) or stacked 5-D form
    (K/V on the second dimension)."""
    if isinstance(paged_kv_cache, (tuple, list)):
        return (_one_cache(paged_kv_cache[0], kv_cache_sf[0]),
                _one_cache(paged_kv_cache[1], kv_cache_sf[1]))
    d, s = paged_kv_cache, kv_cache_sf
    if d.dim() != 5 or s.dim() != 5 or d.shape[1] != 2 or s.shape[1] != 2:
        raise ValueError("a stacked cache is 5-D with K/V on the second dimension")
    # the views' data pointers already carry V's offset inside each page
    return _one_cache(d[:, 0], s[:, 0]), _one_cache(d[:, 1], s[:, 1])


def _dims(cache: PagedCache, layout: int):
    t = cache.data
    if layout == NHD:
        return t.shape[1], t.shape[2], t.shape[3] * 2   # page_size, H, D
    return t.shape[2], t.shape[1], t.shape[3] * 2


def nvfp4_e4m3_max(nvfp4_4over6_config: Optional[NVFP44Over6Config] = None) -> float:
    """Block-scale clamp implied by a resolved recipe: 448 standard, e4m3_max under 4over6."""
    return float(load().nvfp4_e4m3_max(_recipe(nvfp4_4over6_config)))


def nvfp4_make_global_scale(x: torch.Tensor,
                            nvfp4_4over6_config: Optional[NVFP44Over6Config] = None,
                            out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Per-tensor global decode scale amax(|x|) / (6 * e4m3_max), as a 1-element fp32
    CUDA tensor (1.0 for an all-zero tensor)."""
    if not x.is_contiguous():
        raise ValueError("x must be contiguous")
    if out is None:
        out = torch.empty(1, dtype=torch.float32, device=x.device)
    _check("nvfp4_make_global_scale", load().nvfp4_make_global_scale(
        _ptr(x), _dtype_code(x.dtype), x.numel(), _recipe(nvfp4_4over6_config), _ptr(out),
        _stream(x.device)))
    return out


def nvfp4_quantize_append_paged(append_key: torch.Tensor, append_value: torch.Tensor,
                                batch_indices: torch.Tensor, positions: torch.Tensor,
                                paged_kv_cache, kv_cache_sf, kv_indices: torch.Tensor,
                                kv_indptr: torch.Tensor, kv_last_page_len: Optional[torch.Tensor],
                                k_scale, v_scale, kv_layout: str = "NHD",
                                nvfp4_4over6: Optional[NVFP44Over6Config] = None,
                                dev_status: Optional[torch.Tensor] = None) -> None:
    """Quantize [nnz, H, D] fp16/bf16 K/V rows and write them into the paged caches.
    k_scale / v_scale: host floats (the pages' form), or 1-element float32 CUDA tensors,
    which the kernel reads on the device."""
    layout = _layout(kv_layout)
    kc, vc = paged_caches(paged_kv_cache, kv_cache_sf)
    ps, H, D = _dims(kc, layout)
    if append_key.dim() != 3 or append_key.shape != append_value.shape:
        raise ValueError("append_key/append_value must both be [nnz, num_kv_heads, head_dim]")
    if append_key.dtype != append_value.dtype:
        raise ValueError("append_key and append_value must have the same dtype")
    nnz = append_key.shape[0]
    for t in (append_key, append_value):
        if t.shape[1:] != (H, D) or t.stride(2) != 1 or t.stride(1) != D:
            raise ValueError("append rows must be [nnz, H, D] with heads and elements contiguous")
    for t in (batch_indices, positions, kv_indices, kv_indptr):
        if t.dtype != torch.int32 or not t.is_contiguous():
            raise ValueError("index tensors must be contiguous int32")
    if kv_last_page_len is not None and kv_last_page_len.dtype != torch.int32:
        raise ValueError("kv_last_page_len must be int32")
    B = kv_indptr.numel() - 1
    common = (_ptr(append_key), _ptr(append_value), _dtype_code(append_key.dtype), nnz, H, D,
              append_key.stride(0) if nnz else H * D, append_value.stride(0) if nnz else H * D,
              _ptr(batch_indices), _ptr(positions), kc._c(), vc._c(), ps, layout,
              _ptr(kv_indices), kv_indices.numel(), _ptr(kv_indptr), _ptr(kv_last_page_len), B)
    tail = (_recipe(nvfp4_4over6), _ptr(dev_status), *_ws_stream(append_key.device))
    if isinstance(k_scale, torch.Tensor) or isinstance(v_scale, torch.Tensor):
        # scales held on the device (e.g. from nvfp4_make_global_scale): no host round trip
        for t in (k_scale, v_scale):
            if not isinstance(t, torch.Tensor) or t.dtype != torch.float32 or t.numel() < 1:
                raise ValueError("device scales must both be float32 CUDA tensors")
        _check("nvfp4_quantize_append_paged_dev_scale",
               load().nvfp4_quantize_append_paged_dev_scale(*common, _ptr(k_scale),
                                                            _ptr(v_scale), *tail))
    else:
        _check("nvfp4_quantize_append_paged", load().nvfp4_quantize_append_paged(
            *common, float(k_scale), float(v_scale), *tail))


def nvfp4_dequantize_paged(paged_kv_cache, kv_cache_sf, block_tables: torch.Tensor,
                           seq_lens: torch.Tensor, k_scale: torch.Tensor, v_scale: torch.Tensor,
                           output_k: torch.Tensor, output_v: torch.Tensor,
                           kv_layout: str = "NHD",
                           dev_status: Optional[torch.Tensor] = None) -> None:
    """Gather and dequantize pages into contiguous [B, max_seq_len, H, D] outputs; positions
    >= seq_lens are left unchanged."""
    layout = _layout(kv_layout)
    kc, vc = paged_caches(paged_kv_cache, kv_cache_sf)
    ps, H, D = _dims(kc, layout)
    if block_tables.dim() != 2 or block_tables.dtype not in (torch.int32, torch.int64) \
            or not block_tables.is_contiguous():
        raise ValueError("block_tables must be a contiguous [batch, max_pages] int32/int64 tensor")
    if seq_lens.dtype != torch.int32 or not seq_lens.is_contiguous():
        raise ValueError("seq_lens must be contiguous int32")
    for o in (output_k, output_v):
        if o.dim() != 4 or not o.is_contiguous() or o.shape[2:] != (H, D):
            raise ValueError("outputs must be contiguous [batch, max_seq_len, H, D]")
    if output_k.shape != output_v.shape or output_k.dtype != output_v.dtype:
        raise ValueError("output_k and output_v must match")
    for s in (k_scale, v_scale):
        if s.dtype != torch.float32 or s.numel() < 1:
            raise ValueError("k_scale/v_scale must be float32 CUDA tensors")
    B, L = output_k.shape[0], output_k.shape[1]
    _check("nvfp4_dequantize_paged", load().nvfp4_dequantize_paged(
        kc._c(), vc._c(), ps, H, D, layout, _ptr(block_tables),
        I64 if block_tables.dtype == torch.int64 else I32, block_tables.shape[1],
        _ptr(seq_lens), B, _ptr(k_scale), _ptr(v_scale), _ptr(output_k), _ptr(output_v),
        _dtype_code(output_k.dtype), L, _ptr(dev_status), *_ws_stream(output_k.device)))


def nvfp4_materialize_fp8_out_pages(batch_size: int, max_kv_len: int, page_size: int,
                                    num_pages: Optional[int] = None) -> Tuple[int, int]:
    """(pages of the FP8 copy, max_pages_per_seq)."""
    n = ctypes.c_int64()
    m = ctypes.c_int32()
    _check("nvfp4_materialize_fp8_out_pages", load().nvfp4_materialize_fp8_out_pages(
        batch_size, max_kv_len, page_size, -1 if num_pages is None else num_pages,
        ctypes.byref(n), ctypes.byref(m)))
    return n.value, m.value


def nvfp4_materialize_fp8(k_cache: torch.Tensor, v_cache: torch.Tensor,
                          k_block_scales: torch.Tensor, v_block_scales: torch.Tensor,
                          block_tables: torch.Tensor, seq_lens: torch.Tensor, max_kv_len: int,
                          uses_shared_paged_kv_idx: bool = True,
                          out: Optional[torch.Tensor] = None,
                          kv_page_indptr: Optional[torch.Tensor] = None,
                          num_pages: Optional[int] = None, kv_layout: str = "HND",
                          fp8_block_tables: Optional[torch.Tensor] = None,
                          zero_fp8_block_tables: bool = True,
                          dev_status: Optional[torch.Tensor] = None,
                          v_block_scales_layout: str = "linear"):
    """Materialize the active pages as FP8 E4M3. Returns (kv_cache_fp8, fp8_block_tables)
    with kv_cache_fp8 [num_pages + 1, 2, H, page_size, D] (page 0 zero) and
    fp8_block_tables [batch, max_pages_per_seq] int32 (padding 0). v_block_scales_layout
    'interleaved4' reads the V scales in the 4-token-interleaved layout (HND pages)."""
    layout = _layout(kv_layout)
    kc = _one_cache(k_cache, k_block_scales)
    vc = _one_cache(v_cache, v_block_scales)
    ps, H, D = _dims(kc, layout)
    B = seq_lens.numel()
    if kv_page_indptr is not None and num_pages is None:
        raise ValueError("kv_page_indptr requires num_pages")
    n_out, mpps = nvfp4_materialize_fp8_out_pages(B, max_kv_len, ps, num_pages)
    dev = k_cache.device
    if out is None:
        out = torch.empty((n_out, 2, H, ps, D), dtype=torch.float8_e4m3fn, device=dev)
    if out.dim() != 5 or out.shape[1:] != (2, H, ps, D) or not out.is_contiguous():
        raise ValueError("out must be contiguous [num_out_pages, 2, H, page_size, head_dim]")
    if fp8_block_tables is None:
        fp8_block_tables = torch.zeros((B, mpps), dtype=torch.int32, device=dev)
    if fp8_block_tables.shape != (B, mpps) or fp8_block_tables.dtype != torch.int32 \
            or not fp8_block_tables.is_contiguous():
        raise ValueError("fp8_block_tables must be contiguous int32 [batch, max_pages_per_seq]")
    if block_tables.dtype != torch.int32 or not block_tables.is_contiguous():
        raise ValueError("block_tables must be contiguous int32")
    shared = bool(uses_shared_paged_kv_idx)
    if block_tables.dim() != (2 if shared else 3) or (not shared and block_tables.shape[1] != 2):
        raise ValueError("block_tables is [batch, max_num_pages] (shared) or [batch, 2, max_num_pages]")
    _check("nvfp4_materialize_fp8", load().nvfp4_materialize_fp8(
        kc._c(), vc._c(), ps, H, D, layout, _ptr(block_tables), block_tables.shape[-1],
        int(shared), _ptr(seq_lens), B, int(max_kv_len), _ptr(kv_page_indptr),
        -1 if num_pages is None else int(num_pages), _ptr(out), out.shape[0],
        _ptr(fp8_block_tables), int(bool(zero_fp8_block_tables)),
        _sf_layout(v_block_scales_layout), _ptr(dev_status), *_ws_stream(dev)))
    return out, fp8_block_tables


class NVFP4KVMaterializer:
    """Validate once, launch many times ("NVFP4KVMaterializer"): the static layout and the
    device are checked at construction (nvfp4_materializer_prepare); run() launches on the
    current stream through nvfp4_materializer_run with caller-owned outputs, allocates
    nothing and does not synchronize, so it can be captured in a CUDA graph. It writes only
    the active table entries (the caller zeroes the table once per step).

    The prepared launch is specific to the caches' page strides and reserves room for
    `max_batch_size` requests; a run with other strides or a larger batch prepares again
    (host work only, once per new shape)."""

    def __init__(self, num_kv_heads: int, page_size: int, head_dim: int,
                 device: Union[str, int, torch.device] = "cuda",
                 uses_shared_paged_kv_idx: bool = True, kv_layout: str = "HND",
                 v_block_scales_layout: str = "linear", max_batch_size: int = 256):
        if page_size % 4 != 0:
            raise ValueError("page_size must be divisible by 4")
        if head_dim % 64 != 0:
            raise ValueError("head_dim must be divisible by 64")
        self.H, self.ps, self.D = num_kv_heads, page_size, head_dim
        self.device = torch.device(device)
        if self.device.type != "cuda":
            raise ValueError("NVFP4KVMaterializer needs a CUDA device")
        self.shared = bool(uses_shared_paged_kv_idx)
        self.layout = _layout(kv_layout)
        self.v_sf_layout = _sf_layout(v_block_scales_layout)
        if self.v_sf_layout == SF_INTERLEAVED4 and self.layout != HND:
            raise ValueError("4-token-interleaved V scales need HND pages")
        if self.device.index is None:
            self.device = torch.device("cuda", torch.cuda.current_device())
        self._lib = load()
        self._prepared = {}
        # the compact page layout, checked now so that a bad layout fails at construction
        self._max_batch = int(max_batch_size)
        self._prepare(self.ps * self.H * self.D // 2, self.ps * self.H * self.D // 16,
                      self._max_batch)

    def _prepare(self, dps: int, sps: int, max_batch: int) -> _Materializer:
        key = (dps, sps, max_batch)
        m = self._prepared.get(key)
        if m is None:
            m = _Materializer()
            with torch.cuda.device(self.device):
                _check("nvfp4_materializer_prepare", self._lib.nvfp4_materializer_prepare(
                    ctypes.byref(m), self.ps, self.H, self.D, self.layout, int(self.shared),
                    self.v_sf_layout, dps, sps, max_batch))
            self._prepared[key] = m
        return m

    def run(self, k_cache, v_cache, k_block_scales, v_block_scales, block_tables, seq_lens,
            kv_page_indptr, *, out: torch.Tensor, fp8_block_tables: torch.Tensor,
            dev_status: Optional[torch.Tensor] = None):
        B, mpps = fp8_block_tables.shape
        kc = _one_cache(k_cache, k_block_scales)
        vc = _one_cache(v_cache, v_block_scales)
        if B > self._max_batch:
            self._max_batch = 1 << (B - 1).bit_length()
        m = self._prepare(kc.data_page_stride, kc.sf_page_stride, self._max_batch)
        _check("nvfp4_materializer_run", self._lib.nvfp4_materializer_run(
            ctypes.byref(m), kc._c(), vc._c(), _ptr(block_tables), block_tables.shape[-1],
            _ptr(seq_lens), B, mpps, _ptr(kv_page_indptr), out.shape[0] - 1, _ptr(out),
            out.shape[0], _ptr(fp8_block_tables), _ptr(dev_status), *_ws_stream(self.device)))
        return out, fp8_block_tables


def _scale_tensor(global_scale, device: torch.device) -> torch.Tensor:
    if isinstance(global_scale, torch.Tensor):
        if global_scale.dtype != torch.float32 or global_scale.numel() < 1:
            raise ValueError("global_scale must be a float32 CUDA tensor")
        return global_scale
    return torch.tensor([float(global_scale)], dtype=torch.float32, device=device)


def nvfp4_kv_quantize(input: torch.Tensor, global_scale,
                      nvfp4_4over6: Optional[NVFP44Over6Config] = None,
                      out: Optional[Tuple[torch.Tensor, torch.Tensor]] = None,
                      dev_status: Optional[torch.Tensor] = None):
    """Quantize a fp16/bf16 tensor [..., D] (D % 16 == 0) to NVFP4 with linear block scales.
    Returns (fp4_data uint8 [..., D/2], block_scales uint8 [..., D/16]); `global_scale` is
    the decode scale (a 1-element float32 CUDA tensor, or a float)."""
    if input.dim() < 1 or input.stride(-1) != 1:
        raise ValueError("input must have a contiguous last dimension")
    cols = input.shape[-1]
    lead = input.shape[:-1]
    x2 = input.reshape(-1, cols) if input.numel() else input.view(0, cols)
    if x2.stride(-1) != 1:
        raise ValueError("input rows must be contiguous")
    rows = x2.shape[0]
    if out is None:
        fp4 = torch.empty((*lead, cols // 2), dtype=torch.uint8, device=input.device)
        sf = torch.empty((*lead, cols // 16), dtype=torch.uint8, device=input.device)
    else:
        fp4, sf = out
        if fp4.shape != (*lead, cols // 2) or sf.shape != (*lead, cols // 16) \
                or not fp4.is_contiguous() or not sf.is_contiguous():
            raise ValueError("out must be contiguous ([..., D/2], [..., D/16]) uint8 tensors")
    gs = _scale_tensor(global_scale, input.device)
    _check("nvfp4_kv_quantize", load().nvfp4_kv_quantize(
        _ptr(x2), _dtype_code(input.dtype), rows, cols, x2.stride(0) if rows > 1 else cols,
        _ptr(gs), _recipe(nvfp4_4over6), _ptr(fp4), _ptr(sf), _ptr(dev_status),
        *_ws_stream(input.device)))
    return fp4, sf


def nvfp4_kv_dequantize(fp4_data: torch.Tensor, block_scales: torch.Tensor, global_scale,
                        output_dtype: torch.dtype = torch.bfloat16,
                        out: Optional[torch.Tensor] = None,
                        dev_status: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Dequantize NVFP4 codes [..., D/2] with linear block scales [..., D/16] to
    output_dtype [..., D]: e2m1 * block_scale * global_scale."""
    if not fp4_data.is_contiguous() or not block_scales.is_contiguous():
        raise ValueError("fp4_data and block_scales must be contiguous")
    cols = 2 * fp4_data.shape[-1]
    lead = fp4_data.shape[:-1]
    if block_scales.shape != (*lead, cols // 16):
        raise ValueError("block_scales must be [..., D/16]")
    rows = fp4_data.numel() // fp4_data.shape[-1] if fp4_data.shape[-1] else 0
    if out is None:
        out = torch.empty((*lead, cols), dtype=output_dtype, device=fp4_data.device)
    elif out.shape != (*lead, cols) or not out.is_contiguous():
        raise ValueError("out must be a contiguous [..., D] tensor")
    gs = _scale_tensor(global_scale, fp4_data.device)
    _check("nvfp4_kv_dequantize", load().nvfp4_kv_dequantize(
        _ptr(fp4_data), _ptr(block_scales), rows, cols, _ptr(gs), _ptr(out),
        _dtype_code(out.dtype), _ptr(dev_status), *_ws_stream(fp4_data.device)))
    return out


def nvfp4_4over6_code(config: Optional[NVFP44Over6Config]) -> int:
    """Pack a resolved recipe (None = standard NVFP4) into the library's int64 code."""
    code = ctypes.c_int64()
    _check("nvfp4_4over6_code", load().nvfp4_4over6_code(_recipe(config), ctypes.byref(code)))
    return code.value


def nvfp4_4over6_from_code(code: int) -> Optional[NVFP44Over6Config]:
    """Inverse of nvfp4_4over6_code: None for standard NVFP4, else the recipe."""
    on = ctypes.c_int32()
    c = _Config()
    _check("nvfp4_4over6_from_code",
           load().nvfp4_4over6_from_code(int(code), ctypes.byref(on), ctypes.byref(c)))
    if not on.value:
        return None
    return NVFP44Over6Config(e4m3_max=float(c.e4m3_max),
                             err_mode="MSE" if c.err_mode == 1 else "MAE",
                             err_use_fast_math=bool(c.err_use_fast_math))
