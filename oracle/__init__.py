"""CPU oracle for the NVFP4 paged KV-cache operations -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may
import this package. The product library never loads it, and the two share no code.

The arithmetic lives in ``nvfp4_oracle.c`` (plain C11, IEEE binary32 with no contraction,
loops that follow the per-element definitions of the FlashInfer pages
"flashinfer.page.nvfp4_quantize_append_paged_kv_cache",
"flashinfer.quantization.nvfp4_kv_dequantize_paged",
"flashinfer.quantization.kernels.nvfp4_kv_materialize.nvfp4_kv_materialize_fp8" and the
"NVFP4 4over6 Recipes" section of the "flashinfer.quantization" index). This module only
compiles it and marshals numpy arrays into it.

Every function here is pinned by ``tests/test_oracle_*.py`` against facts the pages and
the number formats fix (library casts, brute force, closed forms, invariants), except the
4-token-interleaved V-scale layout (``interleave4_scales`` and the materialize that reads
it): the pages name that layout without defining it, so its parity is unpinned.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvfp4_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libnvfp4_oracle.so")
_lock = threading.Lock()
_lib = None

NHD, HND = 0, 1
MAE, MSE = 0, 1


def compile_source(src: str, out: str) -> str:
    """Compile an oracle source file with gcc (ISO C11, -ffp-contract=off, OpenMP when
    available) into the shared library `out`."""
    base = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
            "-shared", "-Wl,-Bsymbolic", src, "-o", out + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(out + ".tmp", out)
    return out


def build(force: bool = False) -> str:
    """Compile nvfp4_oracle.c into libnvfp4_oracle.so next to it (if stale)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    return compile_source(_SRC, _LIB_PATH)


class _Recipe(ctypes.Structure):
    _fields_ = [("e4m3_max", ctypes.c_float), ("err_mode", ctypes.c_int32),
                ("err_use_fast_math", ctypes.c_int32)]


@dataclass(frozen=True)
class Recipe:
    """A 4over6 recipe: e4m3_max, err_mode (MAE=0 / MSE=1), err_use_fast_math."""
    e4m3_max: float = 448.0
    err_mode: int = MAE
    err_use_fast_math: bool = False


def _recipe_ptr(r: Optional[Recipe]):
    if r is None:
        return None
    return ctypes.pointer(_Recipe(float(r.e4m3_max), int(r.err_mode), int(r.err_use_fast_math)))


def load(path: str):
    """ctypes handle with prototypes for an oracle library at `path`."""
    L = ctypes.CDLL(path)
    d, u32, i32, i64, f32 = (ctypes.c_double, ctypes.c_uint32, ctypes.c_int32,
                             ctypes.c_int64, ctypes.c_float)
    vp = ctypes.c_void_p
    for name in ("oracle_e2m1_decode", "oracle_e4m3_decode", "oracle_f16_decode",
                 "oracle_bf16_decode"):
        getattr(L, name).restype = d
        getattr(L, name).argtypes = [u32]
    for name in ("oracle_e2m1_encode", "oracle_e4m3_encode", "oracle_f16_encode",
                 "oracle_bf16_encode"):
        getattr(L, name).restype = u32
        getattr(L, name).argtypes = [d]
    L.oracle_e4m3_max.restype = f32
    L.oracle_e4m3_max.argtypes = [vp]
    L.oracle_global_scale.restype = f32
    L.oracle_global_scale.argtypes = [vp, i32, i64, vp]
    L.oracle_quantize_block.restype = i32
    L.oracle_quantize_block.argtypes = [vp, i32, f32, vp, vp, vp, vp, vp]
    L.oracle_row_offsets.restype = None
    L.oracle_row_offsets.argtypes = [i32, i64, i64, i64, i64, i64, i64, i64, i64,
                                     vp, vp]
    L.oracle_quantize_append_paged.restype = None
    L.oracle_quantize_append_paged.argtypes = (
        [vp, vp, i32, i64, i32, i32, i64, i64, vp, vp]
        + [vp, vp, i64, i64, vp, vp, i64, i64]
        + [i32, i32, vp, vp, f32, f32, vp, i32])
    L.oracle_dequantize_paged.restype = None
    L.oracle_dequantize_paged.argtypes = (
        [vp, vp, i64, i64, vp, vp, i64, i64, i32, i32, i32, i32, vp, i32, i32, vp,
         i32, f32, f32, vp, vp, i32, i32, i32])
    L.oracle_materialize_fp8.restype = None
    L.oracle_materialize_fp8.argtypes = (
        [vp, vp, i64, i64, vp, vp, i64, i64, i32, i32, i32, i32, vp, i32, i32, vp,
         i32, i32, vp, vp, vp, i32, i32, i32])
    L.oracle_kv_quantize.restype = None
    L.oracle_kv_quantize.argtypes = [vp, i32, i64, i64, i64, f32, vp, vp, vp, i32]
    L.oracle_kv_dequantize.restype = None
    L.oracle_kv_dequantize.argtypes = [vp, vp, i64, i64, f32, vp, i32, i32]
    L.oracle_max_threads.restype = i32
    L.oracle_max_threads.argtypes = []
    return L


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load(build())
    return _lib


def use(handle) -> None:
    """Make every function of this module call `handle` (a library from load()) instead
    of the built oracle; use(None) restores it. For tests that plant mistakes."""
    global _lib
    with _lock:
        _lib = handle


def max_threads() -> int:
    return int(lib().oracle_max_threads())


def _p(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


# --- formats ---------------------------------------------------------------------------

def e2m1_decode(code: int) -> float:
    return lib().oracle_e2m1_decode(code)


def e2m1_encode(v: float) -> int:
    return lib().oracle_e2m1_encode(v)


def e4m3_decode(b: int) -> float:
    return lib().oracle_e4m3_decode(b)


def e4m3_encode(v: float) -> int:
    return lib().oracle_e4m3_encode(v)


def f16_encode(v: float) -> int:
    return lib().oracle_f16_encode(v)


def f16_decode(b: int) -> float:
    return lib().oracle_f16_decode(b)


def bf16_encode(v: float) -> int:
    return lib().oracle_bf16_encode(v)


def bf16_decode(b: int) -> float:
    return lib().oracle_bf16_decode(b)


# --- operations ------------------------------------------------------------------------

def e4m3_max(recipe: Optional[Recipe]) -> float:
    return float(lib().oracle_e4m3_max(_recipe_ptr(recipe)))


def global_scale(x_bits: np.ndarray, is_bf16: bool, recipe: Optional[Recipe]) -> float:
    """x_bits: raw 16-bit patterns (uint16) of the whole tensor."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16).reshape(-1)
    return float(lib().oracle_global_scale(_p(x), int(is_bf16), x.size, _recipe_ptr(recipe)))


def quantize_block(x16_bits: np.ndarray, is_bf16: bool, gs: float,
                   recipe: Optional[Recipe]):
    """Returns (codes[8] uint8, sf byte, chose_b, err_a, err_b)."""
    x = np.ascontiguousarray(x16_bits, dtype=np.uint16).reshape(16)
    codes = np.zeros(8, np.uint8)
    sf = np.zeros(1, np.uint8)
    ea = np.zeros(1, np.float64)
    eb = np.zeros(1, np.float64)
    chose = lib().oracle_quantize_block(_p(x), int(is_bf16), gs, _recipe_ptr(recipe),
                                        _p(codes), _p(sf), _p(ea), _p(eb))
    return codes, int(sf[0]), bool(chose), float(ea[0]), float(eb[0])


def row_offsets(layout: int, page: int, slot: int, h: int, ps: int, H: int, D: int,
                data_page_stride: int, sf_page_stride: int):
    do = ctypes.c_int64()
    so = ctypes.c_int64()
    lib().oracle_row_offsets(layout, page, slot, h, ps, H, D, data_page_stride,
                             sf_page_stride, ctypes.byref(do), ctypes.byref(so))
    return do.value, so.value


@dataclass
class PagedCache:
    """Host copy of one paged NVFP4 cache (K or V) as flat byte arrays."""
    data: np.ndarray
    sf: np.ndarray
    data_page_stride: int
    sf_page_stride: int


def quantize_append_paged(k_bits, v_bits, is_bf16: bool, nnz: int, H: int, D: int,
                          k_row_stride: int, v_row_stride: int, batch_indices, positions,
                          kc: PagedCache, vc: PagedCache, ps: int, layout: int,
                          kv_indices, kv_indptr, k_scale: float, v_scale: float,
                          recipe: Optional[Recipe], nthreads: int = 0):
    bi = np.ascontiguousarray(batch_indices, np.int32)
    po = np.ascontiguousarray(positions, np.int32)
    ki = np.ascontiguousarray(kv_indices, np.int32)
    kp = np.ascontiguousarray(kv_indptr, np.int32)
    kb = np.ascontiguousarray(k_bits, np.uint16).reshape(-1)
    vb = np.ascontiguousarray(v_bits, np.uint16).reshape(-1)
    lib().oracle_quantize_append_paged(
        _p(kb), _p(vb), int(is_bf16), nnz, H, D, k_row_stride, v_row_stride, _p(bi), _p(po),
        _p(kc.data), _p(kc.sf), kc.data_page_stride, kc.sf_page_stride,
        _p(vc.data), _p(vc.sf), vc.data_page_stride, vc.sf_page_stride,
        ps, layout, _p(ki), _p(kp), k_scale, v_scale, _recipe_ptr(recipe),
        nthreads or max_threads())


def dequantize_paged(kc: PagedCache, vc: PagedCache, ps: int, H: int, D: int, layout: int,
                     block_tables: np.ndarray, seq_lens, k_scale: float, v_scale: float,
                     out_k: np.ndarray, out_v: np.ndarray, out_bf16: bool,
                     nthreads: int = 0):
    """out_k/out_v: uint16 [B, max_seq_len, H, D], written in place for t < seq_lens[b]."""
    bt = np.ascontiguousarray(block_tables)
    assert bt.dtype in (np.int32, np.int64) and bt.ndim == 2
    sl = np.ascontiguousarray(seq_lens, np.int32)
    B, L = out_k.shape[0], out_k.shape[1]
    lib().oracle_dequantize_paged(
        _p(kc.data), _p(kc.sf), kc.data_page_stride, kc.sf_page_stride,
        _p(vc.data), _p(vc.sf), vc.data_page_stride, vc.sf_page_stride,
        ps, H, D, layout, _p(bt), int(bt.dtype == np.int64), bt.shape[1], _p(sl), B,
        k_scale, v_scale, _p(out_k), _p(out_v), int(out_bf16), L, nthreads or max_threads())


def materialize_out_pages(batch_size: int, max_kv_len: int, page_size: int,
                          num_pages: Optional[int] = None):
    """(rows of kv_cache_fp8, max_pages_per_seq) as the materialize page describes them."""
    mpps = -(-max_kv_len // page_size)
    n = num_pages if num_pages is not None else batch_size * mpps
    return n + 1, mpps


def materialize_fp8(kc: PagedCache, vc: PagedCache, ps: int, H: int, D: int, layout: int,
                    block_tables: np.ndarray, shared: bool, seq_lens, max_kv_len: int,
                    kv_page_indptr, out: np.ndarray, fp8_block_tables: np.ndarray,
                    zero_tables: bool = True, nthreads: int = 0, v_interleaved4: bool = False):
    """out: uint8 [n_out_pages, 2, H, ps, D]; fp8_block_tables: int32 [B, mpps].
    v_interleaved4: vc.sf holds the V scales in the 4-token-interleaved layout (HND only)."""
    if v_interleaved4 and (layout != 1 or ps % 4 != 0):
        raise ValueError("4-token-interleaved V scales need HND pages with page_size % 4 == 0")
    bt = np.ascontiguousarray(block_tables, np.int32)
    sl = np.ascontiguousarray(seq_lens, np.int32)
    ip = None if kv_page_indptr is None else np.ascontiguousarray(kv_page_indptr, np.int32)
    mnp = bt.shape[-1]
    lib().oracle_materialize_fp8(
        _p(kc.data), _p(kc.sf), kc.data_page_stride, kc.sf_page_stride,
        _p(vc.data), _p(vc.sf), vc.data_page_stride, vc.sf_page_stride,
        ps, H, D, layout, _p(bt), mnp, int(shared), _p(sl), sl.size, max_kv_len, _p(ip),
        _p(out), _p(fp8_block_tables), int(zero_tables), int(bool(v_interleaved4)),
        nthreads or max_threads())


def interleave4_scales(sf_pages: np.ndarray) -> np.ndarray:
    """Linear HND block scales [pages, H, page_size, D/16] (uint8) rewritten in the
    4-token-interleaved layout the materialize parameters name for V: same shape, and within
    each group of four slots of a head the bytes go block-major, slot-minor (the reading the
    oracle's materialize follows)."""
    P, H, ps, nb = sf_pages.shape
    if ps % 4 != 0:
        raise ValueError("page_size must be divisible by 4")
    g = np.ascontiguousarray(sf_pages).reshape(P, H, ps // 4, 4, nb)
    return np.ascontiguousarray(g.transpose(0, 1, 2, 4, 3)).reshape(P, H, ps, nb)


def kv_quantize(x_bits: np.ndarray, is_bf16: bool, gs: float, recipe: Optional[Recipe] = None,
                nthreads: int = 0):
    """Contiguous quantize of uint16 bits [..., cols] (rows = the product of the leading
    dimensions): returns (codes uint8 [..., cols/2], scales uint8 [..., cols/16])."""
    x = np.ascontiguousarray(x_bits, np.uint16)
    cols = x.shape[-1]
    rows = x.size // cols if cols else 0
    codes = np.zeros(x.shape[:-1] + (cols // 2,), np.uint8)
    sf = np.zeros(x.shape[:-1] + (cols // 16,), np.uint8)
    lib().oracle_kv_quantize(_p(x), int(is_bf16), rows, cols, cols, gs, _recipe_ptr(recipe),
                             _p(codes), _p(sf), nthreads or max_threads())
    return codes, sf


def kv_dequantize(codes: np.ndarray, sf: np.ndarray, gs: float, out_bf16: bool,
                  nthreads: int = 0) -> np.ndarray:
    """Contiguous dequantize: codes uint8 [..., cols/2], scales uint8 [..., cols/16] ->
    uint16 bits [..., cols] of the output type."""
    c = np.ascontiguousarray(codes, np.uint8)
    s = np.ascontiguousarray(sf, np.uint8)
    cols = 2 * c.shape[-1]
    rows = c.size // c.shape[-1] if c.shape[-1] else 0
    out = np.zeros(c.shape[:-1] + (cols,), np.uint16)
    lib().oracle_kv_dequantize(_p(c), _p(s), rows, cols, gs, _p(out), int(out_bf16),
                               nthreads or max_threads())
    return out
