"""Run one workload through the CPU oracle and through the CUDA library, identically.

Both sides start from the same seeded inputs (workloads.py) and the same sentinel-filled
buffers, and run: global scales over every K and V row the cache will hold -> prefill
append (if any) -> the measured append -> V page moves (separate K/V tables) -> paged
dequantize -> FP8 materialize. Results come back as host numpy arrays for a byte-by-byte
comparison. The oracle side never sees a value produced by the CUDA side.
"""

from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

import oracle as O
import workloads as W

SENT_CACHE = 0xA5
SENT_OUT16 = 0x7C0F  # a NaN in fp16 and a plain value in bf16: never produced here
SENT_FP8 = 0x5A
SENT_TABLE = -7


@dataclass
class Result:
    gs_k: float
    gs_v: float
    k_data: np.ndarray
    k_sf: np.ndarray
    v_data: np.ndarray
    v_sf: np.ndarray
    out_k: Optional[np.ndarray]
    out_v: Optional[np.ndarray]
    fp8: Optional[np.ndarray]
    tables: Optional[np.ndarray]
    status: int = 0


def oracle_recipe(r: Optional[W.Recipe]):
    return None if r is None else O.Recipe(r.e4m3_max, r.err_mode, r.err_use_fast_math)


def gpu_recipe(r: Optional[W.Recipe]):
    import nvfp4_paged_kv_02_gb300 as nv
    if r is None:
        return None
    return nv.NVFP44Over6Config(r.e4m3_max, "MSE" if r.err_mode else "MAE",
                                bool(r.err_use_fast_math))


def strides(w: W.Workload, pad_data: int = 0, pad_sf: int = 0):
    dps = w.ps * w.H * w.D // 2 + pad_data
    sps = w.ps * w.H * w.D // 16 + pad_sf
    return dps, sps


def mat_shape(w: W.Workload):
    return O.materialize_out_pages(w.B, w.max_kv_len, w.ps, w.mat_num_pages)


def run_oracle(w: W.Workload, out_dtype=None, pad_data: int = 0, pad_sf: int = 0,
               do_dequant=True, do_materialize=True, extra_out_pages: int = 0,
               zero_tables=True, nthreads: int = 0) -> Result:
    is_bf16 = w.dtype == torch.bfloat16
    r = oracle_recipe(w.recipe)
    allk, allv = W.bits16(w.all_k()), W.bits16(w.all_v())
    gs_k = O.global_scale(allk, is_bf16, r)
    gs_v = O.global_scale(allv, is_bf16, r)
    dps, sps = strides(w, pad_data, pad_sf)
    mk = lambda: O.PagedCache(np.full(w.num_pages * dps, SENT_CACHE, np.uint8),
                              np.full(w.num_pages * sps, SENT_CACHE, np.uint8), dps, sps)
    kc, vc = mk(), mk()
    HD = w.H * w.D
    if w.prefill_k is not None:
        O.quantize_append_paged(W.bits16(w.prefill_k), W.bits16(w.prefill_v), is_bf16,
                                w.prefill_k.shape[0], w.H, w.D, HD, HD,
                                w.prefill_batch_indices, w.prefill_positions, kc, vc, w.ps,
                                w.layout, w.kv_indices, w.kv_indptr, gs_k, gs_v, r, nthreads)
    O.quantize_append_paged(W.bits16(w.k), W.bits16(w.v), is_bf16, w.nnz, w.H, w.D, HD, HD,
                            w.batch_indices, w.positions, kc, vc, w.ps, w.layout, w.kv_indices,
                            w.kv_indptr, gs_k, gs_v, r, nthreads)
    res = Result(gs_k, gs_v, kc.data, kc.sf, vc.data, vc.sf, None, None, None, None)
    if do_dequant:
        odt = out_dtype or w.dtype
        ok = np.full((w.B, w.max_seq_len, w.H, w.D), SENT_OUT16, np.uint16)
        ov = ok.copy()
        O.dequantize_paged(kc, vc, w.ps, w.H, w.D, w.layout, w.block_tables, w.seq_lens,
                           gs_k, gs_v, ok, ov, odt == torch.bfloat16, nthreads)
        res.out_k, res.out_v = ok, ov
    if w.v_page_move is not None:
        # separate K/V tables: V pages move to their own placement after the dequant
        src, dst = w.v_page_move
        vd = vc.data.reshape(w.num_pages, dps)
        vs = vc.sf.reshape(w.num_pages, sps)
        vd[dst] = vd[src].copy()
        vs[dst] = vs[src].copy()
    if do_materialize:
        n_out, mpps = mat_shape(w)
        out = np.full((n_out + extra_out_pages, 2, w.H, w.ps, w.D), SENT_FP8, np.uint8)
        tbl = np.full((w.B, mpps), SENT_TABLE, np.int32)
        O.materialize_fp8(kc, vc, w.ps, w.H, w.D, w.layout, w.mat_block_tables, w.mat_shared,
                          w.seq_lens, w.max_kv_len, w.kv_page_indptr, out, tbl, zero_tables,
                          nthreads)
        res.fp8, res.tables = out, tbl
    return res


def _dev_cache(w: W.Workload, dps: int, sps: int, dev, stacked: bool):
    """Sentinel-filled device caches in the documented 4-D (or stacked 5-D) shapes, with
    page strides dps / sps bytes."""
    last_d, last_s = w.D // 2, w.D // 16
    inner = (w.ps, w.H) if w.layout == W.NHD else (w.H, w.ps)
    comp_d = w.ps * w.H * last_d
    comp_s = w.ps * w.H * last_s
    if stacked:
        bd = torch.full((w.num_pages, 2, dps), SENT_CACHE, dtype=torch.uint8, device=dev)
        bs = torch.full((w.num_pages, 2, sps), SENT_CACHE, dtype=torch.uint8, device=dev)
        data = bd[:, :, :comp_d].unflatten(2, (*inner, last_d))
        sf = bs[:, :, :comp_s].unflatten(2, (*inner, last_s))
        return data, sf, bd, bs
    out = []
    for _ in range(2):
        bd = torch.full((w.num_pages, dps), SENT_CACHE, dtype=torch.uint8, device=dev)
        bs = torch.full((w.num_pages, sps), SENT_CACHE, dtype=torch.uint8, device=dev)
        out.append((bd[:, :comp_d].unflatten(1, (*inner, last_d)),
                    bs[:, :comp_s].unflatten(1, (*inner, last_s)), bd, bs))
    return out


def run_gpu(w: W.Workload, out_dtype=None, pad_data: int = 0, pad_sf: int = 0,
            stacked: bool = False, do_dequant=True, do_materialize=True,
            extra_out_pages: int = 0, zero_tables=True, device="cuda") -> Result:
    import nvfp4_paged_kv_02_gb300 as nv
    dev = torch.device(device)
    r = gpu_recipe(w.recipe)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    gk = nv.nvfp4_make_global_scale(w.all_k().to(dev).contiguous(), r)
    gv = nv.nvfp4_make_global_scale(w.all_v().to(dev).contiguous(), r)
    gs_k, gs_v = float(gk.item()), float(gv.item())
    dps, sps = strides(w, pad_data, pad_sf)
    if stacked:
        data, sf, bd, bs = _dev_cache(w, dps, sps, dev, True)
        cache = (data, sf)
        raw = [(bd[:, 0], bs[:, 0]), (bd[:, 1], bs[:, 1])]
        kview = (data[:, 0], sf[:, 0])
        vview = (data[:, 1], sf[:, 1])
    else:
        (kd, ks, kbd, kbs), (vd, vs, vbd, vbs) = _dev_cache(w, dps, sps, dev, False)
        cache = ((kd, vd), (ks, vs))
        raw = [(kbd, kbs), (vbd, vbs)]
        kview, vview = (kd, ks), (vd, vs)
    t = lambda a: torch.as_tensor(np.ascontiguousarray(a)).to(dev)
    kv_indices, kv_indptr, last = t(w.kv_indices), t(w.kv_indptr), t(w.kv_last_page_len)
    lay = "NHD" if w.layout == W.NHD else "HND"
    if w.prefill_k is not None:
        nv.nvfp4_quantize_append_paged(
            w.prefill_k.to(dev), w.prefill_v.to(dev), t(w.prefill_batch_indices),
            t(w.prefill_positions), cache[0], cache[1],
            kv_indices, kv_indptr, last, gs_k, gs_v, lay, r, status)
    if w.nnz:
        nv.nvfp4_quantize_append_paged(
            w.k.to(dev), w.v.to(dev), t(w.batch_indices), t(w.positions), cache[0], cache[1],
            kv_indices, kv_indptr, last, gs_k, gs_v, lay, r, status)
    res = Result(gs_k, gs_v, None, None, None, None, None, None, None, None)
    if do_dequant:
        odt = out_dtype or w.dtype
        ok = torch.full((w.B, w.max_seq_len, w.H, w.D), SENT_OUT16, dtype=torch.int32,
                        device=dev).to(torch.int16).view(odt)
        ov = ok.clone()
        nv.nvfp4_dequantize_paged(cache[0], cache[1], t(w.block_tables), t(w.seq_lens), gk, gv,
                                  ok, ov, lay, status)
        res.out_k = ok.view(torch.int16).cpu().numpy().view(np.uint16)
        res.out_v = ov.view(torch.int16).cpu().numpy().view(np.uint16)
    if w.v_page_move is not None:
        src, dst = t(w.v_page_move[0]).long(), t(w.v_page_move[1]).long()
        raw[1][0][dst] = raw[1][0][src].clone()
        raw[1][1][dst] = raw[1][1][src].clone()
    res.k_data, res.k_sf = raw[0][0].cpu().numpy().reshape(-1), raw[0][1].cpu().numpy().reshape(-1)
    res.v_data, res.v_sf = raw[1][0].cpu().numpy().reshape(-1), raw[1][1].cpu().numpy().reshape(-1)
    if do_materialize:
        n_out, mpps = mat_shape(w)
        out = torch.full((n_out + extra_out_pages, 2, w.H, w.ps, w.D), SENT_FP8,
                         dtype=torch.uint8, device=dev).view(torch.float8_e4m3fn)
        tbl = torch.full((w.B, mpps), SENT_TABLE, dtype=torch.int32, device=dev)
        indptr = None if w.kv_page_indptr is None else t(w.kv_page_indptr)
        nv.nvfp4_materialize_fp8(kview[0], vview[0], kview[1], vview[1], t(w.mat_block_tables),
                                 t(w.seq_lens), w.max_kv_len, w.mat_shared, out, indptr,
                                 w.mat_num_pages, lay, tbl, zero_tables, status)
        res.fp8 = out.view(torch.uint8).cpu().numpy()
        res.tables = tbl.cpu().numpy()
    torch.cuda.synchronize(dev)
    res.status = int(status.item())
    return res


def assert_same(a: Result, b: Result, what: str = ""):
    """Bit-exact comparison of every result of two runs (a: CUDA, b: oracle)."""
    assert a.status == 0, f"{what}: device status {a.status:#x}"
    assert np.float32(a.gs_k).view(np.uint32) == np.float32(b.gs_k).view(np.uint32), (what, a.gs_k, b.gs_k)
    assert np.float32(a.gs_v).view(np.uint32) == np.float32(b.gs_v).view(np.uint32), (what, a.gs_v, b.gs_v)
    for name in ("k_data", "k_sf", "v_data", "v_sf", "out_k", "out_v", "fp8", "tables"):
        x, y = getattr(a, name), getattr(b, name)
        if x is None and y is None:
            continue
        assert x.shape == y.shape, (what, name, x.shape, y.shape)
        bad = np.flatnonzero(x.reshape(-1) != y.reshape(-1))
        assert bad.size == 0, (f"{what}: {name} differs at {bad.size} of {x.size} positions; "
                               f"first {bad[:8].tolist()} gpu={x.reshape(-1)[bad[:8]].tolist()} "
                               f"oracle={y.reshape(-1)[bad[:8]].tolist()}")


# ---- materialize with V scales in the 4-token-interleaved layout ---------------------------

def interleaved_v(w: W.Workload, vc: O.PagedCache) -> O.PagedCache:
    """A copy of an HND host cache whose V scale pages are rewritten by the oracle's layout
    writer (the codes are shared)."""
    body = w.H * w.ps * (w.D // 16)
    sf = vc.sf.copy()
    pages = sf.reshape(w.num_pages, vc.sf_page_stride)
    pages[:, :body] = O.interleave4_scales(
        pages[:, :body].reshape(w.num_pages, w.H, w.ps, w.D // 16)).reshape(w.num_pages, body)
    return O.PagedCache(vc.data, sf, vc.data_page_stride, vc.sf_page_stride)


def hnd_views(w: W.Workload, c: O.PagedCache, dev):
    """The documented HND 4-D device views [pages, H, page_size, D/2 | D/16] of a host cache,
    with its page strides."""
    bd = torch.from_numpy(c.data.copy()).to(dev).view(w.num_pages, c.data_page_stride)
    bs = torch.from_numpy(c.sf.copy()).to(dev).view(w.num_pages, c.sf_page_stride)
    d = bd[:, : w.H * w.ps * w.D // 2].unflatten(1, (w.H, w.ps, w.D // 2))
    s = bs[:, : w.H * w.ps * w.D // 16].unflatten(1, (w.H, w.ps, w.D // 16))
    return d, s


@dataclass
class InterleavedResult:
    got: np.ndarray
    want: np.ndarray
    got_tables: np.ndarray
    want_tables: np.ndarray
    status: int


def run_materialize_interleaved(w: W.Workload, kc: O.PagedCache, vc: O.PagedCache,
                                extra_out_pages: int = 0, zero_tables: bool = True,
                                use_class: bool = False, device="cuda") -> InterleavedResult:
    """FP8 materialize of one HND host cache pair whose V scales are rewritten in the
    4-token-interleaved layout: the oracle and the CUDA library read the same bytes."""
    import nvfp4_paged_kv_02_gb300 as nv
    dev = torch.device(device)
    vil = interleaved_v(w, vc)
    n_out, mpps = mat_shape(w)
    n_out += extra_out_pages
    want = np.full((n_out, 2, w.H, w.ps, w.D), SENT_FP8, np.uint8)
    want_tbl = np.full((w.B, mpps), SENT_TABLE, np.int32)
    O.materialize_fp8(kc, vil, w.ps, w.H, w.D, W.HND, w.mat_block_tables, w.mat_shared,
                      w.seq_lens, w.max_kv_len, w.kv_page_indptr, want, want_tbl, zero_tables,
                      v_interleaved4=True)
    kd, ks = hnd_views(w, kc, dev)
    vd, vs = hnd_views(w, vil, dev)
    t = lambda a: torch.as_tensor(np.ascontiguousarray(a)).to(dev)
    out = torch.full((n_out, 2, w.H, w.ps, w.D), SENT_FP8, dtype=torch.uint8,
                     device=dev).view(torch.float8_e4m3fn)
    tbl = torch.full((w.B, mpps), SENT_TABLE, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    indptr = None if w.kv_page_indptr is None else t(w.kv_page_indptr)
    if use_class:
        m = nv.NVFP4KVMaterializer(w.H, w.ps, w.D, dev, uses_shared_paged_kv_idx=w.mat_shared,
                                   v_block_scales_layout="interleaved4")
        m.run(kd, vd, ks, vs, t(w.mat_block_tables), t(w.seq_lens), indptr, out=out,
              fp8_block_tables=tbl, dev_status=status)
    else:
        nv.nvfp4_materialize_fp8(kd, vd, ks, vs, t(w.mat_block_tables), t(w.seq_lens),
                                 w.max_kv_len, w.mat_shared, out, indptr, w.mat_num_pages, "HND",
                                 tbl, zero_tables, status, v_block_scales_layout="interleaved4")
    torch.cuda.synchronize(dev)
    return InterleavedResult(out.view(torch.uint8).cpu().numpy(), want, tbl.cpu().numpy(),
                             want_tbl, int(status.item()))
