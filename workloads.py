"""Seeded synthetic inputs for the NVFP4 paged KV-cache operations.

This module only draws random numbers and lays out page tables; it holds none of the
quantization arithmetic. Tests feed the same bytes to the CPU oracle and to the CUDA
library, and the benchmark uses the same recipes.

Workloads (the shapes of the FlashInfer pages' APIs: append rows [nnz, H, D], paged caches
NHD [pages, page_size, H, .] / HND [pages, H, page_size, .], block tables [B, max_pages]):

  tiny         B=2, seq_lens {37, 64}, page_size 16, H=2, D=64, NHD, bf16 N(0,1), 8 pages in
               a random permutation; append everything, dequantize, materialize (shared).
  decode       B=64, existing lengths U[512, 4096] plus one new token each, page_size 16,
               H=8, D=128, HND, bf16 N(0,1), pool = used pages + 10% slack, permuted.
  prefill      B=8 x 8192 tokens, page_size 32, H=8, D=128, NHD, fp16 Student-t (nu=3) with
               round(0.001*H*D) (head, channel) columns scaled x20; 4over6 MSE, e4m3_max 256.
  materialize  B=32, lengths round(exp(U[ln 128, ln 32768])), page_size 64, H=8, D=128, HND,
               separate K/V page tables, compact kv_page_indptr; bf16 N(0,1) pre-fill.
  large_pool   B=256, lengths U[1024, 16384], page_size 16, H=8, D=128, HND, a ~40 GB pool
               (K+V codes and scales) with the active pages placed at random; bf16
               N(0, sigma^2) with sigma ~ U[0.5, 4] per (K/V, head); 4over6 MAE, e4m3_max
               256, fp16 error.

Host generation uses numpy PCG64(seed). The large pool's K/V values (9 GB) are drawn on the
device with a seeded torch generator instead; tests copy the rows they check back to the host.
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

NHD, HND = 0, 1


@dataclass
class Recipe:
    e4m3_max: float = 448.0
    err_mode: int = 0  # 0 MAE, 1 MSE
    err_use_fast_math: bool = False


@dataclass
class Workload:
    name: str
    B: int
    H: int
    D: int
    ps: int
    layout: int
    dtype: torch.dtype
    recipe: Optional[Recipe]
    num_pages: int                     # physical pages in each of the K and V pools
    # rows appended by the measured append call
    k: torch.Tensor                    # [nnz, H, D]
    v: torch.Tensor
    batch_indices: np.ndarray          # int32 [nnz]
    positions: np.ndarray              # int32 [nnz]
    # page table after the append (CSR form, as the append API takes it)
    kv_indices: np.ndarray             # int32 [kv_indptr[-1]]
    kv_indptr: np.ndarray              # int32 [B+1]
    kv_last_page_len: np.ndarray       # int32 [B]
    # dequantize inputs
    seq_lens: np.ndarray               # int32 [B], lengths after the append
    block_tables: np.ndarray           # [B, max_pages] int32 or int64
    max_seq_len: int
    # materialize inputs
    mat_shared: bool = True
    mat_block_tables: Optional[np.ndarray] = None  # int32 [B, mnp] or [B, 2, mnp]
    max_kv_len: int = 0
    kv_page_indptr: Optional[np.ndarray] = None    # int32 [B+1]
    mat_num_pages: Optional[int] = None
    # rows appended before the measured call (decode-style workloads), same page table
    prefill_k: Optional[torch.Tensor] = None
    prefill_v: Optional[torch.Tensor] = None
    prefill_batch_indices: Optional[np.ndarray] = None
    prefill_positions: Optional[np.ndarray] = None
    # after all appends, V page src[i] is moved to dst[i] (separate K/V page tables)
    v_page_move: Optional[tuple] = None
    extra: dict = field(default_factory=dict)

    @property
    def nnz(self) -> int:
        return int(self.k.shape[0])

    def all_k(self) -> torch.Tensor:
        """Every K row the cache ends up holding (prefill rows first)."""
        return self.k if self.prefill_k is None else torch.cat([self.prefill_k, self.k])

    def all_v(self) -> torch.Tensor:
        return self.v if self.prefill_v is None else torch.cat([self.prefill_v, self.v])


def bits16(t: torch.Tensor) -> np.ndarray:
    """Raw 16-bit patterns of a CPU fp16/bf16 tensor as a uint16 numpy array."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _to_dtype(x: np.ndarray, dtype: torch.dtype) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(dtype)


def _csr_pages(lens: np.ndarray, ps: int, perm: np.ndarray):
    """Assign ceil(len/ps) physical pages per request from `perm`, in order."""
    npages = (lens + ps - 1) // ps
    indptr = np.zeros(len(lens) + 1, np.int32)
    indptr[1:] = np.cumsum(npages)
    indices = perm[: int(indptr[-1])].astype(np.int32)
    last = np.where(lens > 0, lens - (npages - 1) * ps, 0).astype(np.int32)
    return indices, indptr, last, npages


def _dense_table(indices, indptr, width, dtype=np.int32, pad=-1):
    B = len(indptr) - 1
    bt = np.full((B, width), pad, dtype=dtype)
    for b in range(B):
        n = indptr[b + 1] - indptr[b]
        bt[b, :n] = indices[indptr[b]: indptr[b + 1]]
    return bt


def _rows_for(lens_from: np.ndarray, lens_to: np.ndarray):
    """(batch_indices, positions) of the rows that extend each request from -> to."""
    bi, pos = [], []
    for b, (a, c) in enumerate(zip(lens_from, lens_to)):
        bi.append(np.full(c - a, b, np.int32))
        pos.append(np.arange(a, c, dtype=np.int32))
    if not bi:
        return np.zeros(0, np.int32), np.zeros(0, np.int32)
    return np.concatenate(bi), np.concatenate(pos)


def make_paged(name: str, seed: int, B: int, H: int, D: int, ps: int, layout: int,
               dtype: torch.dtype, lens_old: np.ndarray, lens_new: np.ndarray,
               recipe: Optional[Recipe] = None, slack: float = 0.0, sampler=None,
               bt_dtype=np.int32, bt_pad: int = -1, mat_shared: bool = True,
               compact_indptr: bool = False, max_kv_len: Optional[int] = None,
               extra_pages: int = 0) -> Workload:
    """Generic paged workload: requests grow from lens_old to lens_new; rows of the
    existing prefix are the prefill, new rows are the measured append."""
    rng = np.random.Generator(np.random.PCG64(seed))
    lens_old = np.asarray(lens_old, np.int64)
    lens_new = np.asarray(lens_new, np.int64)
    used = int(((lens_new + ps - 1) // ps).sum())
    P = max(used + int(np.ceil(used * slack)) + extra_pages, 1)
    perm = rng.permutation(P).astype(np.int32)
    indices, indptr, last, npages = _csr_pages(lens_new, ps, perm)
    max_pages = max(int(npages.max()) if B else 0, 1)
    bt = _dense_table(indices, indptr, max_pages, bt_dtype, bt_pad)
    sampler = sampler or (lambda r, n: r.standard_normal((n, H, D), dtype=np.float32))
    bi_pre, pos_pre = _rows_for(np.zeros_like(lens_old), lens_old)
    bi, pos = _rows_for(lens_old, lens_new)
    n_all = len(bi_pre) + len(bi)
    kk = _to_dtype(sampler(rng, n_all), dtype)
    vv = _to_dtype(sampler(rng, n_all), dtype)
    npre = len(bi_pre)
    L = int(lens_new.max()) if B else 0
    mkl = max_kv_len if max_kv_len is not None else max(L, 1)
    mpps = -(-mkl // ps)
    w = Workload(
        name=name, B=B, H=H, D=D, ps=ps, layout=layout, dtype=dtype, recipe=recipe,
        num_pages=P, k=kk[npre:], v=vv[npre:], batch_indices=bi, positions=pos,
        kv_indices=indices, kv_indptr=indptr, kv_last_page_len=last,
        seq_lens=lens_new.astype(np.int32), block_tables=bt, max_seq_len=max(L, 1),
        mat_shared=mat_shared, max_kv_len=mkl)
    if npre:
        w.prefill_k, w.prefill_v = kk[:npre], vv[:npre]
        w.prefill_batch_indices, w.prefill_positions = bi_pre, pos_pre
    # materialize page tables: int32, at least mpps columns
    mbt = _dense_table(indices, indptr, max(mpps, max_pages), np.int32, bt_pad)
    if mat_shared:
        w.mat_block_tables = mbt
    else:
        # V pages live elsewhere: move each V page to a second random placement.
        perm_v = rng.permutation(P).astype(np.int32)
        src = indices.copy()
        dst = perm_v[: len(indices)]
        w.v_page_move = (src, dst)
        vbt = _dense_table(dst, indptr, mbt.shape[1], np.int32, bt_pad)
        w.mat_block_tables = np.stack([mbt, vbt], axis=1)
    if compact_indptr:
        kp = np.zeros(B + 1, np.int32)
        kp[1:] = np.cumsum(npages)
        w.kv_page_indptr = kp
        w.mat_num_pages = int(kp[-1])
    return w


# ---- the named workloads ---------------------------------------------------------------

def tiny(seed: int = 0) -> Workload:
    lens = np.array([37, 64])
    return make_paged("tiny", seed, B=2, H=2, D=64, ps=16, layout=NHD, dtype=torch.bfloat16,
                      lens_old=np.zeros(2, np.int64), lens_new=lens, extra_pages=1)


def decode(seed: int = 1) -> Workload:
    rng = np.random.Generator(np.random.PCG64(seed + 1000))
    old = rng.integers(512, 4096, size=64, endpoint=True)
    return make_paged("decode", seed, B=64, H=8, D=128, ps=16, layout=HND,
                      dtype=torch.bfloat16, lens_old=old, lens_new=old + 1, slack=0.1)


def _student_t_outliers(H: int, D: int, frac: float = 0.001, factor: float = 20.0):
    def sample(rng, n):
        x = rng.standard_t(3.0, size=(n, H, D)).astype(np.float32)
        n_out = int(round(frac * H * D))
        cols = rng.choice(H * D, size=n_out, replace=False)
        for c in cols:
            x[:, c // D, c % D] *= factor
        return x
    return sample


def prefill(seed: int = 2) -> Workload:
    lens = np.full(8, 8192)
    return make_paged("prefill", seed, B=8, H=8, D=128, ps=32, layout=NHD,
                      dtype=torch.float16, lens_old=np.zeros(8, np.int64), lens_new=lens,
                      recipe=Recipe(256.0, 1, False), sampler=_student_t_outliers(8, 128))


def materialize(seed: int = 3) -> Workload:
    rng = np.random.Generator(np.random.PCG64(seed + 1000))
    lens = np.round(np.exp(rng.uniform(np.log(128), np.log(32768), size=32))).astype(np.int64)
    return make_paged("materialize", seed, B=32, H=8, D=128, ps=64, layout=HND,
                      dtype=torch.bfloat16, lens_old=np.zeros(32, np.int64), lens_new=lens,
                      mat_shared=False, compact_indptr=True, max_kv_len=32768)


LARGE_POOL_BYTES = 40e9


def large_pool(seed: int = 4, device: str = "cuda", B: int = 256, min_len: int = 1024,
               max_len: int = 16384, pool_bytes: float = LARGE_POOL_BYTES) -> Workload:
    """The ~40 GB pool workload. Values are drawn on `device` in chunks with a seeded
    torch generator (N(0,1) * sigma[kv, head]); tables are drawn on the host."""
    H, D, ps = 8, 128, 16
    rng = np.random.Generator(np.random.PCG64(seed))
    lens = rng.integers(min_len, max_len, size=B, endpoint=True).astype(np.int64)
    P = int(pool_bytes // (2 * H * ps * (D // 2 + D // 16)))
    npages = (lens + ps - 1) // ps
    used = int(npages.sum())
    assert used <= P
    placement = rng.choice(P, size=used, replace=False).astype(np.int32)
    indptr = np.zeros(B + 1, np.int32)
    indptr[1:] = np.cumsum(npages)
    last = (lens - (npages - 1) * ps).astype(np.int32)
    max_pages = int(npages.max())
    bt = _dense_table(placement, indptr, max_pages, np.int32, 0)
    mkl = max_len
    mpps = -(-mkl // ps)
    mbt = _dense_table(placement, indptr, max(mpps, max_pages), np.int32, 0)
    bi, pos = _rows_for(np.zeros(B, np.int64), lens)
    sigma = rng.uniform(0.5, 4.0, size=(2, H)).astype(np.float32)
    nnz = len(bi)
    k = values_normal((nnz, H, D), torch.bfloat16, seed, sigma[0], device)
    v = values_normal((nnz, H, D), torch.bfloat16, seed + 7919, sigma[1], device)
    return Workload(
        name="large_pool", B=B, H=H, D=D, ps=ps, layout=HND, dtype=torch.bfloat16,
        recipe=Recipe(256.0, 0, True), num_pages=P, k=k, v=v, batch_indices=bi,
        positions=pos, kv_indices=placement, kv_indptr=indptr, kv_last_page_len=last,
        seq_lens=lens.astype(np.int32), block_tables=bt, max_seq_len=int(lens.max()),
        mat_shared=True, mat_block_tables=mbt, max_kv_len=mkl,
        extra={"sigma": sigma})


def values_normal(shape, dtype, seed, sigma_per_head, device, chunk_rows: int = 1 << 18):
    """N(0,1) * sigma[head] drawn on `device` with torch.Generator(seed), in row chunks."""
    nnz, H, D = shape
    out = torch.empty(shape, dtype=dtype, device=device)
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    sig = torch.as_tensor(sigma_per_head, dtype=torch.float32, device=device).view(1, H, 1)
    for r0 in range(0, nnz, chunk_rows):
        r1 = min(nnz, r0 + chunk_rows)
        x = torch.randn((r1 - r0, H, D), generator=g, device=device, dtype=torch.float32)
        out[r0:r1] = (x * sig).to(dtype)
    return out


NAMED = {"tiny": tiny, "decode": decode, "prefill": prefill, "materialize": materialize}


def random_case(seed: int, *, B: int, H: int, D: int, ps: int, layout: int,
                dtype: torch.dtype, recipe: Optional[Recipe] = None, max_len: int = 100,
                min_len: int = 0, prefill_frac: float = 0.5, bt_dtype=np.int32,
                mat_shared: bool = True, compact_indptr: bool = False,
                scale_range=(0.01, 100.0)) -> Workload:
    """Small ragged case for parity sweeps: random lengths (zero allowed), a random share
    already in the cache, values N(0,1) times a random per-row scale."""
    rng = np.random.Generator(np.random.PCG64(seed + 5000))
    lens_new = rng.integers(min_len, max_len, size=B, endpoint=True)
    lens_old = (lens_new * rng.uniform(0, prefill_frac, size=B)).astype(np.int64)
    lo, hi = np.log(scale_range[0]), np.log(scale_range[1])

    def sampler(r, n):
        x = r.standard_normal((n, H, D), dtype=np.float32)
        return x * np.exp(r.uniform(lo, hi, size=(n, 1, 1))).astype(np.float32)

    return make_paged(f"random{seed}", seed, B=B, H=H, D=D, ps=ps, layout=layout, dtype=dtype,
                      lens_old=lens_old, lens_new=lens_new, recipe=recipe, slack=0.25,
                      sampler=sampler, bt_dtype=bt_dtype, mat_shared=mat_shared,
                      compact_indptr=compact_indptr, extra_pages=1)
