"""The seeded inputs against the configurations they stand for: sizes, layouts, dtypes,
recipes, length ranges, page placement, value distributions and the consistency of the page
tables. CPU only; the large pool is built with its own recipe at a reduced batch and pool
size (its full pool size is checked by arithmetic)."""
import numpy as np
import pytest
import torch

import workloads as W


@pytest.fixture(scope="module")
def named():
    return {name: make() for name, make in W.NAMED.items()}


def _rows(w):
    """(batch, position) of every row the cache ends up holding: pre-filled, then appended."""
    if w.prefill_k is None:
        return w.batch_indices.astype(np.int64), w.positions.astype(np.int64)
    return (np.concatenate([w.prefill_batch_indices, w.batch_indices]).astype(np.int64),
            np.concatenate([w.prefill_positions, w.positions]).astype(np.int64))


def _check_tables(w):
    lens = w.seq_lens.astype(np.int64)
    assert np.all(lens > 0)
    npages = np.diff(w.kv_indptr.astype(np.int64))
    assert w.kv_indptr[0] == 0 and np.array_equal(npages, (lens + w.ps - 1) // w.ps)
    assert np.array_equal(w.kv_last_page_len, lens - (npages - 1) * w.ps)
    assert np.all((w.kv_last_page_len >= 1) & (w.kv_last_page_len <= w.ps))
    # pages: distinct, inside the pool
    idx = w.kv_indices.astype(np.int64)
    assert len(np.unique(idx)) == len(idx) and idx.min() >= 0 and idx.max() < w.num_pages
    # the dense tables hold each request's pages in order
    for b in range(w.B):
        row = w.kv_indices[w.kv_indptr[b]:w.kv_indptr[b + 1]]
        assert np.array_equal(w.block_tables[b, :npages[b]], row)
    # every position below a request's length is written exactly once, and nothing else
    bi, pos = _rows(w)
    assert len(bi) == lens.sum() == w.nnz + (0 if w.prefill_k is None else len(w.prefill_k))
    assert np.all((pos >= 0) & (pos < lens[bi]))
    key = bi * (1 << 32) + pos
    assert len(np.unique(key)) == len(key)
    # K and V rows have the declared shape and dtype
    assert tuple(w.k.shape) == (w.nnz, w.H, w.D) and w.k.dtype == w.dtype
    assert w.v.shape == w.k.shape and w.v.dtype == w.dtype


def _moments(t):
    x = t.float()
    return float(x.mean()), float(x.std())


@pytest.mark.parametrize("name", sorted(W.NAMED))
def test_tables_are_consistent(named, name):
    _check_tables(named[name])


def test_tiny(named):
    w = named["tiny"]
    assert (w.B, w.H, w.D, w.ps, w.layout, w.dtype) == (2, 2, 64, 16, W.NHD, torch.bfloat16)
    assert list(w.seq_lens) == [37, 64] and w.recipe is None
    assert w.num_pages == 8 and len(w.kv_indices) == 3 + 4  # 7 of 8 permuted pages
    assert w.prefill_k is None and w.nnz == 101  # every token is appended
    m, s = _moments(torch.cat([w.k, w.v]))
    assert abs(m) < 0.05 and abs(s - 1.0) < 0.05  # N(0, 1)


def test_decode(named):
    w = named["decode"]
    assert (w.B, w.H, w.D, w.ps, w.layout, w.dtype) == (64, 8, 128, 16, W.HND, torch.bfloat16)
    assert w.recipe is None
    old = w.seq_lens.astype(np.int64) - 1
    assert old.min() >= 512 and old.max() <= 4096
    # one new token per request, at position old_len
    assert np.array_equal(w.batch_indices, np.arange(64)) and np.array_equal(w.positions, old)
    used = len(w.kv_indices)
    assert w.num_pages == used + int(np.ceil(used * 0.1))  # pool = used pages + 10 %
    m, s = _moments(w.prefill_k[:20000])
    assert abs(m) < 0.02 and abs(s - 1.0) < 0.02


def test_prefill_outlier_channels(named):
    w = named["prefill"]
    assert (w.B, w.H, w.D, w.ps, w.layout, w.dtype) == (8, 8, 128, 32, W.NHD, torch.float16)
    assert list(w.seq_lens) == [8192] * 8 and w.nnz == 65536 and w.prefill_k is None
    assert w.recipe == W.Recipe(256.0, 1, False)  # 4over6 MSE, e4m3_max 256, fp32 error
    n_out = int(round(0.001 * w.H * w.D))
    assert n_out == 1
    for t in (w.k, w.v):
        # Student-t(3): spread about sqrt(3); an outlier channel is 20 times that
        col_spread = t.float().reshape(w.nnz, -1).abs().median(dim=0).values
        big = col_spread > 8 * col_spread.median()
        assert int(big.sum()) == n_out
        ratio = float(col_spread[big].max() / col_spread[~big].median())
        assert 15.0 < ratio < 25.0


def test_materialize(named):
    w = named["materialize"]
    assert (w.B, w.H, w.D, w.ps, w.layout, w.dtype) == (32, 8, 128, 64, W.HND, torch.bfloat16)
    assert w.recipe is None and w.max_kv_len == 32768
    lens = w.seq_lens.astype(np.int64)
    assert lens.min() >= 128 and lens.max() <= 32768
    # log-uniform: the median length sits near the geometric mean of the range
    assert 1024 / 4 < np.median(lens) < 1024 * 4
    npages = (lens + 63) // 64
    assert np.array_equal(w.kv_page_indptr, np.concatenate([[0], np.cumsum(npages)]))
    assert w.mat_num_pages == npages.sum()
    # separate K and V page tables [B, 2, max_kv_len / page_size]
    assert not w.mat_shared and w.mat_block_tables.shape == (32, 2, 32768 // 64)
    kt, vt = w.mat_block_tables[:, 0], w.mat_block_tables[:, 1]
    for b in range(w.B):
        assert np.array_equal(kt[b, :npages[b]], w.kv_indices[w.kv_indptr[b]:w.kv_indptr[b + 1]])
        assert np.all(kt[b, npages[b]:] == -1) and np.all(vt[b, npages[b]:] == -1)
    src, dst = w.v_page_move
    assert np.array_equal(src, w.kv_indices) and len(np.unique(dst)) == len(dst)
    assert not np.array_equal(kt, vt)


def test_large_pool_recipe():
    H, D, ps = 8, 128, 16
    # the full pool: about 40 GB of K + V codes and scales
    assert int(W.LARGE_POOL_BYTES // (2 * H * ps * (D // 2 + D // 16))) == 2_170_138
    w = W.large_pool(device="cpu", B=4, pool_bytes=2e9)
    assert (w.B, w.H, w.D, w.ps, w.layout, w.dtype) == (4, H, D, ps, W.HND, torch.bfloat16)
    assert w.recipe == W.Recipe(256.0, 0, True)  # 4over6 MAE, e4m3_max 256, fp16 error
    assert w.num_pages == int(2e9 // (2 * H * ps * (D // 2 + D // 16)))
    lens = w.seq_lens.astype(np.int64)
    assert lens.min() >= 1024 and lens.max() <= 16384
    _check_tables(w)
    sigma = w.extra["sigma"]
    assert sigma.shape == (2, H) and sigma.min() >= 0.5 and sigma.max() <= 4.0
    for kv, t in enumerate((w.k, w.v)):
        s = t.float().std(dim=(0, 2)).numpy()
        assert np.allclose(s, sigma[kv], rtol=0.02)  # N(0, sigma^2) per (tensor, head)
