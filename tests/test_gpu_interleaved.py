"""FP8 materialize with V block scales in the 4-token-interleaved layout, CUDA vs oracle.

The materialize parameters name that layout for v_block_scales without defining it; both
sides follow one reading (same [pages, H, page_size, D/16] shape; within each head's page
slice, groups of four slots stored block-major and slot-minor). The V scales are rewritten
on the host by the oracle's layout writer, so both sides read the same bytes; every byte of
the FP8 copy and of the page table is compared. Cases cover the bulk-copy kernel and the
plain-load kernel (scale page strides that are not a multiple of 16), head dims 64..256,
page sizes 4..64, shared and separate K/V tables, compact kv_page_indptr, and the
materialize workload at full size with a cache built by the oracle's own append.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from tests import pipelines as PL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda(gpu_lib):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    yield


def _random_caches(w: W.Workload, pad_data: int, pad_sf: int, seed: int):
    rng = np.random.Generator(np.random.PCG64(seed))
    dps, sps = PL.strides(w, pad_data, pad_sf)
    out = []
    for _ in range(2):
        data = rng.integers(0, 256, w.num_pages * dps, dtype=np.uint8)
        sf = rng.integers(0, 256, w.num_pages * sps, dtype=np.uint8)
        sf[(sf & 0x7F) == 0x7F] = 0x7E  # finite scales only
        out.append(O.PagedCache(data, sf, dps, sps))
    return out


def _compare(w: W.Workload, kc, vc, extra_out_pages=0, zero_tables=True, use_class=False):
    import nvfp4_paged_kv_02_gb300 as nv
    r = PL.run_materialize_interleaved(w, kc, vc, extra_out_pages, zero_tables, use_class)
    assert r.status & ~nv.DEV_LEN_CLAMPED == 0
    bad = np.argwhere(r.got != r.want)
    assert bad.size == 0, f"{len(bad)} FP8 bytes differ, first at {bad[0].tolist()}"
    assert np.array_equal(r.got_tables, r.want_tables)
    return r.got


CASES = [
    # seed, B, H, D, ps, max_len, shared, compact, pad_data, pad_sf
    (500, 4, 2, 64, 4, 30, True, False, 0, 0),
    (501, 5, 8, 128, 16, 200, False, True, 0, 0),
    (502, 3, 4, 256, 8, 90, True, True, 16, 0),
    (503, 6, 1, 128, 64, 300, False, False, 0, 0),
    (504, 4, 8, 128, 16, 130, True, False, 0, 2),    # scale stride % 16 != 0: plain loads
    (505, 3, 2, 64, 32, 100, False, True, 32, 6),    # plain loads, separate tables
    (506, 2, 3, 192, 12, 50, True, True, 0, 0),      # ragged: 12-slot pages, D = 192
]


@pytest.mark.parametrize("case", CASES, ids=[str(c[0]) for c in CASES])
def test_interleaved_v_random_bytes(case):
    seed, B, H, D, ps, max_len, shared, compact, pad_d, pad_s = case
    w = W.random_case(seed, B=B, H=H, D=D, ps=ps, layout=W.HND, dtype=torch.bfloat16,
                      max_len=max_len, min_len=0, mat_shared=shared, compact_indptr=compact)
    kc, vc = _random_caches(w, pad_d, pad_s, seed)
    _compare(w, kc, vc)


def test_interleaved_v_run_form_and_workspace():
    w = W.random_case(510, B=5, H=4, D=128, ps=16, layout=W.HND, dtype=torch.bfloat16,
                      max_len=150, min_len=1, mat_shared=False, compact_indptr=True)
    kc, vc = _random_caches(w, 0, 0, 510)
    got = _compare(w, kc, vc, extra_out_pages=3, zero_tables=False, use_class=True)
    assert (got[-3:] == PL.SENT_FP8).all()


def test_interleaved_v_materialize_workload_full_size():
    """The materialize workload (batch 32, lengths log-uniform in [128, 32768], 64-slot
    pages, separate K/V tables, compact kv_page_indptr) at full size: the cache comes from
    the oracle's append of the workload's rows, its V scales rewritten interleaved."""
    w = W.NAMED["materialize"]()
    o = PL.run_oracle(w, do_dequant=False, do_materialize=False)
    dps, sps = PL.strides(w)
    kc = O.PagedCache(o.k_data, o.k_sf, dps, sps)
    vc = O.PagedCache(o.v_data, o.v_sf, dps, sps)
    _compare(w, kc, vc)


def test_interleaved_equals_linear_copy():
    """The same cache through both layouts: the copies agree byte for byte."""
    import nvfp4_paged_kv_02_gb300 as nv
    w = W.random_case(520, B=4, H=8, D=128, ps=16, layout=W.HND, dtype=torch.bfloat16,
                      max_len=120, min_len=1, mat_shared=True)
    kc, vc = _random_caches(w, 0, 0, 520)
    got = _compare(w, kc, vc)
    dev = torch.device("cuda")
    kd, ks = PL.hnd_views(w, kc, dev)
    vd, vs = PL.hnd_views(w, vc, dev)
    out = torch.full(got.shape, PL.SENT_FP8, dtype=torch.uint8,
                     device=dev).view(torch.float8_e4m3fn)
    nv.nvfp4_materialize_fp8(kd, vd, ks, vs, torch.as_tensor(w.mat_block_tables).to(dev),
                             torch.as_tensor(w.seq_lens).to(dev), w.max_kv_len, True, out=out)
    assert np.array_equal(out.view(torch.uint8).cpu().numpy(), got)
