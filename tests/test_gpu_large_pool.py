"""The large-pool workload at full size (256 requests, 2.29 M tokens, a 40 GB pool), run in
the launch configuration bench.py times (its Step: device-held global scales, append,
dequant, materialize), checked against the CPU oracle: the two global scales over the whole
tensors bit-exactly, and three sampled requests (the first, one drawn at random, the last)
byte by byte -- their cache pages, their dequantized rows and their FP8 pages and table row.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from tests import pipelines as PL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ran(gpu_lib):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import bench
    dev = torch.device("cuda")
    w = W.large_pool(device="cuda")
    step = bench.Step(w, dev)
    step.run()
    torch.cuda.synchronize()
    return w, step


def test_global_scales_and_status(ran):
    w, step = ran
    assert int(step.status.item()) == 0
    r = PL.oracle_recipe(w.recipe)
    for x, g in ((w.k, step.gk), (w.v, step.gv)):
        want = O.global_scale(W.bits16(x.cpu()), True, r)
        assert np.float32(g.item()) == np.float32(want)


@pytest.mark.parametrize("which", ["first", "random", "last"])
def test_sampled_request(ran, which):
    w, step = ran
    b = {"first": 0, "random": int(np.random.default_rng(5).integers(1, w.B - 1)),
         "last": w.B - 1}[which]
    rows = np.flatnonzero(w.batch_indices == b)
    n = len(rows)
    assert n == int(w.seq_lens[b])
    ps, H, D = w.ps, w.H, w.D
    npg = -(-n // ps)
    r = PL.oracle_recipe(w.recipe)
    gs_k, gs_v = float(step.gk.item()), float(step.gv.item())
    idx = torch.from_numpy(rows).to(w.k.device)
    kb, vb = W.bits16(w.k[idx].cpu()), W.bits16(w.v[idx].cpu())
    # the request alone, in a compact cache of its own pages (HND pages of [H, ps, .])
    dps, sps = ps * H * D // 2, ps * H * D // 16
    kc = O.PagedCache(np.zeros(npg * dps, np.uint8), np.zeros(npg * sps, np.uint8), dps, sps)
    vc = O.PagedCache(np.zeros(npg * dps, np.uint8), np.zeros(npg * sps, np.uint8), dps, sps)
    O.quantize_append_paged(kb, vb, True, n, H, D, H * D, H * D, np.zeros(n, np.int32),
                            w.positions[rows].astype(np.int32), kc, vc, ps, w.layout,
                            np.arange(npg, dtype=np.int32), np.array([0, npg], np.int32),
                            gs_k, gs_v, r)
    pages = w.kv_indices[w.kv_indptr[b]:w.kv_indptr[b + 1]]
    for kv, oc in ((0, kc), (1, vc)):
        gd = step.cache[kv][torch.from_numpy(pages.astype(np.int64)).cuda()].cpu().numpy()
        gsf = step.sf[kv][torch.from_numpy(pages.astype(np.int64)).cuda()].cpu().numpy()
        od = oc.data.reshape(npg, H, ps, D // 2)
        osf = oc.sf.reshape(npg, H, ps, D // 16)
        for j in range(npg):
            valid = min(ps, n - j * ps)
            assert np.array_equal(gd[j][:, :valid], od[j][:, :valid]), (kv, j)
            assert np.array_equal(gsf[j][:, :valid], osf[j][:, :valid]), (kv, j)
    # dequant of the request
    ok = np.zeros((1, n, H, D), np.uint16)
    ov = np.zeros_like(ok)
    O.dequantize_paged(kc, vc, ps, H, D, w.layout, np.arange(npg, dtype=np.int32)[None],
                       np.array([n], np.int32), gs_k, gs_v, ok, ov, True)
    assert np.array_equal(W.bits16(step.out_k[b, :n].cpu()), ok[0])
    assert np.array_equal(W.bits16(step.out_v[b, :n].cpu()), ov[0])
    # FP8 pages of the request: page j lands at b * mpps + j + 1; the table row says so
    mpps = step.tables.shape[1]
    fp8 = np.zeros((npg + 1, 2, H, ps, D), np.uint8)
    tab = np.zeros((1, -(-n // ps)), np.int32)
    O.materialize_fp8(kc, vc, ps, H, D, w.layout, np.arange(npg, dtype=np.int32)[None], True,
                      np.array([n], np.int32), n, None, fp8, tab)
    trow = step.tables[b].cpu().numpy()
    assert np.array_equal(trow[:npg], b * mpps + np.arange(npg) + 1)
    assert np.all(trow[npg:] == 0)
    got = step.fp8.view(torch.uint8)[torch.from_numpy(trow[:npg].astype(np.int64)).cuda()].cpu().numpy()
    for j in range(npg):
        valid = min(ps, n - j * ps)
        assert np.array_equal(got[j][:, :, :valid], fp8[j + 1][:, :, :valid]), j
    assert not step.fp8.view(torch.uint8)[0].any()
