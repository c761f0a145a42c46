"""The large-pool workload at full size (256 requests, 2.29 M tokens, a 40 GB pool), run in
the launch configuration bench.py times (its Step: device-held global scales, append,
dequant, materialize), checked against the CPU oracle: the two global scales over the whole
tensors bit-exactly, and three sampled requests (the first, one drawn at random, the last)
byte by byte -- their cache pages, their dequantized rows and their FP8 pages and table row.
The sampled requests are rebuilt by the oracle from the workload's rows and the oracle's own
global scales. The same run also materializes from V scales rewritten in the
4-token-interleaved layout (the call bench.py makes with --v-scales interleaved4), checked on
the same requests against the oracle's interleaved materialize.
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
    # the interleaved-V materialize of the same cache, into a second copy
    P, H, ps, nb = step.sf[1].shape
    v_il = step.sf[1].view(P, H, ps // 4, 4, nb).transpose(3, 4).contiguous().view(P, H, ps, nb)
    fp8_il = torch.full_like(step.fp8.view(torch.uint8), 0x5A).view(torch.float8_e4m3fn)
    tables_il = torch.full_like(step.tables, -7)
    status_il = torch.zeros_like(step.status)
    step.nv.nvfp4_materialize_fp8(
        step.cache[0], step.cache[1], step.sf[0], v_il, step.mat_bt, step.seq_lens,
        w.max_kv_len, w.mat_shared, fp8_il, step.indptr, w.mat_num_pages, step.lay, tables_il,
        True, status_il, v_block_scales_layout="interleaved4")
    torch.cuda.synchronize()
    del v_il
    r = PL.oracle_recipe(w.recipe)
    gs = tuple(float(O.global_scale(W.bits16(x.cpu()), True, r)) for x in (w.k, w.v))
    return w, step, gs, (fp8_il, tables_il, status_il)


def test_global_scales_and_status(ran):
    w, step, gs, il = ran
    assert int(step.status.item()) == 0
    assert int(il[2].item()) == 0
    for g, want in ((step.gk, gs[0]), (step.gv, gs[1])):
        assert np.float32(g.item()) == np.float32(want)


@pytest.mark.parametrize("which", ["first", "random", "last"])
def test_sampled_request(ran, which):
    w, step, (gs_k, gs_v), (fp8_il, tables_il, _) = ran
    b = {"first": 0, "random": int(np.random.default_rng(5).integers(1, w.B - 1)),
         "last": w.B - 1}[which]
    rows = np.flatnonzero(w.batch_indices == b)
    n = len(rows)
    assert n == int(w.seq_lens[b])
    ps, H, D = w.ps, w.H, w.D
    npg = -(-n // ps)
    r = PL.oracle_recipe(w.recipe)
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
    # the same pages materialized from interleaved V scales
    vil = O.PagedCache(vc.data, O.interleave4_scales(vc.sf.reshape(npg, H, ps, D // 16)).reshape(-1),
                       dps, sps)
    fp8i = np.zeros_like(fp8)
    tabi = np.zeros_like(tab)
    O.materialize_fp8(kc, vil, ps, H, D, w.layout, np.arange(npg, dtype=np.int32)[None], True,
                      np.array([n], np.int32), n, None, fp8i, tabi, v_interleaved4=True)
    assert np.array_equal(tables_il[b].cpu().numpy(), trow)
    goti = fp8_il.view(torch.uint8)[torch.from_numpy(trow[:npg].astype(np.int64)).cuda()].cpu().numpy()
    for j in range(npg):
        valid = min(ps, n - j * ps)
        assert np.array_equal(goti[j][:, :, :valid], fp8i[j + 1][:, :, :valid]), j
    assert not fp8_il.view(torch.uint8)[0].any()


def test_fast_math_choices_on_sampled_rows(ran):
    """The large pool's recipe (4over6 MAE, binary16 error) against the oracle on 65,536 rows
    drawn from the whole workload (8.4 M blocks of K and V): the count of blocks whose scale
    byte or codes differ is reported, and must be zero. The error readings make the kernel
    reproduce the oracle's candidate choice exactly, so the fast-math allowance (up to 1e-4
    of blocks, on near-ties) is not drawn on."""
    w, step, (gs_k, gs_v), _ = ran
    rng = np.random.default_rng(17)
    rows = np.sort(rng.choice(w.nnz, size=65536, replace=False))
    b = w.batch_indices[rows].astype(np.int64)
    pos = w.positions[rows].astype(np.int64)
    page = w.kv_indices[w.kv_indptr[b] + pos // w.ps].astype(np.int64)
    slot = pos % w.ps
    pg, sl = torch.from_numpy(page).cuda(), torch.from_numpy(slot).cuda()
    r = PL.oracle_recipe(w.recipe)
    n, nb = len(rows), w.H * w.D // 16
    differ = 0
    for kv, x, gs in ((0, w.k, gs_k), (1, w.v, gs_v)):
        xs = W.bits16(x[torch.from_numpy(rows).to(x.device)].cpu()).reshape(n, w.H * w.D)
        c, s = O.kv_quantize(xs, True, gs, r)
        if w.layout == W.HND:  # [pages, H, ps, .]: the rows' bytes as [n, H, .]
            gc, gsf = step.cache[kv][pg, :, sl], step.sf[kv][pg, :, sl]
        else:
            gc, gsf = step.cache[kv][pg, sl], step.sf[kv][pg, sl]
        gc = gc.cpu().numpy().reshape(n, nb, 8)
        gsf = gsf.cpu().numpy().reshape(n, nb)
        bad = (gc != c.reshape(n, nb, 8)).any(axis=2) | (gsf != s.reshape(n, nb))
        differ += int(bad.sum())
    print(f"blocks differing from the oracle: {differ} of {2 * n * nb}")
    assert differ == 0
