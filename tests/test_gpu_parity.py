"""CUDA library vs CPU oracle, element by element, through the C ABI.

Bit-exact on every byte the operations write (packed codes, scale bytes, dequantized
fp16/bf16, FP8 bytes, page tables) and on every byte they must leave alone (sentinels), for
the named workloads at full size and a sweep of small ragged cases over layouts, dtypes,
page sizes, head dims, table dtypes, recipes, tuple/stacked caches and padded page strides.
Every test runs once with each append kernel (the TMA ring and the direct-load kernel).
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from tests import pipelines as PL

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("append_kernel")]


@pytest.fixture(scope="module", autouse=True)
def _cuda(gpu_lib):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    yield


R_STD = None
R_MAE = W.Recipe(256.0, 0, False)
R_MSE = W.Recipe(256.0, 1, False)
R_MAE16 = W.Recipe(256.0, 0, True)
R_MSE16 = W.Recipe(256.0, 1, True)
R_448 = W.Recipe(448.0, 0, False)


@pytest.mark.parametrize("name", ["tiny", "decode", "prefill", "materialize"])
def test_named_workload(name):
    w = W.NAMED[name]()
    g = PL.run_gpu(w)
    o = PL.run_oracle(w)
    PL.assert_same(g, o, name)


def test_every_kernel_leaves_its_workspace_zero():
    """The ring kernels take work from a counter in the stream's workspace; the last CTA to
    finish sets it back to zero, so the next call starts from zero without a memset. After
    the append, dequant and materialize of a named workload (and the contiguous quantize and
    dequantize),
    every workspace the binding handed out must hold zero."""
    import nvfp4_paged_kv_02_gb300 as nv
    if not nv._dynamic_schedule:
        pytest.skip("fixed shares use no workspace")
    w = W.NAMED["materialize"]()
    g = PL.run_gpu(w)
    o = PL.run_oracle(w)
    PL.assert_same(g, o, "workspace")
    x = torch.randn((4096, 1024), generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    fp4, sf = nv.nvfp4_kv_quantize(x.cuda(), 0.01)
    nv.nvfp4_kv_dequantize(fp4, sf, 0.01)
    torch.cuda.synchronize()
    assert nv._workspaces, "no workspace was used"
    for key, ws in nv._workspaces.items():
        assert int(ws.abs().sum()) == 0, (key, ws.tolist())


CASES = []
for seed, (layout, dt, ps, D, recipe, bt) in enumerate([
    (W.NHD, torch.bfloat16, 16, 128, R_STD, np.int32),
    (W.HND, torch.bfloat16, 16, 128, R_STD, np.int64),
    (W.NHD, torch.float16, 32, 128, R_MSE, np.int32),
    (W.HND, torch.float16, 64, 128, R_MAE, np.int64),
    (W.HND, torch.bfloat16, 16, 128, R_MAE16, np.int32),
    (W.NHD, torch.bfloat16, 4, 64, R_MSE16, np.int32),
    (W.HND, torch.float16, 8, 64, R_MAE16, np.int64),
    (W.NHD, torch.float16, 16, 256, R_MSE16, np.int32),
    (W.HND, torch.bfloat16, 32, 256, R_448, np.int32),
    (W.NHD, torch.bfloat16, 12, 64, R_MAE, np.int32),
    (W.HND, torch.float16, 4, 128, R_STD, np.int32),
    (W.NHD, torch.float16, 64, 64, R_STD, np.int64),
]):
    for H in (1, 3, 8):
        CASES.append(dict(seed=seed * 10 + H, layout=layout, dtype=dt, ps=ps, D=D, recipe=recipe,
                          bt_dtype=bt, H=H))


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"s{c['seed']}-{'NHD' if c['layout'] == 0 else 'HND'}-"
                         f"{str(c['dtype'])[6:]}-ps{c['ps']}-D{c['D']}-H{c['H']}")
def test_random_case(case):
    c = dict(case)
    w = W.random_case(c.pop("seed"), B=7, max_len=150, **c)
    g = PL.run_gpu(w)
    o = PL.run_oracle(w)
    PL.assert_same(g, o, "random")


@pytest.mark.parametrize("D", [16, 32, 48, 80, 96, 192])
@pytest.mark.parametrize("recipe", [R_STD, R_MSE, R_MAE16])
def test_head_dims_without_materialize(D, recipe):
    """Append and dequant take any head_dim % 16 == 0 (the materializer needs % 64)."""
    w = W.random_case(100 + D, B=5, H=3, D=D, ps=8, layout=W.HND if D % 32 else W.NHD,
                      dtype=torch.bfloat16, recipe=recipe, max_len=60)
    g = PL.run_gpu(w, do_materialize=False)
    o = PL.run_oracle(w, do_materialize=False)
    PL.assert_same(g, o, f"D{D}")


@pytest.mark.parametrize("layout", [W.NHD, W.HND])
def test_stacked_and_padded_caches(layout):
    w = W.random_case(200 + layout, B=6, H=4, D=128, ps=16, layout=layout, dtype=torch.float16,
                      recipe=R_MSE16, max_len=90)
    for stacked, pad_d, pad_s in ((True, 0, 0), (False, 256, 16), (True, 64, 32)):
        g = PL.run_gpu(w, stacked=stacked, pad_data=pad_d, pad_sf=pad_s)
        o = PL.run_oracle(w, pad_data=pad_d, pad_sf=pad_s)
        if stacked:
            # the oracle holds K and V apart: compare per cache, page by page
            for name in ("k_data", "k_sf", "v_data", "v_sf"):
                gg, oo = getattr(g, name), getattr(o, name)
                assert np.array_equal(gg, oo), (name, stacked, pad_d)
            for name in ("out_k", "out_v", "fp8", "tables"):
                assert np.array_equal(getattr(g, name), getattr(o, name)), name
            assert g.status == 0
        else:
            PL.assert_same(g, o, f"padded {pad_d}")


def test_dequant_to_other_dtype_and_larger_output():
    """fp16 cache read out as bf16 (and the reverse), into an output longer than every
    request: rows past seq_lens keep the sentinel."""
    w = W.random_case(300, B=5, H=2, D=64, ps=16, layout=W.NHD, dtype=torch.float16, max_len=40)
    w.max_seq_len = 57
    for odt in (torch.bfloat16, torch.float16):
        g = PL.run_gpu(w, out_dtype=odt, do_materialize=False)
        o = PL.run_oracle(w, out_dtype=odt, do_materialize=False)
        PL.assert_same(g, o, str(odt))


def test_materialize_run_form_and_workspace():
    """Without zeroing the table (run() form) only active entries change; a larger
    workspace keeps pages past the end untouched."""
    w = W.random_case(400, B=6, H=2, D=128, ps=8, layout=W.HND, dtype=torch.bfloat16,
                      max_len=70, mat_shared=False, compact_indptr=True)
    g = PL.run_gpu(w, extra_out_pages=3, zero_tables=False, do_dequant=False)
    o = PL.run_oracle(w, extra_out_pages=3, zero_tables=False, do_dequant=False)
    PL.assert_same(g, o, "run form")
    assert (g.tables == PL.SENT_TABLE).any()
    assert (g.fp8[-3:] == PL.SENT_FP8).all()


@pytest.mark.parametrize("shared", [True, False])
def test_materializer_class_matches_oracle(shared):
    """NVFP4KVMaterializer.run() (the prepared C form) against the oracle's materialize with
    run() semantics (only active table entries written), on caches the oracle appended; then
    the same run captured in a CUDA graph and replayed after new lengths are copied into the
    captured tensor, against the oracle on those lengths."""
    import nvfp4_paged_kv_02_gb300 as nv
    w = W.random_case(401 + int(shared), B=4, H=8, D=128, ps=16, layout=W.HND,
                      dtype=torch.bfloat16, max_len=100, compact_indptr=True, mat_shared=shared)
    dev = torch.device("cuda")
    o = PL.run_oracle(w, do_dequant=False, extra_out_pages=2, zero_tables=False)
    dps, sps = PL.strides(w)
    kc = O.PagedCache(o.k_data, o.k_sf, dps, sps)
    vc = O.PagedCache(o.v_data, o.v_sf, dps, sps)
    kd, ks = PL.hnd_views(w, kc, dev)
    vd, vs = PL.hnd_views(w, vc, dev)
    t = lambda a: torch.as_tensor(np.ascontiguousarray(a)).to(dev)
    m = nv.NVFP4KVMaterializer(w.H, w.ps, w.D, dev, uses_shared_paged_kv_idx=shared)
    n_out, mpps = PL.mat_shape(w)
    out = torch.full((n_out + 2, 2, w.H, w.ps, w.D), PL.SENT_FP8, dtype=torch.uint8,
                     device=dev).view(torch.float8_e4m3fn)
    tbl = torch.full((w.B, mpps), PL.SENT_TABLE, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    bt, sl, ip = t(w.mat_block_tables), t(w.seq_lens), t(w.kv_page_indptr)
    m.run(kd, vd, ks, vs, bt, sl, ip, out=out, fp8_block_tables=tbl, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(out.view(torch.uint8).cpu().numpy(), o.fp8)
    assert np.array_equal(tbl.cpu().numpy(), o.tables)
    # graph capture of run(): replay after shorter lengths are copied into the captured
    # tensor (same page reservations), compared with the oracle on those lengths
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        m.run(kd, vd, ks, vs, bt, sl, ip, out=out, fp8_block_tables=tbl)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        m.run(kd, vd, ks, vs, bt, sl, ip, out=out, fp8_block_tables=tbl)
    shorter = np.maximum(w.seq_lens - 17, 1).astype(np.int32)
    sl.copy_(torch.from_numpy(shorter))
    out.view(torch.uint8).fill_(PL.SENT_FP8)
    tbl.fill_(PL.SENT_TABLE)
    graph.replay()
    torch.cuda.synchronize()
    want = np.full_like(o.fp8, PL.SENT_FP8)
    want_tbl = np.full_like(o.tables, PL.SENT_TABLE)
    O.materialize_fp8(kc, vc, w.ps, w.H, w.D, W.HND, w.mat_block_tables, shared, shorter,
                      w.max_kv_len, w.kv_page_indptr, want, want_tbl, False, 0)
    assert np.array_equal(out.view(torch.uint8).cpu().numpy(), want)
    assert np.array_equal(tbl.cpu().numpy(), want_tbl)


def test_codec_edge_values():
    """Blocks built so that x * (1/(S*gs)) hits E2M1 midpoints, saturation, signed zeros
    and subnormal E4M3 scales exactly; checked against the oracle through the C ABI."""
    vals = [6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.1, -0.0, 5.5, -2.25, 0.0, -6.0,
            4.5, 0.5]
    # a row with amax 2688 makes the standard global scale exactly 1, so the probe row's
    # block scale is 1 and its values are the E2M1 inputs themselves
    rows = [np.array([2688.0] + [0.0] * 15, np.float32), np.array(vals, np.float32)]
    rng = np.random.Generator(np.random.PCG64(7))
    for e in range(-16, 4):  # amax sweeping block scales down into E4M3 subnormals
        x = rng.standard_normal(16).astype(np.float32)
        x = x / np.abs(x).max() * np.float32(6.0 * 2.0 ** e)
        rows.append(x)
    x = np.stack(rows)  # [n, 16]
    n = x.shape[0]
    for dt in (torch.bfloat16, torch.float16):
        for recipe in (R_STD, R_MSE, R_MAE16):
            t = torch.from_numpy(x).to(dt).view(n, 1, 16)
            w = W.make_paged("edge", 0, B=1, H=1, D=16, ps=n, layout=W.NHD, dtype=dt,
                             lens_old=np.array([0]), lens_new=np.array([n]), recipe=recipe)
            w.k, w.v = t, -t
            g = PL.run_gpu(w, do_materialize=False)
            o = PL.run_oracle(w, do_materialize=False)
            PL.assert_same(g, o, f"edge {dt} {recipe}")


def test_empty_and_zero_length_requests():
    lens = np.array([0, 5, 0, 17, 0])
    w = W.make_paged("zeros", 3, B=5, H=2, D=64, ps=4, layout=W.HND, dtype=torch.bfloat16,
                     lens_old=lens, lens_new=lens, extra_pages=2)  # nothing new to append
    assert w.nnz == 0
    g = PL.run_gpu(w)
    o = PL.run_oracle(w)
    PL.assert_same(g, o, "zeros")
    w0 = W.make_paged("allzero", 4, B=3, H=2, D=64, ps=4, layout=W.NHD, dtype=torch.bfloat16,
                      lens_old=np.zeros(3), lens_new=np.zeros(3), extra_pages=2)
    g = PL.run_gpu(w0)
    o = PL.run_oracle(w0)
    PL.assert_same(g, o, "allzero")


def test_device_bounds_flags():
    """Bad device-held indices are skipped and reported, never written out of bounds."""
    import nvfp4_paged_kv_02_gb300 as nv
    dev = torch.device("cuda")
    ps, H, D, P = 4, 2, 64, 6
    kd = torch.full((P, ps, H, D // 2), 0xA5, dtype=torch.uint8, device=dev)
    ks = torch.full((P, ps, H, D // 16), 0xA5, dtype=torch.uint8, device=dev)
    vd, vs = kd.clone(), ks.clone()
    x = torch.randn(4, H, D, device=dev, dtype=torch.bfloat16)
    i32 = lambda a: torch.tensor(a, dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    # row 0 fine; row 1 bad batch; row 2 position past the described space; row 3 bad page
    nv.nvfp4_quantize_append_paged(
        x, x, i32([0, 5, 0, 1]), i32([1, 0, 9, 2]), (kd, vd), (ks, vs), i32([2, 3, 99]),
        i32([0, 2, 3]), i32([4, 3]), 0.01, 0.01, "NHD", None, st)
    torch.cuda.synchronize()
    assert int(st.item()) == nv.DEV_BAD_BATCH | nv.DEV_BAD_POSITION | nv.DEV_BAD_PAGE
    changed = (kd != 0xA5).any(dim=(1, 2, 3)).cpu().numpy()
    assert changed.tolist() == [False, False, True, False, False, False]
    # dequant: a length beyond the output is clamped and reported; a bad page is skipped
    st.zero_()
    ok = torch.zeros((2, 8, H, D), dtype=torch.bfloat16, device=dev)
    ov = ok.clone()
    g = torch.ones(1, device=dev)
    nv.nvfp4_dequantize_paged((kd, vd), (ks, vs), i32([[2, 3], [-1, 4]]), i32([12, 3]), g, g,
                              ok, ov, "NHD", st)
    torch.cuda.synchronize()
    assert int(st.item()) == nv.DEV_LEN_CLAMPED | nv.DEV_BAD_PAGE
    assert (ok[1] == 0).all()
    # materialize: an output page outside the workspace is skipped and reported
    st.zero_()
    out = torch.zeros((3, 2, H, ps, D), dtype=torch.uint8, device=dev).view(torch.float8_e4m3fn)
    tbl = torch.zeros((2, 2), dtype=torch.int32, device=dev)
    nv.nvfp4_materialize_fp8(kd, vd, ks, vs, i32([[2, 3], [1, 4]]), i32([8, 3]), 8, True, out,
                             i32([0, 2, 7]), 2, "NHD", tbl, True, st)
    torch.cuda.synchronize()
    assert int(st.item()) == nv.DEV_BAD_OUT_PAGE


@pytest.mark.parametrize("numel", [0, 1, 15, 16, 17, 1000, 4096 * 7 + 5, 1 << 16, (1 << 16) + 1,
                                   (1 << 16) + 31, 3 << 20, 1 << 23, (1 << 23) + 3 * 8192 + 17])
@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float16])
def test_global_scale(numel, dt):
    import nvfp4_paged_kv_02_gb300 as nv
    g = torch.Generator().manual_seed(numel)
    x = (torch.randn(numel, generator=g) * 3).to(dt)
    for recipe, orecipe in ((None, None), (nv.NVFP44Over6Config(256.0, "MSE"), O.Recipe(256.0, 1))):
        got = nv.nvfp4_make_global_scale(x.cuda(), recipe).item()
        want = O.global_scale(W.bits16(x), dt == torch.bfloat16, orecipe)
        assert np.float32(got).view(np.uint32) == np.float32(want).view(np.uint32), (got, want)


@pytest.mark.parametrize("numel", [1000, 1 << 16, (1 << 16) + 17, 1 << 20, (1 << 23) + 5])
@pytest.mark.parametrize("where", [0, -1, "mid"])
def test_global_scale_max_at_edges(numel, where):
    """The tensor's largest magnitude (negative) at the first, last or a middle element, for
    sizes scanned by one CTA and by many."""
    import nvfp4_paged_kv_02_gb300 as nv
    x = (torch.randn(numel, generator=torch.Generator().manual_seed(numel)) * 0.5)
    i = numel // 2 + 3 if where == "mid" else where
    x[i] = -1000.0
    x = x.to(torch.bfloat16)
    got = nv.nvfp4_make_global_scale(x.cuda()).item()
    want = O.global_scale(W.bits16(x), True, None)
    assert np.float32(got).view(np.uint32) == np.float32(want).view(np.uint32), (got, want)


def test_append_with_device_scales():
    """The device-scale append writes exactly what the host-scale append writes; a device
    scale that is not positive finite is reported and nothing is written."""
    import nvfp4_paged_kv_02_gb300 as nv
    dev = torch.device("cuda")
    w = W.random_case(500, B=4, H=4, D=128, ps=16, layout=W.HND, dtype=torch.bfloat16,
                      recipe=R_MAE16, max_len=80)
    t = lambda a: torch.as_tensor(np.ascontiguousarray(a)).to(dev)
    r = PL.gpu_recipe(w.recipe)
    outs = []
    for use_dev in (False, True):
        kd = torch.full((w.num_pages, w.H, w.ps, w.D // 2), 0xA5, dtype=torch.uint8, device=dev)
        ks = torch.full((w.num_pages, w.H, w.ps, w.D // 16), 0xA5, dtype=torch.uint8, device=dev)
        vd, vs = kd.clone(), ks.clone()
        gk = nv.nvfp4_make_global_scale(w.k.to(dev), r)
        gv = nv.nvfp4_make_global_scale(w.v.to(dev), r)
        sk, sv = (gk, gv) if use_dev else (gk.item(), gv.item())
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        nv.nvfp4_quantize_append_paged(w.k.to(dev), w.v.to(dev), t(w.batch_indices),
                                       t(w.positions), (kd, vd), (ks, vs), t(w.kv_indices),
                                       t(w.kv_indptr), t(w.kv_last_page_len), sk, sv, "HND", r, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        outs.append([x.cpu().numpy() for x in (kd, ks, vd, vs)])
    for a, b in zip(*outs):
        assert np.array_equal(a, b)
    for bad in (0.0, -1.0, float("inf"), float("nan")):
        kd = torch.full((w.num_pages, w.H, w.ps, w.D // 2), 0xA5, dtype=torch.uint8, device=dev)
        ks = torch.full((w.num_pages, w.H, w.ps, w.D // 16), 0xA5, dtype=torch.uint8, device=dev)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        g_bad = torch.tensor([bad], dtype=torch.float32, device=dev)
        g_ok = torch.tensor([0.01], dtype=torch.float32, device=dev)
        nv.nvfp4_quantize_append_paged(w.k.to(dev), w.v.to(dev), t(w.batch_indices),
                                       t(w.positions), (kd, kd.clone()), (ks, ks.clone()),
                                       t(w.kv_indices), t(w.kv_indptr), None, g_ok, g_bad, "HND",
                                       r, st)
        torch.cuda.synchronize()
        assert int(st.item()) == nv.DEV_BAD_SCALE
        assert (kd == 0xA5).all() and (ks == 0xA5).all()


@pytest.mark.parametrize("what", ["wide_rows", "sf_stride_not_16", "big_pages"])
def test_direct_load_kernels(what):
    """Shapes the shared-memory ring cannot take run the direct-load kernels: an append row
    of more than 24 KB per tensor (16 heads x 1024), scale pages whose stride is not a
    multiple of 16 bytes (no bulk copy), and pages larger than a 48 KB stage (128 slots x 8
    heads x 128)."""
    if what == "wide_rows":
        w = W.random_case(700, B=3, H=16, D=1024, ps=4, layout=W.NHD, dtype=torch.bfloat16,
                          recipe=R_MAE16, max_len=9)
        kw = {}
    elif what == "sf_stride_not_16":
        w = W.random_case(701, B=5, H=4, D=128, ps=16, layout=W.HND, dtype=torch.float16,
                          recipe=R_MSE, max_len=70)
        kw = dict(pad_data=16, pad_sf=8)
    else:
        w = W.random_case(702, B=3, H=8, D=128, ps=128, layout=W.HND, dtype=torch.bfloat16,
                          recipe=R_STD, max_len=300)
        kw = {}
    g = PL.run_gpu(w, **kw)
    o = PL.run_oracle(w, **kw)
    PL.assert_same(g, o, what)


def test_largest_batch():
    """16384 requests (the largest batch a CTA's shared-memory scan takes), lengths 0..5."""
    lens = np.arange(16384) % 6
    w = W.make_paged("maxbatch", 9, B=16384, H=1, D=64, ps=4, layout=W.HND,
                     dtype=torch.bfloat16, lens_old=np.zeros(16384, np.int64), lens_new=lens,
                     extra_pages=3)
    g = PL.run_gpu(w)
    o = PL.run_oracle(w)
    PL.assert_same(g, o, "max batch")


@pytest.mark.parametrize("recipe", [R_STD, R_MAE16, R_MSE])
def test_append_order_split_and_repeat(recipe):
    """Rows appended in any order, split over several calls, or appended twice, leave the
    same bytes in the cache as one in-order call; the result is also the oracle's."""
    import nvfp4_paged_kv_02_gb300 as nv
    dev = torch.device("cuda")
    w = W.random_case(800, B=6, H=4, D=128, ps=16, layout=W.HND, dtype=torch.bfloat16,
                      recipe=recipe, max_len=120, min_len=10, prefill_frac=0.0)
    r = PL.gpu_recipe(recipe)
    t = lambda a: torch.as_tensor(np.ascontiguousarray(a)).to(dev)
    gk = float(nv.nvfp4_make_global_scale(w.k.to(dev).contiguous(), r).item())
    gv = float(nv.nvfp4_make_global_scale(w.v.to(dev).contiguous(), r).item())
    shape = (w.num_pages, w.H, w.ps)

    def fresh():
        return ((torch.full((*shape, w.D // 2), 0xA5, dtype=torch.uint8, device=dev),
                 torch.full((*shape, w.D // 2), 0xA5, dtype=torch.uint8, device=dev)),
                (torch.full((*shape, w.D // 16), 0xA5, dtype=torch.uint8, device=dev),
                 torch.full((*shape, w.D // 16), 0xA5, dtype=torch.uint8, device=dev)))

    def append(cache, rows):
        rows = np.asarray(rows, np.int64)
        idx = torch.from_numpy(rows)
        nv.nvfp4_quantize_append_paged(
            w.k[idx].to(dev), w.v[idx].to(dev), t(w.batch_indices[rows]), t(w.positions[rows]),
            cache[0], cache[1], t(w.kv_indices), t(w.kv_indptr), t(w.kv_last_page_len), gk, gv,
            "HND", r)

    def host(cache):
        return [x.cpu().numpy() for pair in cache for x in pair]

    order = np.arange(w.nnz)
    base = fresh()
    append(base, order)
    want = host(base)
    perm = np.random.default_rng(8).permutation(w.nnz)
    for rows_list in ([perm], [order[: w.nnz // 3], order[w.nnz // 3:]],
                      [perm[::2], perm[1::2]], [order, order]):
        c = fresh()
        for rows in rows_list:
            append(c, rows)
        for a, b in zip(host(c), want):
            assert np.array_equal(a, b)
    o = PL.run_oracle(w, do_dequant=False, do_materialize=False)
    assert np.array_equal(want[0].reshape(-1), o.k_data) and np.array_equal(want[1].reshape(-1), o.v_data)
    assert np.array_equal(want[2].reshape(-1), o.k_sf) and np.array_equal(want[3].reshape(-1), o.v_sf)


@pytest.mark.parametrize("gk,gv", [(1e-40, 0.01), (0.02, 3e-39), (1e37, 1e38), (2.5e38, 1e-30),
                                   (7e-39, 7e-39)])
@pytest.mark.parametrize("recipe", [R_STD, R_MSE, R_MAE16])
def test_extreme_global_scales(gk, gv, recipe):
    """Global scales whose 6*gs or 4*gs (or their reciprocals) are subnormal or overflow take
    the general division path; the result still matches the oracle (paged append and the
    contiguous quantize)."""
    import nvfp4_paged_kv_02_gb300 as nv
    dev = torch.device("cuda")
    gk, gv = float(np.float32(gk)), float(np.float32(gv))
    w = W.random_case(900, B=3, H=2, D=64, ps=8, layout=W.NHD, dtype=torch.bfloat16,
                      recipe=recipe, max_len=40, min_len=5, prefill_frac=0.0,
                      scale_range=(1e-3, 1e3))
    t = lambda a: torch.as_tensor(np.ascontiguousarray(a)).to(dev)
    shape = (w.num_pages, w.ps, w.H)
    kc = [torch.full((*shape, w.D // 2), 0xA5, dtype=torch.uint8, device=dev) for _ in range(2)]
    ks = [torch.full((*shape, w.D // 16), 0xA5, dtype=torch.uint8, device=dev) for _ in range(2)]
    nv.nvfp4_quantize_append_paged(w.k.to(dev), w.v.to(dev), t(w.batch_indices), t(w.positions),
                                   tuple(kc), tuple(ks), t(w.kv_indices), t(w.kv_indptr),
                                   t(w.kv_last_page_len), gk, gv, "NHD", PL.gpu_recipe(recipe))
    dps, sps = PL.strides(w)
    oc = [O.PagedCache(np.full(w.num_pages * dps, 0xA5, np.uint8),
                       np.full(w.num_pages * sps, 0xA5, np.uint8), dps, sps) for _ in range(2)]
    HD = w.H * w.D
    O.quantize_append_paged(W.bits16(w.k), W.bits16(w.v), True, w.nnz, w.H, w.D, HD, HD,
                            w.batch_indices, w.positions, oc[0], oc[1], w.ps, W.NHD,
                            w.kv_indices, w.kv_indptr, gk, gv, PL.oracle_recipe(recipe))
    for i in range(2):
        assert np.array_equal(kc[i].cpu().numpy().reshape(-1), oc[i].data), i
        assert np.array_equal(ks[i].cpu().numpy().reshape(-1), oc[i].sf), i
    # contiguous form with the K scale
    x = w.k.reshape(w.nnz, HD)
    fp4, sf = nv.nvfp4_kv_quantize(x.to(dev), gk, PL.gpu_recipe(recipe))
    c, s_ = O.kv_quantize(W.bits16(x), True, gk, PL.oracle_recipe(recipe))
    assert np.array_equal(fp4.cpu().numpy(), c) and np.array_equal(sf.cpu().numpy(), s_)
