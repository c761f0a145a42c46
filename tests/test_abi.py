"""The C-ABI library without a GPU: it builds for sm_103a, loads, exports every function
include/nvfp4kv.h declares, and its host-side validation rejects bad arguments before any
device work (those paths return before the first CUDA call, so they run on CPU)."""
import ctypes
import math
import os
import re
import subprocess

import pytest

import nvfp4_paged_kv_02_gb300 as nv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nvfp4kv.h")


def declared_functions():
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w]+\**\s+\**(nvfp4_\w+)\s*\(", text, re.M)))


@pytest.fixture(scope="module")
def lib():
    return nv.load()


def test_header_declares_the_operations():
    fns = declared_functions()
    for f in ("nvfp4_quantize_append_paged", "nvfp4_dequantize_paged", "nvfp4_materialize_fp8",
              "nvfp4_make_global_scale", "nvfp4_e4m3_max", "nvfp4_last_error_string"):
        assert f in fns, fns


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", nv.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r" T (\w+)$", out, re.M))
    for f in declared_functions():
        assert f in exported, f
        assert hasattr(lib, f)
    # nothing but the C ABI is exported from the library's own code
    assert {e for e in exported if e.startswith("nvfp4")} == set(declared_functions())


def test_abi_version_and_e4m3_max(lib):
    assert lib.nvfp4_abi_version() == 5
    assert nv.nvfp4_e4m3_max(None) == 448.0
    assert nv.nvfp4_e4m3_max(nv.NVFP44Over6Config(256.0, "MSE")) == 256.0


def test_out_pages_helper(lib):
    assert nv.nvfp4_materialize_fp8_out_pages(32, 32768, 64) == (32 * 512 + 1, 512)
    assert nv.nvfp4_materialize_fp8_out_pages(2, 64, 16) == (9, 4)
    assert nv.nvfp4_materialize_fp8_out_pages(3, 100, 16, num_pages=11) == (12, 7)


FAKE = 1 << 20  # a well-aligned non-null address; never dereferenced on these paths


def cache(ps=16, H=8, D=128, pages=4, data=FAKE, dstride=None, sstride=None):
    return nv._Cache(data, FAKE, dstride if dstride is not None else ps * H * D // 2,
                     sstride if sstride is not None else ps * H * D // 16, pages)


def append(lib, **kw):
    a = dict(k=FAKE, v=FAKE, dtype=1, nnz=4, H=8, D=128, ks=1024, vs=1024, kc=cache(), vc=cache(),
             ps=16, layout=0, B=2, k_scale=0.5, v_scale=0.5, recipe=None, ws=None)
    a.update(kw)
    return lib.nvfp4_quantize_append_paged(
        ctypes.c_void_p(a["k"]), ctypes.c_void_p(a["v"]), a["dtype"], a["nnz"], a["H"], a["D"],
        a["ks"], a["vs"], ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE), a["kc"], a["vc"],
        a["ps"], a["layout"], ctypes.c_void_p(FAKE), 16, ctypes.c_void_p(FAKE), None, a["B"],
        a["k_scale"], a["v_scale"], a["recipe"], None,
        None if a["ws"] is None else ctypes.c_void_p(a["ws"]), None)


def err(lib):
    return lib.nvfp4_last_error_string().decode()


@pytest.mark.parametrize("kw,code,text", [
    (dict(D=24), nv.ERR_INVALID_ARG, "head_dim"),
    (dict(D=0), nv.ERR_INVALID_ARG, "head_dim"),
    (dict(H=0), nv.ERR_INVALID_ARG, "num_kv_heads"),
    (dict(ps=0), nv.ERR_INVALID_ARG, "page_size"),
    (dict(layout=2), nv.ERR_INVALID_ARG, "kv_layout"),
    (dict(dtype=7), nv.ERR_INVALID_ARG, "dtype"),
    (dict(nnz=-1), nv.ERR_INVALID_ARG, "nnz"),
    (dict(k_scale=0.0), nv.ERR_INVALID_ARG, "positive finite"),
    (dict(v_scale=-1.0), nv.ERR_INVALID_ARG, "positive finite"),
    (dict(k_scale=math.inf), nv.ERR_INVALID_ARG, "positive finite"),
    (dict(v_scale=math.nan), nv.ERR_INVALID_ARG, "positive finite"),
    (dict(k=FAKE + 8), nv.ERR_ALIGNMENT, "aligned"),
    (dict(ks=1028), nv.ERR_ALIGNMENT, "aligned"),
    (dict(ks=512), nv.ERR_INVALID_ARG, "row strides"),
    (dict(kc=cache(data=FAKE + 4)), nv.ERR_ALIGNMENT, "16-byte"),
    (dict(kc=cache(dstride=1000)), nv.ERR_INVALID_ARG, "data_page_stride"),
    (dict(vc=cache(sstride=10)), nv.ERR_INVALID_ARG, "sf_page_stride"),
    (dict(B=0), nv.ERR_INVALID_ARG, "batch_size"),
])
def test_append_rejects(lib, kw, code, text):
    assert append(lib, **kw) == code
    assert text in err(lib)


@pytest.mark.parametrize("cfg,text", [
    ((0.0, 0, 0), "e4m3_max"), ((500.0, 0, 0), "e4m3_max"), ((math.nan, 0, 0), "e4m3_max"),
    ((256.0, 2, 0), "err_mode"), ((256.0, 0, 3), "err_use_fast_math"),
])
def test_recipe_rejects(lib, cfg, text):
    r = ctypes.pointer(nv._Config(*cfg))
    assert append(lib, recipe=r) == nv.ERR_INVALID_ARG
    assert text in err(lib)


def test_empty_append_is_a_no_op(lib):
    assert append(lib, nnz=0) == nv.OK
    assert err(lib) == ""


def dequant(lib, **kw):
    a = dict(kc=cache(), vc=cache(), ps=16, H=8, D=128, layout=1, tdt=0, maxp=4, B=2, out=FAKE,
             odt=1, L=64, ws=None)
    a.update(kw)
    return lib.nvfp4_dequantize_paged(
        a["kc"], a["vc"], a["ps"], a["H"], a["D"], a["layout"], ctypes.c_void_p(FAKE), a["tdt"],
        a["maxp"], ctypes.c_void_p(FAKE), a["B"], ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE),
        ctypes.c_void_p(a["out"]), ctypes.c_void_p(FAKE), a["odt"], a["L"], None,
        None if a["ws"] is None else ctypes.c_void_p(a["ws"]), None)


@pytest.mark.parametrize("kw,code,text", [
    (dict(tdt=3), nv.ERR_INVALID_ARG, "table_dtype"),
    (dict(odt=5), nv.ERR_INVALID_ARG, "out_dtype"),
    (dict(out=FAKE + 2), nv.ERR_ALIGNMENT, "aligned"),
    (dict(B=20000), nv.ERR_UNSUPPORTED, "batch_size"),
    (dict(D=40), nv.ERR_INVALID_ARG, "head_dim"),
])
def test_dequant_rejects(lib, kw, code, text):
    assert dequant(lib, **kw) == code
    assert text in err(lib)


def test_empty_dequant_is_a_no_op(lib):
    assert dequant(lib, B=0) == nv.OK
    assert dequant(lib, L=0) == nv.OK


def materialize(lib, **kw):
    a = dict(kc=cache(), vc=cache(), ps=16, H=8, D=128, layout=1, mnp=4, shared=1, B=2, mkl=64,
             indptr=None, npages=-1, out=FAKE, nout=9, vsf=nv.SF_LINEAR, ws=None)
    a.update(kw)
    return lib.nvfp4_materialize_fp8(
        a["kc"], a["vc"], a["ps"], a["H"], a["D"], a["layout"], ctypes.c_void_p(FAKE), a["mnp"],
        a["shared"], ctypes.c_void_p(FAKE), a["B"], a["mkl"],
        None if a["indptr"] is None else ctypes.c_void_p(a["indptr"]), a["npages"],
        ctypes.c_void_p(a["out"]), a["nout"], ctypes.c_void_p(FAKE), 1, a["vsf"], None,
        None if a["ws"] is None else ctypes.c_void_p(a["ws"]), None)


@pytest.mark.parametrize("kw,code,text", [
    (dict(D=96, kc=cache(D=96), vc=cache(D=96)), nv.ERR_INVALID_ARG, "divisible by 64"),
    (dict(ps=6, kc=cache(ps=6), vc=cache(ps=6)), nv.ERR_INVALID_ARG, "divisible by 4"),
    (dict(mnp=3), nv.ERR_INVALID_ARG, "columns"),
    (dict(nout=8), nv.ERR_INVALID_ARG, "num_pages + 1"),
    (dict(indptr=FAKE), nv.ERR_INVALID_ARG, "requires num_pages"),
    (dict(indptr=FAKE, npages=20, nout=20), nv.ERR_INVALID_ARG, "num_pages + 1"),
    (dict(out=FAKE + 16), nv.ERR_ALIGNMENT, "32-byte"),
    (dict(vsf=2), nv.ERR_INVALID_ARG, "v_scale_layout"),
    (dict(vsf=nv.SF_INTERLEAVED4, layout=0), nv.ERR_UNSUPPORTED, "HND pages only"),
])
def test_materialize_rejects(lib, kw, code, text):
    assert materialize(lib, **kw) == code
    assert text in err(lib)


@pytest.mark.parametrize("kw,code,text", [
    (dict(D=96), nv.ERR_INVALID_ARG, "divisible by 64"),
    (dict(ps=6), nv.ERR_INVALID_ARG, "divisible by 4"),
    (dict(maxb=0), nv.ERR_INVALID_ARG, "max_batch_size"),
    (dict(maxb=20000), nv.ERR_INVALID_ARG, "max_batch_size"),
    (dict(dps=16 * 8 * 64 - 16), nv.ERR_INVALID_ARG, "smaller than a page"),
    (dict(dps=16 * 8 * 64 + 8), nv.ERR_ALIGNMENT, "multiple of 16"),
    (dict(sps=16 * 8 * 8 + 1), nv.ERR_ALIGNMENT, "even"),
    (dict(vsf=2), nv.ERR_INVALID_ARG, "v_scale_layout"),
    (dict(vsf=nv.SF_INTERLEAVED4, layout=0), nv.ERR_UNSUPPORTED, "HND pages only"),
])
def test_materializer_prepare_rejects(lib, kw, code, text):
    a = dict(ps=16, H=8, D=128, layout=1, shared=1, vsf=nv.SF_LINEAR, dps=16 * 8 * 64,
             sps=16 * 8 * 8, maxb=64)
    a.update(kw)
    m = nv._Materializer()
    m.magic = 123
    assert lib.nvfp4_materializer_prepare(ctypes.byref(m), a["ps"], a["H"], a["D"], a["layout"],
                                          a["shared"], a["vsf"], a["dps"], a["sps"],
                                          a["maxb"]) == code
    assert text in err(lib)
    assert m.magic == 0  # a failed prepare leaves the struct unusable


def test_materializer_run_needs_a_prepared_struct(lib):
    m = nv._Materializer()
    assert lib.nvfp4_materializer_run(
        ctypes.byref(m), cache(), cache(), ctypes.c_void_p(FAKE), 4, ctypes.c_void_p(FAKE), 2, 4,
        None, -1, ctypes.c_void_p(FAKE), 9, ctypes.c_void_p(FAKE), None, None,
        None) == nv.ERR_INVALID_ARG
    assert "not prepared" in err(lib)
    assert lib.nvfp4_materializer_run(
        None, cache(), cache(), ctypes.c_void_p(FAKE), 4, ctypes.c_void_p(FAKE), 2, 4, None, -1,
        ctypes.c_void_p(FAKE), 9, ctypes.c_void_p(FAKE), None, None, None) == nv.ERR_INVALID_ARG


def test_materializer_interleaved_needs_hnd():
    with pytest.raises(ValueError, match="HND"):
        nv.NVFP4KVMaterializer(8, 16, 128, "cuda", kv_layout="NHD",
                               v_block_scales_layout="interleaved4")
    with pytest.raises(KeyError):
        nv.NVFP4KVMaterializer(8, 16, 128, "cuda", v_block_scales_layout="swizzled")


def test_global_scale_rejects(lib):
    f = lib.nvfp4_make_global_scale
    assert f(ctypes.c_void_p(FAKE), 3, 16, None, ctypes.c_void_p(FAKE), None) == nv.ERR_INVALID_ARG
    assert f(ctypes.c_void_p(FAKE), 1, -1, None, ctypes.c_void_p(FAKE), None) == nv.ERR_INVALID_ARG
    assert f(ctypes.c_void_p(FAKE), 1, 16, None, None, None) == nv.ERR_INVALID_ARG
    assert f(ctypes.c_void_p(FAKE + 2), 1, 16, None, ctypes.c_void_p(FAKE), None) == nv.ERR_ALIGNMENT


def test_ops_refuse_cpu_tensors():
    import torch
    with pytest.raises(ValueError):
        nv.nvfp4_make_global_scale(torch.zeros(16, dtype=torch.bfloat16))


def test_dev_scale_append_rejects_null_scales(lib):
    f = lib.nvfp4_quantize_append_paged_dev_scale
    r = f(ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE), 1, 4, 8, 128, 1024, 1024,
          ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE), cache(), cache(), 16, 0,
          ctypes.c_void_p(FAKE), 16, ctypes.c_void_p(FAKE), None, 2, None, ctypes.c_void_p(FAKE),
          None, None, None, None)
    assert r == nv.ERR_INVALID_ARG and "scale" in err(lib)


def kv_quantize(lib, **kw):
    a = dict(x=FAKE, dt=1, rows=4, cols=128, stride=128, gs=FAKE, out=FAKE, recipe=None)
    a.update(kw)
    return lib.nvfp4_kv_quantize(ctypes.c_void_p(a["x"]) if a["x"] else None, a["dt"], a["rows"],
                                 a["cols"], a["stride"],
                                 ctypes.c_void_p(a["gs"]) if a["gs"] else None, a["recipe"],
                                 ctypes.c_void_p(a["out"]), ctypes.c_void_p(FAKE), None, None,
                                 None)


@pytest.mark.parametrize("kw,code,text", [
    (dict(dt=7), nv.ERR_INVALID_ARG, "dtype"),
    (dict(cols=40), nv.ERR_INVALID_ARG, "cols"),
    (dict(cols=0), nv.ERR_INVALID_ARG, "cols"),
    (dict(rows=-1), nv.ERR_INVALID_ARG, "rows"),
    (dict(stride=64), nv.ERR_INVALID_ARG, "row_stride"),
    (dict(x=FAKE + 8), nv.ERR_ALIGNMENT, "aligned"),
    (dict(stride=132), nv.ERR_ALIGNMENT, "aligned"),
    (dict(out=FAKE + 4), nv.ERR_ALIGNMENT, "aligned"),
    (dict(gs=0), nv.ERR_INVALID_ARG, "null"),
])
def test_kv_quantize_rejects(lib, kw, code, text):
    assert kv_quantize(lib, **kw) == code
    assert text in err(lib)


def kv_dequantize(lib, **kw):
    a = dict(fp4=FAKE, rows=4, cols=128, gs=FAKE, out=FAKE, odt=1, ws=None)
    a.update(kw)
    return lib.nvfp4_kv_dequantize(ctypes.c_void_p(a["fp4"]), ctypes.c_void_p(FAKE), a["rows"],
                                   a["cols"], ctypes.c_void_p(a["gs"]) if a["gs"] else None,
                                   ctypes.c_void_p(a["out"]), a["odt"], None,
                                   ctypes.c_void_p(a["ws"]) if a["ws"] else None, None)


@pytest.mark.parametrize("kw,code,text", [
    (dict(odt=3), nv.ERR_INVALID_ARG, "out_dtype"),
    (dict(cols=24), nv.ERR_INVALID_ARG, "cols"),
    (dict(rows=-2), nv.ERR_INVALID_ARG, "rows"),
    (dict(fp4=FAKE + 4), nv.ERR_ALIGNMENT, "aligned"),
    (dict(out=FAKE + 8), nv.ERR_ALIGNMENT, "aligned"),
    (dict(gs=0), nv.ERR_INVALID_ARG, "null"),
])
def test_kv_dequantize_rejects(lib, kw, code, text):
    assert kv_dequantize(lib, **kw) == code
    assert text in err(lib)


def test_empty_contiguous_ops_are_no_ops(lib):
    assert kv_quantize(lib, rows=0) == nv.OK
    assert kv_dequantize(lib, rows=0) == nv.OK


def test_a_misaligned_workspace_is_rejected(lib):
    """The work-distribution workspace must be 8-byte aligned (NULL is allowed)."""
    assert append(lib, ws=FAKE + 4) == nv.ERR_ALIGNMENT and "workspace" in err(lib)
    assert dequant(lib, ws=FAKE + 4) == nv.ERR_ALIGNMENT and "workspace" in err(lib)
    assert materialize(lib, ws=FAKE + 2) == nv.ERR_ALIGNMENT and "workspace" in err(lib)
    assert kv_dequantize(lib, ws=FAKE + 4) == nv.ERR_ALIGNMENT and "workspace" in err(lib)
