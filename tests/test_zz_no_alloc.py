"""nvfp4_dequantize_paged_no_alloc: the paged dequantize for callers that cannot hand the
library any device memory (a memory planner that owns every byte, or code that must not
call cudaMalloc). It keeps its work queue in an array the library holds instead of in a
caller's workspace. Called here through the C ABI, twice in a row, and compared byte for
byte with nvfp4_dequantize_paged on the same cache, which takes a workspace from the
binding. This file is collected last, so a run that stops at its first failure has run
every other test before it; it also passes on its own in a fresh process."""
import ctypes

import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


def test_no_alloc_dequant_matches_the_workspace_call(gpu_lib):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import bench
    nv = gpu_lib
    lib = nv.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    # enough requests and pages that the work queue hands out thousands of items
    w = W.random_case(900, B=24, H=8, D=128, ps=16, layout=W.HND, dtype=torch.bfloat16,
                      recipe=W.Recipe(256.0, 0, True), max_len=1200, min_len=300)
    step = bench.Step(w, dev)
    step._global_scales()
    step._append()
    ref_k = torch.full_like(step.out_k, 0.5)
    ref_v = torch.full_like(step.out_v, 0.5)
    nv.nvfp4_dequantize_paged(step.cache, step.sf, step.bt, step.seq_lens, step.gk, step.gv,
                              ref_k, ref_v, "HND")
    kc, vc = nv.paged_caches(step.cache, step.sf)
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    for call in range(2):
        out_k = torch.full_like(step.out_k, 0.5)
        out_v = torch.full_like(step.out_v, 0.5)
        rc = lib.nvfp4_dequantize_paged_no_alloc(
            kc._c(), vc._c(), w.ps, w.H, w.D, nv.HND, ptr(step.bt), nv.I32, step.bt.shape[1],
            ptr(step.seq_lens), w.B, ptr(step.gk), ptr(step.gv), ptr(out_k), ptr(out_v),
            nv.BF16, out_k.shape[1], ptr(status),
            ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream))
        assert rc == nv.OK, lib.nvfp4_last_error_string().decode()
        torch.cuda.synchronize(dev)
        assert int(status.item()) == 0, (call, hex(int(status.item())))
        # bit-exact, including the rows past each request's length (left at 0.5)
        assert torch.equal(out_k.view(torch.int16), ref_k.view(torch.int16)), call
        assert torch.equal(out_v.view(torch.int16), ref_v.view(torch.int16)), call
