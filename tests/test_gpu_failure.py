"""Failure detection in the pipelined kernels, without a GPU fault.

Every shared-memory stage wait in the TMA-fed kernels is bounded. Here the host makes a
wait run out: NVFP4KV_TEST_STALL_PIPELINE=1 makes each CTA's producer withhold its first
stage (a barrier nothing completes) and shortens the wait limit. The contiguous quantize
runs the append's pipeline and the contiguous dequantize a ring of its own; both are checked
the same way. The call must come back
on its own with NVFP4_DEV_TIMEOUT set, and the CUDA context must stay usable: the same call
without the switch then matches the CPU oracle.
"""
import os

import numpy as np
import pytest
import torch

import workloads as W
from tests import pipelines as PL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda(gpu_lib):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    yield


@pytest.fixture
def stall_env():
    os.environ["NVFP4KV_TEST_STALL_PIPELINE"] = "1"
    # a call this small would run the append's direct-load kernel, which has no ring
    os.environ["NVFP4KV_TEST_APPEND_KERNEL"] = "ring"
    try:
        yield
    finally:
        os.environ.pop("NVFP4KV_TEST_STALL_PIPELINE", None)
        os.environ.pop("NVFP4KV_TEST_APPEND_KERNEL", None)


def _case():
    return W.random_case(600, B=6, H=8, D=128, ps=16, layout=W.HND, dtype=torch.bfloat16,
                         recipe=W.Recipe(256.0, 0, True), max_len=120, min_len=20)


def test_stalled_pipelines_report_timeout_and_recover(stall_env):
    import nvfp4_paged_kv_02_gb300 as nv
    w = _case()
    dev = torch.device("cuda")
    t = lambda a: torch.as_tensor(np.ascontiguousarray(a)).to(dev)
    kd = torch.zeros((w.num_pages, w.H, w.ps, w.D // 2), dtype=torch.uint8, device=dev)
    ks = torch.zeros((w.num_pages, w.H, w.ps, w.D // 16), dtype=torch.uint8, device=dev)
    vd, vs = kd.clone(), ks.clone()
    g = torch.tensor([0.01], dtype=torch.float32, device=dev)
    r = PL.gpu_recipe(w.recipe)
    for op in ("append", "dequant", "materialize", "kv_quantize", "kv_dequantize"):
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        if op == "append":
            nv.nvfp4_quantize_append_paged(w.k.to(dev), w.v.to(dev), t(w.batch_indices),
                                           t(w.positions), (kd, vd), (ks, vs), t(w.kv_indices),
                                           t(w.kv_indptr), None, g, g, "HND", r, st)
        elif op == "dequant":
            ok = torch.zeros((w.B, w.max_seq_len, w.H, w.D), dtype=torch.bfloat16, device=dev)
            nv.nvfp4_dequantize_paged((kd, vd), (ks, vs), t(w.block_tables), t(w.seq_lens), g, g,
                                      ok, ok.clone(), "HND", st)
        elif op == "materialize":
            nv.nvfp4_materialize_fp8(kd, vd, ks, vs, t(w.mat_block_tables), t(w.seq_lens),
                                     w.max_kv_len, True, kv_layout="HND", dev_status=st)
        elif op == "kv_quantize":  # the contiguous quantize shares the append's pipeline
            nv.nvfp4_kv_quantize(w.k.to(dev).reshape(w.nnz, -1), g, r, dev_status=st)
        else:  # nnz rows of 1024 elements: whole chunks of the contiguous dequantize's ring
            codes = torch.zeros((w.nnz, w.H * w.D // 2), dtype=torch.uint8, device=dev)
            scales = torch.zeros((w.nnz, w.H * w.D // 16), dtype=torch.uint8, device=dev)
            nv.nvfp4_kv_dequantize(codes, scales, g, torch.bfloat16, dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) & nv.DEV_TIMEOUT, (op, int(st.item()))
    # the context is still usable: a normal run matches the oracle
    os.environ.pop("NVFP4KV_TEST_STALL_PIPELINE", None)
    g_res = PL.run_gpu(w)
    o_res = PL.run_oracle(w)
    PL.assert_same(g_res, o_res, "after stall")
