"""Benchmark of the NVFP4 paged KV-cache hot path on GB300.

One step is the whole path over one batch of synthetic input: the global decode scales of
K and V, quantize-and-append of every token into the paged NVFP4 pool, paged dequantize of
every request into contiguous bf16, and the FP8 materialize of every active page.

Default workload ("large_pool"): batch 256, lengths U[1024, 16384] (about 2.2 M tokens),
page_size 16, 8 KV heads, head_dim 128, HND, a ~40 GB pool with the active pages placed at
random, bf16 N(0, sigma^2) with sigma ~ U[0.5, 4] per (K/V, head), 4over6 MAE with
e4m3_max 256 and fp16 error. Inputs (9 GB) are larger than L2, so no flush is needed.

Metric: algorithmic HBM bytes of the step (data only; index traffic excluded) / step time,
in GB/s; per-op GB/s, % of 8 TB/s, % of the measured copy bandwidth and tokens/s as well.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Under torchrun each rank runs its own replica of the workload on its own GPU (the path
shards by request with no exchange): weak scaling, max time over ranks.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "HBM GB/s (% of 8 TB/s) and tokens/s per op: append, dequant_paged, materialize"
NOMINAL_HBM_GBS = 8000.0


def arith_dtype(w: W.Workload) -> str:
    """The arithmetic the path computes in: binary32 everywhere, plus binary16 for the
    4over6 error under the fast-math recipe."""
    r = w.recipe
    return "f32+f16" if r is not None and r.err_use_fast_math else "f32"


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d.get("hbm_gbs", 6800.0)), "measured"
    return 6800.0, "fallback"


# ---------------------------------------------------------------------------------------
# algorithmic bytes (data only) of each op for a workload
# ---------------------------------------------------------------------------------------

def op_bytes(w: W.Workload, n_active_pages: int):
    H, D, ps = w.H, w.D, w.ps
    row = H * D
    nnz = w.nnz
    toks = int(np.minimum(w.seq_lens, w.max_seq_len).sum())
    return {
        "global_scale": 2 * nnz * row * 2,
        "append": nnz * H * (4 * D + D + D // 8),
        "dequant_paged": toks * H * (D + D // 8 + 4 * D),
        "materialize": n_active_pages * ps * H * (3 * D + D // 8) + 2 * H * ps * D
        + w.B * (-(-w.max_kv_len // ps)) * 4,
    }, {"global_scale": nnz, "append": nnz, "dequant_paged": toks,
        "materialize": n_active_pages * ps}


# ---------------------------------------------------------------------------------------
# replicas: the slowest rank's time
# ---------------------------------------------------------------------------------------

def max_over_ranks(x: float, dev: torch.device) -> float:
    """The largest value of x over all ranks (x itself when not running distributed)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return x
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------------------
# DRAM traffic of a kernel, from a committed ncu summary
# ---------------------------------------------------------------------------------------

CSRC = os.path.join(ROOT, "nvfp4_paged_kv_02_gb300", "csrc")
KERNEL_SOURCES = {
    "append": ["append.cu"], "dequant_paged": ["dequant.cu"],
    "materialize": ["materialize.cu"], "kv_quantize": ["append.cu"],
    "kv_dequantize": ["dequant.cu"],
}
SHARED_SOURCES = ["device.cuh", "internal.h", "pipeline.cuh", "scan.cuh"]
TRAFFIC_FILES = [os.path.join(ROOT, "profiles", f)
                 for f in ("dram_traffic_large_pool.md", "dram_traffic_contig.md")]


def source_hash(op: str) -> str:
    """First 16 hex digits of the sha256 of the op's translation unit and shared headers."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[op] + SHARED_SOURCES:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def traffic_per_launch(op: str, units: int):
    """DRAM bytes (read + write) per launch of the op's kernel, from ncu captures of the same
    kernel at two sizes: traffic = marginal bytes per unit * units + bytes at zero units (the
    second is negative: output lines still dirty in L2 when the kernel ends, written back
    later). None when there is no capture or the kernel's sources changed since."""
    want = source_hash(op)
    for path in TRAFFIC_FILES:
        if not os.path.exists(path):
            continue
        with open(path) as f:
            for ln in f:
                cells = [c.strip().strip("`") for c in ln.strip().strip("|").split("|")]
                if len(cells) >= 12 and cells[0] == op and cells[1] == want:
                    try:
                        return float(cells[8]) * units + float(cells[9])
                    except ValueError:
                        return None
    return None


# ---------------------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    INTERVAL_MS = 20

    def __init__(self, out_path: str):
        self.path = out_path
        self.proc = None

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.INTERVAL_MS)], stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self, t0: float = 0.0, t1: float = float("inf")):
        """Stop sampling; summarize the samples taken between host times t0 and t1."""
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        want = vis.split(",")[int(os.environ.get("LOCAL_RANK", "0"))] if vis else None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for ln in f:
                parts = [p.strip() for p in ln.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    whole, _, frac = parts[0].partition(".")
                    ts = time.mktime(time.strptime(whole, "%Y/%m/%d %H:%M:%S"))
                    ts += float("0." + frac) if frac.isdigit() else 0.0
                except ValueError:
                    continue
                if not (t0 - 0.05 <= ts <= t1 + 0.05):
                    continue
                parts = parts[1:]
                if want is not None and want.isdigit() and parts[0] != want:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm),
                "interval_ms": self.INTERVAL_MS, "window_s": round(t1 - t0, 3)}


# ---------------------------------------------------------------------------------------
# the device state of one step
# ---------------------------------------------------------------------------------------

class Step:
    """Buffers and launches of one pass of the hot path on the current device."""

    def __init__(self, w: W.Workload, dev: torch.device, v_scales: str = "linear"):
        import nvfp4_paged_kv_02_gb300 as nv
        self.nv, self.w, self.dev = nv, w, dev
        r = w.recipe
        self.recipe = None if r is None else nv.NVFP44Over6Config(
            r.e4m3_max, "MSE" if r.err_mode else "MAE", bool(r.err_use_fast_math))
        t = lambda a: torch.as_tensor(np.ascontiguousarray(a)).to(dev)
        if v_scales not in ("linear", "interleaved4"):
            raise ValueError(v_scales)
        if v_scales == "interleaved4" and w.layout != W.HND:
            raise SystemExit("4-token-interleaved V scales need an HND workload")
        self.v_scales = v_scales
        inner = (w.ps, w.H) if w.layout == W.NHD else (w.H, w.ps)
        self.cache = tuple(torch.empty((w.num_pages, *inner, w.D // 2), dtype=torch.uint8,
                                       device=dev) for _ in range(2))
        self.sf = tuple(torch.empty((w.num_pages, *inner, w.D // 16), dtype=torch.uint8,
                                    device=dev) for _ in range(2))
        self.k, self.v = w.k.to(dev), w.v.to(dev)
        self.bi, self.pos = t(w.batch_indices), t(w.positions)
        self.kv_indices, self.kv_indptr = t(w.kv_indices), t(w.kv_indptr)
        self.last = t(w.kv_last_page_len)
        self.bt, self.seq_lens = t(w.block_tables), t(w.seq_lens)
        self.mat_bt = t(w.mat_block_tables)
        self.indptr = None if w.kv_page_indptr is None else t(w.kv_page_indptr)
        self.out_k = torch.empty((w.B, w.max_seq_len, w.H, w.D), dtype=w.dtype, device=dev)
        self.out_v = torch.empty_like(self.out_k)
        n_out, mpps = nv.nvfp4_materialize_fp8_out_pages(w.B, w.max_kv_len, w.ps, w.mat_num_pages)
        self.fp8 = torch.empty((n_out, 2, w.H, w.ps, w.D), dtype=torch.float8_e4m3fn, device=dev)
        self.tables = torch.empty((w.B, mpps), dtype=torch.int32, device=dev)
        self.gk = torch.empty(1, dtype=torch.float32, device=dev)
        self.gv = torch.empty(1, dtype=torch.float32, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.lay = "NHD" if w.layout == W.NHD else "HND"
        # per tensor: one launch for a global scale of at most 2^16 elements, else amax + finalize
        gs_launches = 1 if self.k.numel() <= (1 << 16) else 2
        self.launches_per_step = 2 * gs_launches + 3  # 2 global scales, append, dequant, materialize
        if w.prefill_k is not None:
            # rows already in the cache before the measured append (untimed)
            pk, pv = w.prefill_k.to(dev), w.prefill_v.to(dev)
            nv.nvfp4_make_global_scale(torch.cat([pk, self.k]), self.recipe, out=self.gk)
            nv.nvfp4_make_global_scale(torch.cat([pv, self.v]), self.recipe, out=self.gv)
            nv.nvfp4_quantize_append_paged(
                pk, pv, t(w.prefill_batch_indices), t(w.prefill_positions), self.cache, self.sf,
                self.kv_indices, self.kv_indptr, self.last, float(self.gk.item()),
                float(self.gv.item()), self.lay, self.recipe, self.status)
            del pk, pv

        self.mat_v_sf = self.sf[1]
        if v_scales == "interleaved4":
            # The measured append writes the same bytes at every step. Its V scales, rewritten
            # once in the 4-token-interleaved layout, are what the materialize then reads.
            self._global_scales()
            self._append()
            P, Hh, ps, nb = self.sf[1].shape
            self.mat_v_sf = self.sf[1].view(P, Hh, ps // 4, 4, nb).transpose(3, 4) \
                .contiguous().view(P, Hh, ps, nb)
        self._ops = [self._global_scales, self._append, self._dequant, self._materialize]

    NAMES = ("global_scale", "append", "dequant_paged", "materialize")

    def _global_scales(self):
        self.nv.nvfp4_make_global_scale(self.k, self.recipe, out=self.gk)
        self.nv.nvfp4_make_global_scale(self.v, self.recipe, out=self.gv)

    def _append(self):
        # the scales stay on the device: no host round trip inside the step
        self.nv.nvfp4_quantize_append_paged(
            self.k, self.v, self.bi, self.pos, self.cache, self.sf, self.kv_indices,
            self.kv_indptr, self.last, self.gk, self.gv, self.lay, self.recipe, self.status)

    def _dequant(self):
        self.nv.nvfp4_dequantize_paged(self.cache, self.sf, self.bt, self.seq_lens, self.gk,
                                       self.gv, self.out_k, self.out_v, self.lay, self.status)

    def _materialize(self):
        w = self.w
        self.nv.nvfp4_materialize_fp8(
            self.cache[0], self.cache[1], self.sf[0], self.mat_v_sf, self.mat_bt, self.seq_lens,
            w.max_kv_len, w.mat_shared, self.fp8, self.indptr, w.mat_num_pages, self.lay,
            self.tables, True, self.status, v_block_scales_layout=self.v_scales)

    def run(self, ev=None, flush=None):
        run_ops(self._ops, ev, flush)

    def diagnostics(self):
        """Share of the FP8 copy's active-page elements at +-448, the E4M3 maximum: the
        products e2m1 * S that saturated, plus any exactly equal to 448. Read once, after
        the timed steps."""
        pages = self.tables[self.tables > 0].flatten()
        fp8 = self.fp8.view(torch.uint8)
        at_max = 0
        for c in torch.split(pages.long(), 4096):
            at_max += int(((fp8[c] & 0x7F) == 0x7E).sum().item())
        total = pages.numel() * fp8[0].numel()
        return {"materialize_fp8_at_448_fraction": at_max / total if total else 0.0}

    def op_bytes(self):
        return op_bytes(self.w, active_pages(self.w))

    def config(self):
        w = self.w
        return {"workload": w.name, "batch": w.B, "tokens": w.nnz, "page_size": w.ps,
                "num_kv_heads": w.H, "head_dim": w.D,
                "kv_layout": "NHD" if w.layout == W.NHD else "HND",
                "input_dtype": str(w.dtype).replace("torch.", ""),
                "recipe": None if w.recipe is None else vars(w.recipe),
                "pool_pages": w.num_pages, "active_pages": active_pages(w),
                "materialize_v_scales": self.v_scales}


def run_ops(ops, ev=None, flush=None):
    """Run the ops in order; ev (two events per op) brackets each op; flush, when given,
    runs before each op, outside its events."""
    for i, op in enumerate(ops):
        if flush is not None:
            flush()
        if ev is not None:
            ev[2 * i].record()
        op()
        if ev is not None:
            ev[2 * i + 1].record()


class ContigStep:
    """The contiguous form ("FP4 KV Cache Quantization": nvfp4_kv_quantize and
    nvfp4_kv_dequantize) on the large-pool K and V rows, each a [tokens, H*D] tensor: the two
    global scales, the quantize of each tensor, then the dequantize of each."""

    NAMES = ("global_scale", "kv_quantize", "kv_dequantize")

    def __init__(self, w: W.Workload, dev: torch.device):
        import nvfp4_paged_kv_02_gb300 as nv
        self.nv, self.w, self.dev = nv, w, dev
        r = w.recipe
        self.recipe = None if r is None else nv.NVFP44Over6Config(
            r.e4m3_max, "MSE" if r.err_mode else "MAE", bool(r.err_use_fast_math))
        self.rows, self.cols = w.nnz, w.H * w.D
        self.k = w.k.to(dev).view(self.rows, self.cols)
        self.v = w.v.to(dev).view(self.rows, self.cols)
        u8 = dict(dtype=torch.uint8, device=dev)
        self.q = [(torch.empty((self.rows, self.cols // 2), **u8),
                   torch.empty((self.rows, self.cols // 16), **u8)) for _ in range(2)]
        self.out = [torch.empty((self.rows, self.cols), dtype=w.dtype, device=dev)
                    for _ in range(2)]
        self.gk = torch.empty(1, dtype=torch.float32, device=dev)
        self.gv = torch.empty(1, dtype=torch.float32, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        gs_launches = 1 if self.k.numel() <= (1 << 16) else 2
        self.launches_per_step = 2 * gs_launches + 4  # 2 global scales, 2 quantize, 2 dequantize
        self._ops = [self._global_scales, self._quantize, self._dequantize]

    def _global_scales(self):
        self.nv.nvfp4_make_global_scale(self.k, self.recipe, out=self.gk)
        self.nv.nvfp4_make_global_scale(self.v, self.recipe, out=self.gv)

    def _quantize(self):
        for x, g, q in ((self.k, self.gk, self.q[0]), (self.v, self.gv, self.q[1])):
            self.nv.nvfp4_kv_quantize(x, g, self.recipe, out=q, dev_status=self.status)

    def _dequantize(self):
        for q, g, o in ((self.q[0], self.gk, self.out[0]), (self.q[1], self.gv, self.out[1])):
            self.nv.nvfp4_kv_dequantize(q[0], q[1], g, o.dtype, out=o)

    def run(self, ev=None, flush=None):
        run_ops(self._ops, ev, flush)

    def op_bytes(self):
        n = self.rows * self.cols
        per = 2 * n * 2 + 2 * (n // 2 + n // 16)  # both tensors: 16-bit side + codes + scales
        return ({"global_scale": 2 * n * 2, "kv_quantize": per, "kv_dequantize": per},
                {"global_scale": self.rows, "kv_quantize": self.rows,
                 "kv_dequantize": self.rows})

    def config(self):
        w = self.w
        return {"workload": "contig", "source": "large_pool K and V rows", "tokens": self.rows,
                "cols": self.cols, "input_dtype": str(w.dtype).replace("torch.", ""),
                "recipe": None if w.recipe is None else vars(w.recipe)}


def make_workload(name: str, dev: torch.device, batch: int = 256,
                  pool_gb: float = W.LARGE_POOL_BYTES / 1e9) -> W.Workload:
    if name in ("large_pool", "contig"):
        return W.large_pool(device=str(dev), B=batch, pool_bytes=pool_gb * 1e9)
    return W.NAMED[name]()


def active_pages(w: W.Workload) -> int:
    mpps = -(-w.max_kv_len // w.ps)
    return int(np.minimum(-(-w.seq_lens.astype(np.int64) // w.ps), mpps).sum())


# ---------------------------------------------------------------------------------------
# the other configurations, measured after the headline step
# ---------------------------------------------------------------------------------------

# (key, workload, V-scale layout of the materialize input)
SECONDARY = (("decode", "decode", "linear"), ("prefill", "prefill", "linear"),
             ("materialize", "materialize", "linear"),
             ("materialize_v_interleaved4", "materialize", "interleaved4"),
             ("contig", "contig", "linear"))


def time_ops(step, dev: torch.device, n_steps: int, warmup: int = 3):
    """Mean device time (ms) per op of `step` over n_steps timed steps after `warmup`
    untimed ones. When every op moves under 1 GB, L2 is flushed before each op (256 MB
    written, then 256 MB read), outside the op's events."""
    nbytes, _ = step.op_bytes()
    small = max(nbytes.values()) < 1e9
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if small else None
    flush_read = torch.zeros(256 << 20, dtype=torch.uint8, device=dev) if small else None
    count = [0]

    def flush_l2():
        count[0] += 1
        flush.fill_(count[0] & 0xFF)
        flush_read.sum()

    for _ in range(warmup):
        step.run()
    n_ops = len(step.NAMES)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * n_ops)]
           for _ in range(n_steps)]
    torch.cuda.synchronize(dev)
    for s in range(n_steps):
        step.run(evs[s], flush_l2 if small else None)
    torch.cuda.synchronize(dev)
    op_ms = {k: float(np.mean([evs[s][2 * i].elapsed_time(evs[s][2 * i + 1])
                               for s in range(n_steps)]))
             for i, k in enumerate(step.NAMES)}
    return op_ms, small


def op_table(step, op_ms, peak: float):
    nbytes, ntok = step.op_bytes()
    out = {}
    for k, ms in op_ms.items():
        gbs = nbytes[k] / (ms * 1e-3) / 1e9
        out[k] = {"us": ms * 1e3, "bytes": nbytes[k], "GB_s": gbs,
                  "pct_of_8TBs": 100 * gbs / NOMINAL_HBM_GBS,
                  "pct_of_measured_copy": 100 * gbs / peak,
                  "tokens_per_s": ntok[k] / (ms * 1e-3)}
    return out


def materialize_host_cost(step, n_calls: int = 200, layers: int = 32):
    """Host time per call (CPU clock, microseconds) of issuing the materialize four ways on
    the materialize workload ("NVFP4KVMaterializer": the functional call validates every
    tensor and allocates the block table each time, the class validates once): the
    functional nvfp4_materialize_fp8 (allocating its outputs), NVFP4KVMaterializer.run()
    with caller-owned outputs, the prepared C entry point called through ctypes with its
    arguments marshalled once, and one replay of a CUDA graph holding `layers` run() calls,
    per layer. Only the enqueueing is timed; the device work drains outside the timer."""
    nv, w, dev = step.nv, step.w, step.dev
    lay = step.lay
    kd, vd = step.cache
    ks, vs = step.sf
    args = (kd, vd, ks, vs, step.mat_bt, step.seq_lens)

    def per_call(fn, n):
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for _ in range(n):
            fn()
        t1 = time.perf_counter()
        torch.cuda.synchronize(dev)
        return (t1 - t0) / n * 1e6

    def functional():
        nv.nvfp4_materialize_fp8(*args, w.max_kv_len, w.mat_shared, None, step.indptr,
                                 w.mat_num_pages, lay)

    m = nv.NVFP4KVMaterializer(w.H, w.ps, w.D, dev, uses_shared_paged_kv_idx=w.mat_shared,
                               kv_layout=lay, max_batch_size=w.B)
    out, tables = step.fp8, step.tables

    def run():
        m.run(*args, step.indptr, out=out, fp8_block_tables=tables)

    # the C entry point alone, its arguments marshalled once (ctypes call overhead included)
    import ctypes
    L = nv.load()
    kc, vc = nv._one_cache(kd, ks), nv._one_cache(vd, vs)
    prepared = m._prepare(kc.data_page_stride, kc.sf_page_stride, m._max_batch)
    vp = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    c_args = (ctypes.byref(prepared), kc._c(), vc._c(), vp(step.mat_bt), step.mat_bt.shape[-1],
              vp(step.seq_lens), tables.shape[0], tables.shape[1], vp(step.indptr),
              out.shape[0] - 1, vp(out), out.shape[0], vp(tables), None,
              *nv._ws_stream(dev))

    def c_run():
        if L.nvfp4_materializer_run(*c_args) != 0:
            raise RuntimeError("nvfp4_materializer_run failed")

    for fn in (functional, run, c_run):  # warm-up: first-call set-up, allocator, shapes
        fn()
        fn()
    res = {"functional_us": per_call(functional, n_calls), "materializer_run_us": per_call(run, n_calls),
           "c_abi_run_us": per_call(c_run, n_calls)}
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        run()
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(layers):
            run()
    graph.replay()
    torch.cuda.synchronize(dev)
    res["graph_replay_us_per_layer"] = per_call(graph.replay, max(4, n_calls // layers)) / layers
    res["graph_layers"] = layers
    res["calls"] = n_calls
    return res


def measure_configs(w_large: W.Workload, dev: torch.device, n_steps: int = 20):
    """Per-op figures of the decode, prefill and materialize workloads (the last also with V
    scales in the 4-token-interleaved layout) and of the contiguous form (on the large pool's
    K and V rows), each timed on its own after the headline step."""
    peak, _ = measured_peaks()
    out = {}
    for name, wl, v_scales in SECONDARY:
        w = w_large if wl == "contig" else make_workload(wl, dev)
        step = ContigStep(w, dev) if wl == "contig" else Step(w, dev, v_scales)
        op_ms, small = time_ops(step, dev, n_steps)
        status = int(step.status.item())
        host = materialize_host_cost(step) if name == "materialize" else None
        out[name] = {"config": step.config(), "steps": n_steps,
                     "l2": "flushed before every op" if small else "inputs larger than L2",
                     "ops": op_table(step, op_ms, peak), "device_status": status,
                     "gpu_launches": step.launches_per_step * n_steps}
        if host is not None:
            out[name]["host_cost"] = host
        del step
        torch.cuda.empty_cache()
    return out


# ---------------------------------------------------------------------------------------
# the CPU oracle on a bounded sample (baseline and reference arm)
# ---------------------------------------------------------------------------------------

def oracle_sample(w: W.Workload, n_req: int, max_tokens: int = 0):
    """A sub-batch of the workload (its first n_req requests, their rows, a compact pool)
    as host arrays, plus its algorithmic bytes. With max_tokens > 0 the sample instead
    takes whole requests in order until max_tokens rows, the last one cut short."""
    lens_all = w.seq_lens.astype(np.int64)
    if max_tokens > 0:
        cum = np.cumsum(lens_all)
        n_req = int(np.searchsorted(cum, max_tokens)) + 1
        n_req = min(n_req, w.B)
    sel = np.arange(min(n_req, w.B))
    lens = lens_all[sel].copy()
    if max_tokens > 0:
        before = int(lens[:-1].sum())
        lens[-1] = max(1, min(lens[-1], max_tokens - before))
    rows = np.isin(w.batch_indices, sel) & (w.positions < lens[np.minimum(w.batch_indices, len(sel) - 1)])
    sub = W.make_paged("sample", 0, B=len(sel), H=w.H, D=w.D, ps=w.ps, layout=w.layout,
                       dtype=w.dtype, lens_old=np.zeros(len(sel), np.int64), lens_new=lens,
                       recipe=w.recipe, sampler=lambda r, n: np.zeros((n, w.H, w.D), np.float32),
                       max_kv_len=w.max_kv_len, extra_pages=1)
    sub.k = w.k[torch.from_numpy(np.flatnonzero(rows)).to(w.k.device)].cpu()
    sub.v = w.v[torch.from_numpy(np.flatnonzero(rows)).to(w.v.device)].cpu()
    sub.batch_indices = w.batch_indices[rows]
    sub.positions = w.positions[rows]
    nb, _ = op_bytes(sub, active_pages(sub))
    return sub, sum(nb.values())


def time_oracle(sub: W.Workload, nthreads: int = 0) -> float:
    from tests import pipelines as PL
    t0 = time.perf_counter()
    PL.run_oracle(sub, nthreads=nthreads)
    return time.perf_counter() - t0


def contig_sample(w: W.Workload, n_rows: int):
    """The first n_rows token rows of K and V as [n, H*D] host tensors, plus the algorithmic
    bytes of the contiguous step on them."""
    n = max(1, min(n_rows, w.nnz))
    k = w.k[:n].reshape(n, -1).cpu()
    v = w.v[:n].reshape(n, -1).cpu()
    e = k.numel()
    return (k, v), 2 * e * 2 + 2 * (2 * (2 * e * 2 + 2 * (e // 2 + e // 16)))


def time_oracle_contig(kv, recipe) -> float:
    import oracle
    t0 = time.perf_counter()
    for x in kv:
        bits = W.bits16(x)
        bf16 = x.dtype == torch.bfloat16
        gs = oracle.global_scale(bits, bf16, recipe)
        codes, sf = oracle.kv_quantize(bits, bf16, gs, recipe)
        oracle.kv_dequantize(codes, sf, gs, bf16)
    return time.perf_counter() - t0


def cpu_baseline_contig(w: W.Workload, target_s: float = 15.0):
    import oracle
    n = 4096
    kv, nbytes = contig_sample(w, n)
    dt = time_oracle_contig(kv, w.recipe)
    while dt < target_s / 4 and n < w.nnz:
        n = min(w.nnz, max(n + 1, int(n * min(8.0, target_s / 2 / max(dt, 1e-3)))))
        kv, nbytes = contig_sample(w, n)
        dt = time_oracle_contig(kv, w.recipe)
    return {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": oracle.max_threads(),
            "kind": "oracle",
            "sample": f"first {n} of {w.nnz} K and V rows of the contig workload, whole step, "
                      f"{dt:.1f} s"}


def cpu_baseline(w: W.Workload, target_s: float = 15.0):
    import oracle
    cores = oracle.max_threads()
    n = 1
    sub, nbytes = oracle_sample(w, n)
    dt = time_oracle(sub)
    while dt < target_s / 4 and n < w.B:
        n = min(w.B, max(n + 1, int(n * min(8.0, target_s / 2 / max(dt, 1e-3)))))
        sub, nbytes = oracle_sample(w, n)
        dt = time_oracle(sub)
    # the same oracle on one core, on a smaller sample (whole requests up to 4096 tokens)
    one, one_bytes = oracle_sample(w, 0, max_tokens=4096)
    dt1 = time_oracle(one, nthreads=1)
    n1 = int(one.seq_lens.astype(np.int64).sum())
    return {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"first {n} of {w.B} requests ({sub.nnz} tokens) of the {w.name} workload, "
                      f"whole step, {dt:.1f} s",
            "single_thread": {"value": one_bytes / dt1 / 1e9, "unit": "GB/s", "cores": 1,
                              "sample": f"first {n1} cached tokens ({one.B} requests), "
                                        f"whole step, {dt1:.1f} s"}}


def reference_arm(args, w: W.Workload):
    """The CPU oracle as the reference implementation: K timed steps (after W untimed) on a
    bounded sample of the same workload."""
    import oracle
    # size one step's sample so that all W + K steps take about two minutes
    per_step = 120.0 / max(1, args.steps + args.warmup)
    if args.workload == "contig":
        kv, _ = contig_sample(w, 8192)
        t1 = time_oracle_contig(kv, w.recipe)
        n_rows = int(max(64, min(w.nnz, 8192 * per_step / max(t1, 1e-4))))
        kv, nbytes = contig_sample(w, n_rows)
        timer = lambda: time_oracle_contig(kv, w.recipe)
        sample = f"first {kv[0].shape[0]} of {w.nnz} K and V rows"
        sample_cfg = {"workload": "contig", "sample_rows": kv[0].shape[0]}
    else:
        probe, _ = oracle_sample(w, 0, max_tokens=2048)
        t1 = time_oracle(probe)
        probe_tok = int(probe.seq_lens.astype(np.int64).sum())
        all_tok = int(w.seq_lens.astype(np.int64).sum())
        n_tok = int(max(16, min(all_tok, probe_tok * per_step / max(t1, 1e-4))))
        sub, nbytes = oracle_sample(w, 0, max_tokens=n_tok)
        timer = lambda: time_oracle(sub)
        n_s = int(sub.seq_lens.astype(np.int64).sum())
        sample = f"first {n_s} of {all_tok} cached tokens (first {sub.B} of {w.B} requests)"
        sample_cfg = {"workload": w.name, "sample_requests": sub.B, "sample_tokens": n_s}
    for _ in range(args.warmup):
        timer()
    times = [timer() for _ in range(args.steps)]
    dt = sum(times) / len(times)
    v = nbytes / dt / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": arith_dtype(w),
            "data": "synthetic", "config": sample_cfg,
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": oracle.max_threads(),
                             "kind": "oracle",
                             "sample": f"{sample}, whole step per timed step"},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="large_pool",
                    choices=["large_pool", "decode", "prefill", "materialize", "tiny", "contig"])
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--batch", type=int, default=256, help="large_pool: requests")
    ap.add_argument("--pool-gb", type=float, default=W.LARGE_POOL_BYTES / 1e9,
                    help="large_pool: pool size (K+V codes and scales), GB")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="large_pool: skip timing the other configurations afterwards")
    ap.add_argument("--v-scales", default="linear", choices=["linear", "interleaved4"],
                    help="layout of the V block scales the materialize reads (HND workloads)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    if args.impl == "reference":
        if rank == 0:
            w = make_workload(args.workload, torch.device("cuda", local) if torch.cuda.is_available()
                              else torch.device("cpu"), args.batch, args.pool_gb)
            reference_arm(args, w)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import nvfp4_paged_kv_02_gb300 as nv
    nv.load()
    w = make_workload(args.workload, dev, args.batch, args.pool_gb)
    step = ContigStep(w, dev) if args.workload == "contig" else Step(w, dev, args.v_scales)
    nbytes, ntok = step.op_bytes()
    n_ops = len(step.NAMES)
    total_bytes = sum(nbytes.values())
    small = max(nbytes.values()) < 1e9
    # L2 flush before every op of workloads whose ops are under 1 GB (so no op reads what the
    # one before it left in L2): write 256 MB, then read another 256 MB, so that the flush's
    # own dirty lines are written back before the op starts instead of competing with it
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if small else None
    flush_read = torch.zeros(256 << 20, dtype=torch.uint8, device=dev) if small else None

    for _ in range(args.warmup):
        step.run()
    torch.cuda.synchronize(dev)
    if int(step.status.item()) != 0:
        raise SystemExit(f"device status {int(step.status.item()):#x} after warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * n_ops)]
           for _ in range(args.steps)]

    flushes = [0]

    def flush_l2():
        flushes[0] += 1
        flush.fill_(flushes[0] & 0xFF)
        flush_read.sum()

    fd, clock_path = tempfile.mkstemp(prefix=f"nvfp4kv_clocks_rank{rank}_", suffix=".csv")
    os.close(fd)
    clocks = ClockSampler(clock_path)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    clocks.start()
    time.sleep(0.5)  # let the sampler come up before the timed region
    torch.cuda.synchronize(dev)
    step_ms = []
    h0 = time.time()
    for s in range(args.steps):
        step.run(evs[s], flush_l2 if flush is not None else None)
    torch.cuda.synchronize(dev)
    h1 = time.time()
    clk = clocks.stop(h0, h1)
    for s in range(args.steps):
        if flush is None:
            step_ms.append(evs[s][0].elapsed_time(evs[s][2 * n_ops - 1]))
        else:  # the device time of the ops, without the flushes between them
            step_ms.append(sum(evs[s][2 * i].elapsed_time(evs[s][2 * i + 1])
                               for i in range(n_ops)))
    ms = max_over_ranks(float(np.mean(step_ms)), dev)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    # per-op device time (mean over steps)
    seg = {k: (2 * i, 2 * i + 1) for i, k in enumerate(step.NAMES)}
    op_ms = {k: float(np.mean([evs[s][a].elapsed_time(evs[s][b]) for s in range(args.steps)]))
             for k, (a, b) in seg.items()}
    peak, peak_kind = measured_peaks()
    ops = {}
    for k in seg:
        gbs = nbytes[k] / (op_ms[k] * 1e-3) / 1e9
        ops[k] = {"us": op_ms[k] * 1e3, "bytes": nbytes[k], "GB_s": gbs,
                  "pct_of_8TBs": 100 * gbs / NOMINAL_HBM_GBS,
                  "pct_of_measured_copy": 100 * gbs / peak,
                  "tokens_per_s": ntok[k] / (op_ms[k] * 1e-3)}
    dom = max(step.NAMES[1:], key=lambda k: op_ms[k])
    value = world * total_bytes / (ms * 1e-3) / 1e9
    status = int(step.status.item())
    diag = step.diagnostics() if isinstance(step, Step) else None

    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(step, w, args, total_bytes, world)
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w) if isinstance(step, Step) else cpu_baseline_contig(w)
    configs = None
    if rank == 0 and args.workload == "large_pool" and not args.no_configs:
        cfg_main = step.config()
        launches = step.launches_per_step
        del step  # frees the pool and the outputs before the other workloads run
        torch.cuda.empty_cache()
        configs = measure_configs(w, dev)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": arith_dtype(w),
            "data": "synthetic",
            "config": {**(cfg_main if configs is not None else step.config()),
                       "l2": "flushed before every op (256 MB write, then 256 MB read), "
                             "outside the timed ops" if small
                       else "inputs larger than L2 (129 MB); no flush",
                       "parallelism": f"replicas x{world}"},
            "ops": ops,
            "roofline": {"bound": "hbm", "kernel": dom,
                         "achieved": nbytes[dom] / (op_ms[dom] * 1e-3) / 1e9,
                         "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                         "frac": nbytes[dom] / (op_ms[dom] * 1e-3) / 1e9 / peak,
                         "traffic": traffic_per_launch(dom, ntok[dom])},
            "clocks": clk,
            "gpu_launches": (launches if configs is not None else step.launches_per_step)
            * args.steps,
            "e2e": e2e, "cpu_baseline": cpu, "device_status": status,
            "diagnostics": diag,
            "configs": configs,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def measure_e2e(step, w: W.Workload, args, total_bytes: int, world: int):
    """The same step through the public API with the appended K/V rows in pinned host
    memory: every step copies its rows to the device, runs the path and reads back the
    step's summary (the two global scales and the device status word). Steps are pipelined
    the way a serving loop would run them: the copies of step i+1 (on a copy stream, into
    the other of two device input buffers) overlap the compute of step i; a buffer is
    refilled only after the step that read it has finished.

    The paged cache, the dequantized K/V and the FP8 copy stay on the device, as a serving
    loop keeps them. A second figure also reads the dequantized rows of every request back
    to pinned host memory each step (on a third stream; the next step's compute waits until
    that read is done, since it rewrites the same outputs)."""
    dev = step.dev
    comp = torch.cuda.current_stream(dev)
    copy = torch.cuda.Stream(dev)
    back = torch.cuda.Stream(dev)
    hk = torch.empty(step.k.shape, dtype=step.k.dtype, pin_memory=True)
    hv = torch.empty(step.v.shape, dtype=step.v.dtype, pin_memory=True)
    hk.copy_(step.k)
    hv.copy_(step.v)
    bufs = [(step.k, step.v), (torch.empty_like(step.k), torch.empty_like(step.v))]
    res = [torch.empty(3, dtype=torch.float32, pin_memory=True) for _ in range(2)]
    summary = [torch.empty(3, dtype=torch.float32, device=dev) for _ in range(2)]
    copied = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    read_done = torch.cuda.Event()
    for e in done:
        e.record(comp)
    read_done.record(comp)
    # the dequantized output to read back: every request's rows (paged form), or the two
    # [rows, cols] outputs (contiguous form); (device view, pinned host view) pairs
    readback = []

    def one(i, read_back=False):
        b = i % 2
        k, v = bufs[b]
        with torch.cuda.stream(copy):
            copy.wait_event(done[b])  # the step that last read this buffer has finished
            k.copy_(hk, non_blocking=True)
            v.copy_(hv, non_blocking=True)
            copied[b].record(copy)
        comp.wait_event(copied[b])
        if read_back:
            comp.wait_event(read_done)  # the previous step's outputs have been read back
        step.k, step.v = k, v
        step.run()
        sm = summary[b]
        sm[0] = step.gk[0]
        sm[1] = step.gv[0]
        sm[2] = step.status[0].float()
        res[b].copy_(sm, non_blocking=True)
        done[b].record(comp)
        if read_back:
            back.wait_stream(comp)
            with torch.cuda.stream(back):
                for src, dst in readback:
                    dst.copy_(src, non_blocking=True)
                read_done.record(back)

    def windows(read_back=False):
        for i in range(2):
            one(i, read_back)
        torch.cuda.synchronize(dev)
        a = torch.cuda.Event(enable_timing=True)
        z = torch.cuda.Event(enable_timing=True)
        # five timed windows of n steps; the median window is reported (the host link is
        # shared with the rest of the machine: a window that lands on a burst of other
        # traffic runs up to 1.5x longer, while the quiet ones sit at the link's 211 GB/s)
        n = max(4, min(args.steps, 6))
        out = []
        for _ in range(5):
            a.record(comp)
            copy.wait_stream(comp)  # the timed copies start after the start event
            for i in range(n):
                one(i, read_back)
            comp.wait_stream(copy)
            comp.wait_stream(back)
            z.record(comp)
            torch.cuda.synchronize(dev)
            out.append(a.elapsed_time(z) / n)
        return out

    fd, clock_path = tempfile.mkstemp(prefix="nvfp4kv_clocks_e2e_", suffix=".csv")
    os.close(fd)
    clocks = ClockSampler(clock_path)
    clocks.start()
    time.sleep(0.3)
    h0 = time.time()
    wins = windows()
    h1 = time.time()
    clk = clocks.stop(h0, h1)
    ms = max_over_ranks(float(np.median(wins)), dev)
    h2d = hk.numel() * hk.element_size() + hv.numel() * hv.element_size()
    # the host link alone: one copy of the K rows, for reading the e2e figure against
    a = torch.cuda.Event(enable_timing=True)
    z = torch.cuda.Event(enable_timing=True)
    a.record(comp)
    bufs[1][0].copy_(hk, non_blocking=True)
    z.record(comp)
    torch.cuda.synchronize(dev)
    link = hk.numel() * hk.element_size() / (a.elapsed_time(z) * 1e-3) / 1e9

    if isinstance(step, ContigStep):
        for o in step.out:
            readback.append((o, torch.empty(o.shape, dtype=o.dtype, pin_memory=True)))
    else:
        lens = np.minimum(w.seq_lens.astype(np.int64), w.max_seq_len)
        host = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
                for o in (step.out_k, step.out_v)]
        for r, n in enumerate(lens):
            if n > 0:
                readback.append((step.out_k[r, :n], host[0][r, :n]))
                readback.append((step.out_v[r, :n], host[1][r, :n]))
    wins_rb = windows(read_back=True)
    ms_rb = max_over_ranks(float(np.median(wins_rb)), dev)
    d2h_rb = sum(src.numel() * src.element_size() for src, _ in readback) + 12
    step.k, step.v = bufs[0]
    return {"value": world * total_bytes / (ms * 1e-3) / 1e9, "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": 12, "ms_per_step": ms,
            "value_counts": "appended K/V rows copied in, the step's summary (two global "
                            "scales and the status word) read back",
            "resident_on_device": (["NVFP4 codes and block scales of K and V",
                                    "dequantized K and V"] if isinstance(step, ContigStep)
                                   else ["paged K/V cache (codes and block scales)",
                                         "dequantized K/V (out_k, out_v)",
                                         "FP8 copy and fp8_block_tables"]),
            "pipelined": "copies of step i+1 overlap the compute of step i (two buffers)",
            "windows_ms_per_step": wins, "host_to_device_gbs": link, "clocks": clk,
            "with_dequant_readback": {
                "value": world * total_bytes / (ms_rb * 1e-3) / 1e9, "unit": "GB/s",
                "ms_per_step": ms_rb, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h_rb,
                "reads_back": ("both dequantized [rows, cols] outputs and the summary"
                               if isinstance(step, ContigStep) else
                               "every request's dequantized K and V rows (rows < seq_lens) and "
                               "the summary"),
                "windows_ms_per_step": wins_rb}}


if __name__ == "__main__":
    main()
