"""bench.py end to end on the GPU, in a child process: the code paths of the default run
(the large-pool step, the other configurations, e2e with and without the readback, the CPU
baseline) on a 16-request, 2 GB pool, the contiguous workload, and the reference arm. Each
must exit 0 and print one JSON line with the keys of the measurement contract."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SMALL = ["--batch", "16", "--pool-gb", "2", "--steps", "3", "--warmup", "3"]


@pytest.fixture(scope="module", autouse=True)
def _cuda(gpu_lib):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    yield


def _run(args, timeout=900):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                       capture_output=True, text=True, timeout=timeout)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, r.stdout[-3000:]
    return json.loads(lines[0])


def _check_e2e(e, readback_key):
    assert e["value"] > 0 and e["unit"] == "GB/s"
    assert e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] == 12
    assert e["resident_on_device"] and len(e["windows_ms_per_step"]) == 5
    rb = e[readback_key]
    assert rb["value"] > 0 and rb["d2h_bytes_per_step"] > e["d2h_bytes_per_step"]


def test_default_run_paths_on_a_small_pool():
    d = _run(SMALL)
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "cpu_baseline", "e2e", "clocks", "gpu_launches", "configs"):
        assert key in d, key
    assert d["value"] > 0 and d["n_gpus"] == 1 and d["device_status"] == 0
    assert d["config"]["workload"] == "large_pool" and d["gpu_launches"] > 0
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["peak"] > 0 and 0 < rf["frac"] < 2
    assert set(d["ops"]) == {"global_scale", "append", "dequant_paged", "materialize"}
    _check_e2e(d["e2e"], "with_dequant_readback")
    cpu = d["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["value"] > 0 and cpu["cores"] >= 1 and cpu["sample"]
    assert set(d["configs"]) == {"decode", "prefill", "materialize", "materialize_v_interleaved4",
                                 "contig"}
    for name, cfg in d["configs"].items():
        assert cfg["device_status"] == 0, name
        assert all(op["us"] > 0 for op in cfg["ops"].values()), name
    assert d["configs"]["materialize_v_interleaved4"]["config"]["materialize_v_scales"] == "interleaved4"
    assert d["configs"]["materialize"]["host_cost"]["c_abi_run_us"] > 0


def test_contiguous_workload():
    d = _run(["--workload", "contig", *SMALL, "--no-cpu-baseline"])
    assert set(d["ops"]) == {"global_scale", "kv_quantize", "kv_dequantize"}
    assert d["device_status"] == 0 and d["configs"] is None
    _check_e2e(d["e2e"], "with_dequant_readback")


def test_reference_arm():
    d = _run(["--impl", "reference", "--steps", "1", "--warmup", "1"])
    assert d["impl"] == "reference" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
