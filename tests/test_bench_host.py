"""Host logic of bench.py that needs no GPU: the DRAM-traffic model behind
`roofline.traffic` (reported only while a kernel's sources hash to the captured ones) and
the arithmetic of the committed traffic tables."""
import os
import re

import pytest

import bench

PROFILES = os.path.join(bench.ROOT, "profiles")
TABLES = ["dram_traffic_large_pool.md", "dram_traffic_contig.md"]
HEADER = ("| op | source sha256 (16 hex) | units (small) | DRAM read (small) | DRAM write (small) "
          "| units (large) | DRAM read (large) | DRAM write (large) | marginal bytes per unit "
          "| bytes at zero units | algorithmic bytes per unit | kernel |")


def _write_table(path, op, digest, small, large, alg=5248):
    (u1, r1, w1), (u2, r2, w2) = small, large
    slope = ((r2 + w2) - (r1 + w1)) / (u2 - u1)
    icpt = (r1 + w1) - slope * u1
    with open(path, "w") as f:
        f.write(HEADER + "\n|" + "---|" * 12 + "\n")
        f.write(f"| {op} | {digest} | {u1} | {r1} | {w1} | {u2} | {r2} | {w2} | {slope:.1f} "
                f"| {icpt:.0f} | {alg} | `k` |\n")


def test_traffic_follows_the_two_size_fit_when_the_sources_match(tmp_path, monkeypatch):
    path = tmp_path / "traffic.md"
    _write_table(path, "append", bench.source_hash("append"), (100, 400000, 90000),
                 (300, 1200000, 290000))
    monkeypatch.setattr(bench, "TRAFFIC_FILES", [str(path)])
    # 5000 B per unit beyond the first, minus 10 kB left in L2 at the end of a launch
    assert bench.traffic_per_launch("append", 1000) == pytest.approx(5000.0 * 1000 - 10000)


def test_traffic_is_null_after_a_source_change(tmp_path, monkeypatch):
    path = tmp_path / "traffic.md"
    _write_table(path, "append", "0" * 16, (100, 400000, 90000), (300, 1200000, 290000))
    monkeypatch.setattr(bench, "TRAFFIC_FILES", [str(path)])
    assert bench.traffic_per_launch("append", 1000) is None
    monkeypatch.setattr(bench, "TRAFFIC_FILES", [str(tmp_path / "missing.md")])
    assert bench.traffic_per_launch("append", 1000) is None


def test_source_hash_covers_the_kernel_and_shared_headers():
    h = bench.source_hash("append")
    assert re.fullmatch(r"[0-9a-f]{16}", h)
    assert h == bench.source_hash("kv_quantize")  # the same translation unit
    assert h != bench.source_hash("dequant_paged")


@pytest.mark.parametrize("name", TABLES)
def test_committed_traffic_rows_add_up(name):
    rows = []
    with open(os.path.join(PROFILES, name)) as f:
        for ln in f:
            cells = [c.strip().strip("`") for c in ln.strip().strip("|").split("|")]
            if len(cells) == 12 and cells[0] in bench.KERNEL_SOURCES:
                rows.append(cells)
    assert rows
    for op, digest, u1, r1, w1, u2, r2, w2, slope, icpt, alg, _ in rows:
        assert re.fullmatch(r"[0-9a-f]{16}", digest)
        u1, r1, w1, u2, r2, w2, alg = map(int, (u1, r1, w1, u2, r2, w2, alg))
        slope, icpt = float(slope), float(icpt)
        assert slope == pytest.approx(((r2 + w2) - (r1 + w1)) / (u2 - u1), abs=0.05)
        # (the slope is printed to 0.1 B, the intercept from the unrounded slope)
        assert icpt == pytest.approx((r1 + w1) - slope * u1, abs=0.05 * u1 + 1.0)
        # reads scale with the units (bytes per unit equal at both sizes, within 0.5 %)
        assert r1 / u1 == pytest.approx(r2 / u2, rel=5e-3)
        # each further unit costs its algorithmic bytes (no re-reads), within 1 %
        assert slope == pytest.approx(alg, rel=0.01)
        # what is missing at zero units is output still dirty in L2 (129 MB) at the end
        assert -2 * 129e6 <= icpt <= 0
