"""Host logic of bench.py that needs no GPU: the DRAM-traffic lookup behind
`roofline.traffic` (reported only while a kernel's sources hash to the captured ones) and
the arithmetic of the committed traffic tables."""
import os
import re

import pytest

import bench

PROFILES = os.path.join(bench.ROOT, "profiles")
TABLES = ["dram_traffic_large_pool.md", "dram_traffic_contig.md"]


def _write_table(path, op, digest, units, rd, wr):
    with open(path, "w") as f:
        f.write("| op | source sha256 (16 hex) | units in capture | DRAM read (B) | DRAM write (B) "
                "| bytes per unit (read + write) | algorithmic bytes per unit | kernel |\n")
        f.write("|---|---|---|---|---|---|---|---|\n")
        f.write(f"| {op} | {digest} | {units} | {rd} | {wr} | {(rd + wr) / units:.1f} | 5248 | `k` |\n")


def test_traffic_scales_with_units_when_the_sources_match(tmp_path, monkeypatch):
    path = tmp_path / "traffic.md"
    _write_table(path, "append", bench.source_hash("append"), 100, 400000, 100000)
    monkeypatch.setattr(bench, "TRAFFIC_FILES", [str(path)])
    assert bench.traffic_per_launch("append", 1000) == pytest.approx(5000.0 * 1000)


def test_traffic_is_null_after_a_source_change(tmp_path, monkeypatch):
    path = tmp_path / "traffic.md"
    _write_table(path, "append", "0" * 16, 100, 400000, 100000)
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
            if len(cells) == 8 and cells[0] in bench.KERNEL_SOURCES:
                rows.append(cells)
    assert rows
    for op, digest, units, rd, wr, per_unit, alg, _ in rows:
        assert re.fullmatch(r"[0-9a-f]{16}", digest)
        units, rd, wr, per_unit, alg = int(units), int(rd), int(wr), float(per_unit), int(alg)
        assert per_unit == pytest.approx((rd + wr) / units, abs=0.05)
        # no kernel moves more DRAM bytes than its algorithmic bytes (no re-reads)
        assert per_unit <= alg
