"""Host logic of bench.py that needs no GPU: the recorded row-pass DRAM
traffic is reported only for the kernel source it was taken on and for rows
of the recorded length, and it scales with the rows of a launch."""

import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _write(tmp_path, **over):
    with open(bench.PROFILE_TRAFFIC) as f:
        d = json.load(f)
    d.update(over)
    p = tmp_path / "traffic.json"
    p.write_text(json.dumps(d))
    return str(p), d


def test_traffic_scales_with_rows(tmp_path, monkeypatch):
    p, d = _write(tmp_path, kernel_hash=bench.kernel_hash())
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", p)
    per_row = (d["dram_bytes_read_measured"] + d["dram_bytes_write_measured"]) / d["rows_measured"]
    assert bench.recorded_traffic(d["rows_measured"], d["vocab"]) == per_row * d["rows_measured"]
    assert bench.recorded_traffic(3 * d["rows_measured"], d["vocab"]) == 3 * per_row * d["rows_measured"]


def test_traffic_withheld_for_another_kernel_or_row_length(tmp_path, monkeypatch):
    p, d = _write(tmp_path, kernel_hash="0" * 16)
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", p)
    assert bench.recorded_traffic(100, d["vocab"]) is None
    p, d = _write(tmp_path, kernel_hash=bench.kernel_hash())
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", p)
    assert bench.recorded_traffic(100, d["vocab"] + 1) is None
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", str(tmp_path / "missing.json"))
    assert bench.recorded_traffic(100, d["vocab"]) is None

