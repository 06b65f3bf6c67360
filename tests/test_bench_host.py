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



def test_workload_names_follow_the_config():
    """Each config's line names its own workload (sizes, dtype, filter)."""
    assert "B=256 k=15 V=151936 bf16" in bench.workload_desc("c4", "default")
    assert "top-k 50 + top-p 0.9" in bench.workload_desc("c4", "default")
    assert "top-p 0.9 alone" in bench.workload_desc("c4p", "default")
    assert "B=1 k=4 V=1024 fp32" in bench.workload_desc("c1", "t1")
    assert "greedy" in bench.workload_desc("c2", "greedy")
    assert "N(0,2.0^2)" in bench.workload_desc("c3", "s2")
    assert "ragged" in bench.workload_desc("c5", "default")
    assert "B=64" in bench.workload_desc("c4", "default", batch=64)


def test_required_bytes_skip_greedy_draft_rows():
    """Greedy requests read their target rows only; sampled ones every row."""
    from speculative_decoding_verification_13_gb300 import workloads
    b = workloads.make_batch_from_params("t", [3, 2, 4], [1.0, 0.0, 0.5], [1.0] * 3, 64,
                                         bench_dtype(), 5)
    nbytes, rows = bench.required_bytes(b)
    assert rows == (4 + 3 + 5) + (3 + 4)
    assert nbytes == rows * 64 * 4


def test_unfiltered_workloads_pass_no_filter_arrays():
    """Configs without a filter call the library with top_k = top_p = None
    (one launch fewer); filtered ones pass their arrays."""
    from speculative_decoding_verification_13_gb300 import workloads
    b = workloads.make_batch("c1", "t1")
    assert b.filters() == (None, None)
    assert int(b.top_k.abs().sum()) == 0 and bool((b.top_p == 1).all())
    f = workloads.make_batch("c4", batch=2).filters()
    assert f[0] is not None and f[1] is not None


def bench_dtype():
    import torch
    return torch.float32
