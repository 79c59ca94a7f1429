"""The bench's DRAM-traffic figure (`roofline.traffic`): it comes from the ncu
capture recorded in profiles/traffic.json only while the captured kernel's
sources are unchanged, and it is never below the kernel's algorithmic bytes
(every input read once, every output written once)."""
import json
import os

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _records():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        return json.load(f)


@pytest.mark.parametrize("row", sorted(bench.TRAFFIC_KERNEL))
def test_a_record_exists_for_every_row_with_a_traffic_kernel(row):
    key = f"{bench.TRAFFIC_KERNEL[row]}@{bench.STEP_WORKLOAD.name}"
    rec = _records()[key]
    assert rec["dram_bytes_per_launch"] > 0
    assert len(rec["source_sha256"]) == 64
    assert "--clock-control none" in rec["capture"]


@pytest.mark.parametrize("row", sorted(bench.TRAFFIC_KERNEL))
def test_traffic_is_dropped_once_the_sources_change(row, monkeypatch):
    rec = _records()[f"{bench.TRAFFIC_KERNEL[row]}@{bench.STEP_WORKLOAD.name}"]
    monkeypatch.setattr(bench, "kernel_source_hash", lambda kernel: rec["source_sha256"])
    got, note = bench.dram_traffic(row)
    assert got == rec["dram_bytes_per_launch"] and note == rec["capture"]
    monkeypatch.setattr(bench, "kernel_source_hash", lambda kernel: "0" * 64)
    got, note = bench.dram_traffic(row)
    assert got is None and "changed" in note


def test_recorded_traffic_is_at_least_the_algorithmic_bytes():
    """Forward: Q, K, V read and O written in bf16, LSE in fp32.  Backward:
    Q, K, V, dO read (bf16) with LSE and D (fp32), dK and dV written (bf16),
    and the fp32 dQ accumulator written once (its reduce-adds land in L2)."""
    w = bench.STEP_WORKLOAD
    t = w.B * w.H * w.L * w.d
    rows = w.B * w.H * w.L
    algo = {"fwd": 4 * t * 2 + rows * 4,
            "bwd": 4 * t * 2 + 2 * rows * 4 + 2 * t * 2 + t * 4}
    recs = _records()
    for row, kernel in bench.TRAFFIC_KERNEL.items():
        got = recs[f"{kernel}@{w.name}"]["dram_bytes_per_launch"]
        assert got >= algo[row], (row, got, algo[row])
