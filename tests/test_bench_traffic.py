"""The roofline's `traffic` figure comes from the committed ncu summary only when that
summary was taken on the current decode source and on the workload the line reports."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _summary():
    with open(os.path.join(ROOT, "profiles", "decode_traffic.json")) as f:
        return json.load(f)


def test_summary_names_its_workload():
    j = _summary()
    for state in ("f32", "bf16"):
        e = j["launches"][state]
        assert e["batch"] == bench.HEADLINE_B and e["num_slots"] == bench.NUM_SLOTS
        assert e["dram_bytes_per_launch"] == (e["measured_dram_read_bytes"]
                                              + e["measured_dram_write_bytes"])


@pytest.mark.parametrize("state", ["f32", "bf16"])
def test_traffic_only_for_the_captured_workload(state):
    e = _summary()["launches"][state]
    if _summary()["source_digest"] != bench.kernel_source_digest():
        assert bench.ncu_traffic(state, e["batch"], e["num_slots"]) is None
        return
    assert bench.ncu_traffic(state, e["batch"], e["num_slots"]) == e
    assert bench.ncu_traffic(state, 1, 2) is None
    assert bench.ncu_traffic(state, e["batch"], 2 * e["num_slots"]) is None
