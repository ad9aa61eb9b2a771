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


def _args(**kw):
    import argparse
    ns = dict(prefill_tokens=4096, no_varlen=False, no_single=False, varlen_max=8192)
    ns.update(kw)
    return argparse.Namespace(**ns)


def test_prefill_cases_default_and_small_varlen():
    """The default cases are the two the bench line reports; --no-single and --varlen-max
    select the small varlen case the prefill profile is captured on."""
    names = [n for n, _ in bench.prefill_cases(_args())]
    assert names == ["single_4096_bypass", "varlen_8seq_conv"]
    cases = bench.prefill_cases(_args(no_single=True, varlen_max=2048))
    assert [n for n, _ in cases] == ["varlen_8seq_conv_max2048"]
    inp = cases[0][1]()
    lens = inp.cu_seqlens[1:] - inp.cu_seqlens[:-1]
    assert lens.size == 8 and lens.max() <= 2048 and inp.conv_w is not None
    assert bench.prefill_cases(_args(no_single=True, no_varlen=True)) == []
