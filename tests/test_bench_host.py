"""Host logic of bench.py (no GPU): the algorithmic byte model behind every
roofline fraction, and the lookup of committed ncu traffic.

The byte model is pinned to sizes worked out by hand from the Qwen2.5-shaped
pair's shapes: the draft streams 988 MB per forward (24 layers of 14.9 M
parameters plus a 151936 x 896 head, bf16) and the base 14.14 GB per verify
(28 layers of 233 M parameters plus a 151936 x 3584 head); K/V per cached
position and token is 12.3 KB (draft) and 57.3 KB (base).
"""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from layer_drafting_draft_b300 import synth  # noqa: E402

QWEN = synth.WORKLOADS["qwen2.5_0.5b_7b_bf16"]


def test_weight_stream_bytes_of_the_qwen_pair():
    pb = bench.phase_bytes(QWEN, 4, 0, 1)
    assert pb["draft_fwd"] == pytest.approx(988.0e6, rel=2e-3)
    # context 0: verify = base weights + 5 embedding rows + the 5 rows' K/V writes
    kv_writes = 5 * 57344
    assert pb["verify"] - kv_writes - 5 * 3584 * 2 == pytest.approx(14.14e9, rel=2e-3)
    assert pb["draft"] == pytest.approx(4 * pb["draft_fwd"] + 8 * 12288, rel=1e-12)
    assert pb["fuzzy"] == pytest.approx(3 * pb["draft_fwd"] + 3 * 12288, rel=1e-12)


def test_kv_bytes_per_position():
    assert bench.kv_bytes(QWEN["draft"], 2, 1, 1) == 2 * 12288
    assert bench.kv_bytes(QWEN["base"], 2, 1, 1) == 2 * 57344
    # B sequences: weights once, K/V and embedding rows per sequence
    one, four = bench.phase_bytes(QWEN, 4, 4096, 1), bench.phase_bytes(QWEN, 4, 4096, 4)
    w = bench.phase_bytes(QWEN, 4, 0, 1)["verify"] - 5 * 57344 - 5 * 7168
    assert four["verify"] - w == pytest.approx(4 * (one["verify"] - w), rel=1e-12)


def test_traffic_only_for_the_captured_workload_and_rows():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        t = json.load(f)
    for name in ("base.gv_gateup", "base.tc_gateup"):
        for e in t[name]:
            got = bench.measured_traffic(name, e["workload"], e["rows"])
            assert got in (e["dram_bytes_per_launch"], None)   # None once the kernel sources change
            assert bench.measured_traffic(name, e["workload"], e["rows"] + 1) is None
            assert bench.measured_traffic(name, "qwen2.5_longctx_bf16", e["rows"]) is None
    e = t["base.tc_gateup"][0]
    assert bench.measured_traffic("no.such_pass", e["workload"], e["rows"]) is None
    # two workloads of one pass keep their own figures
    by = {e["workload"]: e["dram_bytes_per_launch"] for e in t["base.tc_gateup"]}
    assert bench.measured_traffic("base.tc_gateup", "llama3_8b_70b_bf16", 5) == by["llama3_8b_70b_bf16"]
    assert bench.measured_traffic("base.tc_gateup", "qwen2.5_0.5b_7b_bf16", 5) == by["qwen2.5_0.5b_7b_bf16"]
