"""CPU checks of bench.py's host logic: the bytes a step counts, the keys of the
committed ncu traffic figures and when they are reported, the CPU baseline's
fields, and the reference arm's JSON line (the oracle timed on the host cores).
No GPU is used."""
import argparse
import contextlib
import io
import json

import pytest

import bench
from memory_bound_row_gb300 import workloads as W


def test_algorithmic_bytes_per_step():
    # M x N x (in + out element size); row padding is not counted; the
    # normalisations add their weight (and bias) vectors once per launch.
    w = W.WORKLOADS["fp32_8192x5000_ld5120"]
    assert bench.op_bytes("softmax", w) == 8192 * 5000 * (4 + 4)
    n = bench.op_workload("rmsnorm", "bf16_32768x8192")
    assert bench.op_bytes("rmsnorm", n) == 32768 * 8192 * (2 + 2) + 8192 * 2
    assert bench.op_bytes("layernorm", n) == 32768 * 8192 * (2 + 2) + 2 * 8192 * 2


def test_traffic_keys():
    assert bench.traffic_key("softmax", "fp16_512x131072") == "fp16_512x131072"
    assert bench.traffic_key("softmax", "bf16_causal_16x32x2048", True) == "causal:bf16_causal_16x32x2048"
    assert bench.traffic_key("layernorm", "bf16_32768x8192") == "layernorm:bf16_32768x8192"
    assert bench.traffic_key("rmsnorm", "fp16_512x131072", True) == "rmsnorm:fp16_512x131072"


def test_committed_traffic_is_reported_only_for_the_sources_it_was_taken_on(monkeypatch):
    with open(bench.TRAFFIC_FILE) as f:
        data = json.load(f)
    entries = {k: v for k, v in data.items() if not k.startswith("_")}
    assert entries
    for key, ent in entries.items():
        # per-launch DRAM bytes of a full launch: no more than the algorithmic
        # bytes plus a few percent (no re-reads), and at least the reads
        assert 0 < ent["dram_bytes_read"] <= ent["dram_bytes_per_launch"], key
        assert ent["dram_bytes_per_launch"] <= 1.05 * ent["algorithmic_bytes"], key
        assert "ncu" in ent["command"] and "--clock-control none" in ent["command"], key
    key, ent = next(iter(entries.items()))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: ent["kernel_source_hash"])
    assert bench.ncu_traffic(key) == ent["dram_bytes_per_launch"]
    assert bench.ncu_traffic("no such workload") is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "not the captured sources")
    assert bench.ncu_traffic(key) is None


def test_cpu_baseline_reports_the_oracle_on_a_bounded_sample():
    w = W.custom(64, 1000, "f32", seed=3)
    x = W.generate(w, "cpu")
    b = bench.cpu_baseline(w, x, "softmax", seconds=0.3)
    assert b["kind"] == "oracle" and b["unit"] == "GB/s" and b["value"] > 0 and b["cores"] >= 1
    assert "rows" in b["sample"] and b["single_thread"]["value"] > 0
    wn = W.custom(16, 512, "bf16", seed=4)
    bn = bench.cpu_baseline(wn, W.generate(wn, "cpu"), "layernorm", seconds=0.2)
    assert bn["value"] > 0 and "layernorm" in bn["sample"]


@pytest.mark.parametrize("op", ["softmax", "rmsnorm"])
def test_reference_arm_prints_one_json_line_with_the_contract_keys(op):
    args = argparse.Namespace(op=op, steps=2, warmup=1, gpus=1)
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(args, ["fp32_1024x1024"])
    lines = [json.loads(s) for s in buf.getvalue().splitlines() if s.strip()]
    assert len(lines) == 1
    d = lines[0]
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["metric"] == bench.OP_METRIC[op] and d["unit"] == "GB/s"
    assert d["value"] > 0 and d["higher_is_better"] is True and d["vs_baseline"] is None
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] == "fp32_1024x1024"


def test_graph_size_gives_long_kernels_several_replays():
    # K = 20 (the driver's run): a 1.4 ms launch is replayed alone 20 times,
    # a 0.17 ms launch in graphs of 5, a 50 us launch in one graph of 20.
    assert bench.pick_graph_launches(20, 1, 1.37) == 1
    assert bench.pick_graph_launches(20, 1, 0.171) == 5
    assert bench.pick_graph_launches(20, 2, 0.05) == 20
    assert bench.pick_graph_launches(2000, 2, 0.003) == 50
    # a multiple of the rotating buffer sets where one fits
    assert bench.pick_graph_launches(24, 4, 0.05) == 12
    for k in (1, 3, 7, 20, 400):
        g = bench.pick_graph_launches(k, 3, 0.2)
        assert k % g == 0 and 1 <= g <= 64


def test_default_workload_is_the_largest():
    sizes = {n: W.WORKLOADS[n].algorithmic_bytes for n in W.ORDER}
    assert bench.DEFAULT_WORKLOAD == max(sizes, key=sizes.get) == "bf16_causal_16x32x2048"
