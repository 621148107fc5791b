"""The bench's host-side bookkeeping (no GPU): batch overrides rename the
workload, and DRAM traffic from a committed ncu record is reported only for
the workload and kernel code it was taken on (comments aside)."""
import json
import os

import bench


def test_with_batch_renames_and_keeps_the_rest():
    w = bench.with_batch(bench.PREFILL, 1)
    assert w.B == 1 and w.name == bench.PREFILL.name.replace("_b4_", "_b1_", 1)
    assert (w.H, w.Sq, w.d, w.causal, w.seed) == (bench.PREFILL.H, bench.PREFILL.Sq, bench.PREFILL.d,
                                                   bench.PREFILL.causal, bench.PREFILL.seed)
    d = bench.with_batch(bench.DECODE, 8)
    assert d.B == 8 and "_b8_" in d.name and "_b64_" not in d.name


def test_traffic_record_needs_matching_workload_and_source(tmp_path, monkeypatch):
    sources = ["exact_tiled_attention_gb300/csrc/prefill_fwd.cu"]
    src = tmp_path / sources[0]
    src.parent.mkdir(parents=True)
    src.write_bytes(open(os.path.join(os.path.dirname(os.path.abspath(bench.__file__)), sources[0]), "rb").read())
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    key = "k<128>"
    rec = {key: {"dram_bytes_per_launch": 123, "workload": "causal_bf16_b4_h16_s8192_d128 (full size)",
                 "source_sha": bench.kernel_source_hash(sources)}}
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "ncu_traffic.json").write_text(json.dumps(rec))
    assert bench.ncu_traffic(key, sources, "causal_bf16_b4_h16_s8192_d128") == 123
    assert bench.ncu_traffic(key, sources, "causal_bf16_b1_h16_s8192_d128") is None  # another batch
    assert bench.ncu_traffic("other", sources, "causal_bf16_b4_h16_s8192_d128") is None
    original = src.read_bytes()
    src.write_bytes(original + b"\n// a comment\n/* and a block\n comment */\n")
    assert bench.ncu_traffic(key, sources, "causal_bf16_b4_h16_s8192_d128") == 123  # comments only
    src.write_bytes(original + b"\nstatic int changed = 1;\n")
    assert bench.ncu_traffic(key, sources, "causal_bf16_b4_h16_s8192_d128") is None  # stale source


def test_host_info_names_cpu_and_versions():
    h = bench.host_info()
    assert h["cpu_model"] and h["cpu_model"] != ""
    assert h["host_cores"] >= 1 and h["torch"] == bench.torch.__version__


def test_cpu_oracle_backward_on_tiny_workload():
    val, cores, sample = bench.cpu_oracle_backward(bench.WORKLOADS["tiny_fwd_fp16"])
    assert val > 0 and cores >= 1 and "KV head 0" in sample


def test_leg_roofline_row_keeps_the_figures():
    leg = {"workload": "w", "ms_per_call": 1.5, "cpu_baseline": {"value": 0.01},
           "roofline": {"bound": "tensor", "achieved": 10.0, "peak": 20.0, "unit": "TFLOP/s", "frac": 0.5,
                        "traffic": None}}
    row = bench.leg_roofline(leg, "k")
    assert row == {"workload": "w", "kernel": "k", "bound": "tensor", "achieved": 10.0, "peak": 20.0,
                   "unit": "TFLOP/s", "frac": 0.5, "traffic": None, "ms": 1.5, "cpu_baseline": 0.01}
