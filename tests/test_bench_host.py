"""The bench's host-side bookkeeping (no GPU): batch overrides rename the
workload, and DRAM traffic from a committed ncu record is reported only for
the workload and kernel source it was taken on."""
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
    src.write_bytes(src.read_bytes() + b"\n// changed\n")
    assert bench.ncu_traffic(key, sources, "causal_bf16_b4_h16_s8192_d128") is None  # stale source
