"""Benchmark of the exact-attention hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gbattn|reference]
                    [--workload prefill|decode]

Default workload ("prefill"): the causal bf16 prefill forward, q/k/v
[4, 16, 8192, 128], reported as attention TFLOP/s (4*B*H*Sq*Sk*d, halved for
causal) against the measured dense bf16 tensor peak.  The split-KV decode
workload (64 sequences x 32 query / 8 KV heads, 32768-slot bf16 cache, valid
lengths uniform on [1024, 32768], 16 chunks) is measured in the same run and
reported under "decode" (HBM GB/s of algorithmic bytes against the measured
copy bandwidth); `--workload decode` makes it the headline instead.

One step = one call of the hot path over one batch of resident synthetic
input.  W warm-up steps, then exactly K steps timed with CUDA events on the
launching stream, bracketed by a barrier and a device synchronize; the
inputs (>= 512 MiB per step) exceed the 129 MB L2, so no flush is needed.
Under torchrun every rank runs its own independent copy of the workload
(weak scaling, no data-path collective); rank 0 prints one JSON line with the
whole-job throughput (work of all ranks / max time over ranks).

--impl reference times the fp64 CPU oracle on the host cores on a bounded
sample of the same workload (the baseline, not the target).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from exact_tiled_attention_gb300.inputs import WORKLOADS, make_workload  # noqa: E402

PREFILL = WORKLOADS["causal_bf16_b4_h16_s8192_d128"]
DECODE = WORKLOADS["decode_splitkv_bf16_b64_hq32_hkv8_sk32768_d128"]
# The other forward workloads, measured in the default run under "prefill_other"
# (the tiny one is a parity case only: a few microseconds per launch).
OTHER_PREFILL = [WORKLOADS["prefill_fp16_b1_h8_s4096_d64"],
                 WORKLOADS["gqa_causal_bf16_b2_hq32_hkv8_s4096_d128"],
                 WORKLOADS["noncausal_bf16_b4_h16_s8192_d128"]]
# The CTA-pair forward (attn_fwd_pair: non-causal, d = 128), measured in the
# default run under "cta_pair" on the non-causal workload above.
PAIR = WORKLOADS["noncausal_bf16_b4_h16_s8192_d128"]
# Backward workloads (d = 128), measured in the default run under "backward".
BACKWARD = [WORKLOADS["causal_bf16_b4_h16_s8192_d128"], WORKLOADS["gqa_causal_bf16_b2_hq32_hkv8_s4096_d128"],
            WORKLOADS["prefill_fp16_b1_h8_s4096_d64"]]
PREFILL_METRIC = "attention fwd TFLOP/s (% BF16 tensor peak)"
DECODE_METRIC = "decode HBM GB/s (% peak)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# --------------------------------------------------------------------------- helpers
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def host_info() -> dict:
    """CPU model, host core count, torch and CUDA versions: recorded with every
    CPU baseline (the oracle's rate depends on the host; the seeded inputs on
    the torch version)."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.lower().startswith("model name"):
                model = ln.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if not model:
        try:
            with open("/proc/cpuinfo") as f:
                for ln in f:
                    if ln.lower().startswith(("model name", "cpu part")):
                        model = ln.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    return {"cpu_model": model or "unknown", "host_cores": os.cpu_count(), "torch": torch.__version__,
            "cuda": torch.version.cuda,
            "gpu": torch.cuda.get_device_name() if torch.cuda.is_available() else None}


def prefill_flops(w) -> float:
    f = 4.0 * w.B * w.H * w.Sq * w.Sk * w.d
    return f / 2 if w.causal else f


def prefill_algorithmic_bytes(w) -> int:
    e = 2  # bf16/fp16
    return (w.B * w.H * w.Sq * w.d * e * 2          # Q read, O written
            + 2 * w.B * w.Hkv * w.Sk * w.d * e      # K, V read once
            + w.B * w.H * w.Sq * 4)                 # LSE written


def decode_algorithmic_bytes(w, lens) -> int:
    e = 2
    kv = int(np.sum(lens)) * w.Hkv * w.d * e * 2                     # valid K and V rows once
    partials = w.B * w.H * w.n_split * (w.d + 2) * 4 * 2              # written, then read by the merge
    qo = w.B * w.H * w.d * e * 2 + w.B * w.H * 4 + w.B * 4             # q, O, LSE, lengths
    return kv + partials + qo


def kernel_source_hash(files) -> str:
    """Hash of the kernel sources with comments and runs of white space
    removed: an edit to a comment leaves the committed DRAM figures valid,
    any change to the code itself invalidates them."""
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), encoding="utf-8") as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


PREFILL_SOURCES = ["exact_tiled_attention_gb300/csrc/prefill_fwd.cu",
                   "exact_tiled_attention_gb300/csrc/gbattn_ptx.cuh"]
PAIR_SOURCES = ["exact_tiled_attention_gb300/csrc/prefill_pair.cu",
                "exact_tiled_attention_gb300/csrc/gbattn_ptx.cuh"]
FP8_SOURCES = ["exact_tiled_attention_gb300/csrc/prefill_fp8.cu",
               "exact_tiled_attention_gb300/csrc/gbattn_ptx.cuh"]
BWD_SOURCES = {True: ["exact_tiled_attention_gb300/csrc/backward_atomic.cu",
                      "exact_tiled_attention_gb300/csrc/gbattn_ptx.cuh"],
               False: ["exact_tiled_attention_gb300/csrc/backward.cu",
                       "exact_tiled_attention_gb300/csrc/gbattn_ptx.cuh"]}
DECODE_SOURCES = ["exact_tiled_attention_gb300/csrc/decode_splitkv.cu",
                  "exact_tiled_attention_gb300/csrc/gbattn_ptx.cuh"]


def ncu_traffic(kernel_key: str, sources, workload: str):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel source changed since the counters were taken or the record is for
    another workload (another batch size, say)."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel_key)
    if not e or e.get("source_sha") != kernel_source_hash(sources):
        return None
    if not e.get("workload", "").startswith(workload):
        return None
    return e.get("dram_bytes_per_launch")


def with_batch(w, B: int):
    """The workload `w` at batch size B, its name carrying the new batch."""
    import dataclasses

    return dataclasses.replace(w, B=B, name=re.sub(r"_b\d+_", f"_b{B}_", w.name, count=1))


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- distributed
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------- GPU arm
def time_steps(fn, steps, warmup, world, stream):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1e3  # seconds


def time_steps_flushed(fn, steps, warmup, world, stream, flush_buf):
    """Per-launch CUDA-event timing with an L2 flush (a write of a buffer
    larger than L2) before every launch, outside the timed interval; returns
    the summed launch seconds."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for e0, e1 in evs:
        flush_buf.zero_()
        e0.record(stream)
        fn()
        e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    return sum(e0.elapsed_time(e1) for e0, e1 in evs) / 1e3


L2_BYTES = 129 * 1000 * 1000


def prefill_footprint(w) -> int:
    return prefill_algorithmic_bytes(w)


def bench_prefill(args, world, rank, peaks, peak_kind, w=None, with_e2e=True, pair=False):
    from exact_tiled_attention_gb300 import attn_fwd, attn_fwd_pair, gbattn_device_status

    w = w or PREFILL
    stream = torch.cuda.current_stream()
    q, k, v = make_workload(w, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.Sq), dtype=torch.float32, device="cuda")
    if pair:
        assert not w.causal and w.d == 128 and not with_e2e
        run = lambda: attn_fwd_pair(q, k, v, scale=w.scale, out=o, lse=lse, stream=stream)  # noqa: E731
    else:
        run = lambda: attn_fwd(q, k, v, scale=w.scale, causal=w.causal, out=o, lse=lse, stream=stream)  # noqa: E731
    flushed = prefill_footprint(w) < 2 * L2_BYTES
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    if flushed:
        flush_buf = torch.empty(4 * L2_BYTES // 4, dtype=torch.float32, device="cuda")
        secs = time_steps_flushed(run, args.steps, args.warmup, world, stream, flush_buf)
        del flush_buf
        l2_note = (f"inputs+outputs {prefill_footprint(w) / 1e6:.0f} MB < 2x L2: a 516 MB buffer is "
                   "written before every launch, outside its CUDA-event interval")
    else:
        secs = time_steps(run, args.steps, args.warmup, world, stream)
        l2_note = f"inputs+outputs {prefill_footprint(w) / 1e6:.0f} MB per step > 129 MB L2; no flush"
    clocks = sampler.stop()
    if gbattn_device_status() != 0:
        raise RuntimeError("a kernel reported a bounded-wait timeout")
    secs = max_over_ranks(secs, world)
    flops = prefill_flops(w)
    tflops_job = flops * args.steps * world / secs / 1e12
    per_launch = secs / args.steps
    achieved = flops / per_launch / 1e12
    peak = peaks["bf16_tflops"]
    key = f"prefill_fwd_kernel<{w.d},{'bf16' if w.dtype == torch.bfloat16 else 'fp16'},"
    key += ("causal>" if w.causal else "noncausal>") + ("" if w is PREFILL else f"@{w.name}")
    if pair:
        key = f"prefill_pair_kernel<{'bf16' if w.dtype == torch.bfloat16 else 'fp16'}>@{w.name}"
    traffic = ncu_traffic(key, PAIR_SOURCES if pair else PREFILL_SOURCES, w.name)
    dtype_name = "bf16" if w.dtype == torch.bfloat16 else "fp16"
    if not with_e2e:
        return {"workload": w.name, "impl": "cta_pair" if pair else "one_cta", "value": round(tflops_job, 3),
                "unit": "TFLOP/s",
                "ms_per_launch": round(per_launch * 1e3, 5), "steps": args.steps, "dtype": dtype_name,
                "flops_per_launch": flops,
                "roofline": {"bound": "tensor", "achieved": round(achieved, 3), "peak": peak,
                             "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                             "peak_kind": f"{peak_kind} bf16 burst (fp16 dense rate is the same)"},
                "l2": l2_note, "clocks": clocks}

    # end to end through the public API: every step copies its q, k, v in
    # from pinned host memory and its O and LSE back out.  Steps are
    # pipelined over two device buffer sets: step i+1's inputs go up on a
    # copy stream while step i computes, and step i's results come down on a
    # second copy stream (each step's copies stay inside the timed region).
    hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
    hos = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for _ in range(2)]
    hls = [torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True) for _ in range(2)]
    bufs = [(q, k, v, o, lse)] + [tuple(torch.empty_like(t) for t in (q, k, v, o, lse))]
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ev = {name: [torch.cuda.Event() for _ in range(2)] for name in ("in", "done", "out")}
    started = [False, False]

    def e2e_step(i):
        b = i % 2
        dq, dk, dv, do_, dl = bufs[b]
        if started[b]:
            up.wait_event(ev["done"][b])      # step i-2 finished reading this input set
            stream.wait_event(ev["out"][b])   # step i-2's results copied out of this output set
        with torch.cuda.stream(up):
            dq.copy_(hq, non_blocking=True)
            dk.copy_(hk, non_blocking=True)
            dv.copy_(hv, non_blocking=True)
            ev["in"][b].record(up)
        stream.wait_event(ev["in"][b])
        attn_fwd(dq, dk, dv, scale=w.scale, causal=w.causal, out=do_, lse=dl, stream=stream)
        ev["done"][b].record(stream)
        down.wait_event(ev["done"][b])
        with torch.cuda.stream(down):
            hos[b].copy_(do_, non_blocking=True)
            hls[b].copy_(dl, non_blocking=True)
            ev["out"][b].record(down)
        started[b] = True

    def time_e2e(steps, warmup):
        for i in range(warmup):
            e2e_step(i)
        torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        up.wait_event(e0)
        down.wait_event(e0)
        for i in range(warmup, warmup + steps):
            e2e_step(i)
        for b in range(2):
            stream.wait_event(ev["out"][b])
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / 1e3

    e2e_steps = max(3, min(args.steps, 20))
    e2e_secs = max_over_ranks(time_e2e(e2e_steps, 3), world)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = hos[0].numel() * hos[0].element_size() + hls[0].numel() * hls[0].element_size()
    line = {
        "metric": PREFILL_METRIC,
        "value": round(tflops_job, 3),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(secs / args.steps * 1e3, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": dtype_name,
        "data": "synthetic i.i.d. N(0,1), seeded",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "Hkv": w.Hkv, "Sq": w.Sq, "Sk": w.Sk,
                   "d": w.d, "causal": w.causal, "flops_per_step": flops,
                   "l2": l2_note,
                   "parallelism": f"replicas x{world} (independent problems per GPU)",
                   "torch": torch.__version__},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 3), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                     "peak_kind": f"{peak_kind} bf16 burst",
                     "frac_of_sustained": round(achieved / peaks.get("bf16_tflops_sustained", peak), 4),
                     "algorithmic_bytes": prefill_algorithmic_bytes(w)},
        "e2e": {"value": round(flops * e2e_steps * world / e2e_secs / 1e12, 3), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "note": "steps pipelined over two device buffer sets: inputs of step i+1 copied in "
                        "while step i computes, results of step i copied out on a second stream"},
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    return line


def bench_decode(args, world, rank, peaks, peak_kind, steps=None, warmup=None):
    from exact_tiled_attention_gb300 import attn_decode_splitkv, attn_decode_workspace_bytes, gbattn_device_status

    steps = steps or args.steps
    warmup = warmup if warmup is not None else args.warmup
    w = DECODE
    stream = torch.cuda.current_stream()
    q, k, v, sl = make_workload(w, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H), dtype=torch.float32, device="cuda")
    ws = torch.empty(attn_decode_workspace_bytes(w.B, w.H, w.n_split, w.d), dtype=torch.uint8,
                     device="cuda")
    run = lambda: attn_decode_splitkv(q, k, v, sl, scale=w.scale, n_split=w.n_split, workspace=ws,  # noqa: E731
                                      out=o, lse=lse, stream=stream)
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    secs = time_steps(run, steps, warmup, world, stream)
    clocks = sampler.stop()
    if gbattn_device_status() != 0:
        raise RuntimeError("a kernel reported a bounded-wait timeout")
    secs = max_over_ranks(secs, world)
    lens = sl.cpu().numpy()
    nbytes = decode_algorithmic_bytes(w, lens)
    per_step = secs / steps
    gbs_job = nbytes * steps * world / secs / 1e9
    achieved = nbytes / per_step / 1e9
    peak = peaks["hbm_gbs"]
    traffic = ncu_traffic("decode_partial_kernel<128,bf16>", DECODE_SOURCES, w.name)

    # end to end: only the step's inputs move each step (q and lengths in,
    # O and LSE out); the KV cache is resident state, copied in once before.
    hq = q.cpu().pin_memory()
    hsl = sl.cpu().pin_memory()
    ho = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
    hl = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)

    def e2e_step():
        q.copy_(hq, non_blocking=True)
        sl.copy_(hsl, non_blocking=True)
        attn_decode_splitkv(q, k, v, sl, scale=w.scale, n_split=w.n_split, workspace=ws, out=o, lse=lse,
                            stream=stream)
        ho.copy_(o, non_blocking=True)
        hl.copy_(lse, non_blocking=True)

    e2e_steps = max(3, min(steps, 20))
    e2e_secs = max_over_ranks(time_steps(e2e_step, e2e_steps, 3, world, stream), world)
    return {
        "metric": DECODE_METRIC,
        "value": round(gbs_job, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": steps,
        "warmup": warmup,
        "ms_per_step": round(per_step * 1e3, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic i.i.d. N(0,1), seeded; lengths uniform on [1024, 32768]",
        "config": {"workload": w.name, "B": w.B, "Hq": w.H, "Hkv": w.Hkv, "Sk_max": w.Sk, "d": w.d,
                   "n_split": w.n_split, "sum_valid_len": int(np.sum(lens)),
                   "algorithmic_bytes_per_step": nbytes,
                   "l2": "KV cache 8.6 GB > 129 MB L2; no flush",
                   "parallelism": f"replicas x{world} (independent problems per GPU)",
                   "torch": torch.__version__},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "peak_kind": f"{peak_kind} copy bandwidth"},
        "e2e": {"value": round(nbytes * e2e_steps * world / e2e_secs / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": hq.numel() * 2 + hsl.numel() * 4,
                "d2h_bytes_per_step": ho.numel() * 2 + hl.numel() * 4},
        "gpu_launches": 2 * steps,
        "clocks": clocks,
    }


def bench_backward(args, world, rank, peaks, peak_kind, w=None, steps=None, warmup=None, atomic=False):
    """attn_bwd (or, with atomic, attn_bwd_atomic) on a forward workload: O and
    LSE from one attn_fwd call (not timed), then the backward's three kernels
    timed per step.  FLOPs: the pages' convention of 2.5x the forward (five
    matmul-shaped products instead of two), i.e. 10*B*H*Sq*Sk*d, halved for
    causal."""
    from exact_tiled_attention_gb300 import (attn_bwd, attn_bwd_atomic, attn_bwd_atomic_workspace_bytes,
                                             attn_bwd_workspace_bytes, attn_fwd, gbattn_device_status)
    from exact_tiled_attention_gb300.inputs import make_generator, randn

    w = w or PREFILL
    steps = steps or args.steps
    warmup = warmup if warmup is not None else args.warmup
    stream = torch.cuda.current_stream()
    q, k, v = make_workload(w, device="cuda")
    do = randn(q.shape, q.dtype, make_generator(w.seed + 100, "cuda"), "cuda")
    o, lse = attn_fwd(q, k, v, scale=w.scale, causal=w.causal, stream=stream)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws_fn, fn = (attn_bwd_atomic_workspace_bytes, attn_bwd_atomic) if atomic else (attn_bwd_workspace_bytes, attn_bwd)
    ws = torch.empty(ws_fn(w.B, w.H, w.Sq, w.d), dtype=torch.uint8, device="cuda")
    run = lambda: fn(q, k, v, o, lse, do, scale=w.scale, causal=w.causal, workspace=ws,  # noqa: E731
                     dq=dq, dk=dk, dv=dv, stream=stream)
    footprint = 9 * q.numel() * 2 + ws.numel()
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    if footprint < 2 * L2_BYTES:
        flush_buf = torch.empty(4 * L2_BYTES // 4, dtype=torch.float32, device="cuda")
        secs = time_steps_flushed(run, steps, warmup, world, stream, flush_buf)
        del flush_buf
        l2_note = "L2 flushed before every call (516 MB write outside the event interval)"
    else:
        secs = time_steps(run, steps, warmup, world, stream)
        l2_note = f"inputs, outputs and workspace {footprint / 1e6:.0f} MB > 129 MB L2; no flush"
    clocks = sampler.stop()
    if gbattn_device_status() != 0:
        raise RuntimeError("a kernel reported a bounded-wait timeout")
    secs = max_over_ranks(secs, world)
    flops = 2.5 * prefill_flops(w)
    per_call = secs / steps
    achieved = flops / per_call / 1e12
    peak = peaks["bf16_tflops"]
    return {"metric": "attention bwd TFLOP/s (% BF16 tensor peak)", "workload": w.name,
            "impl": "atomic_dq (attn_bwd_atomic)" if atomic else "two_owner (attn_bwd)",
            "value": round(flops * steps * world / secs / 1e12, 3), "unit": "TFLOP/s",
            "ms_per_call": round(per_call * 1e3, 4), "steps": steps, "warmup": warmup,
            "flops_per_call": flops, "flop_convention": "2.5 x forward (10*B*H*Sq*Sk*d, /2 causal)",
            "kernels_per_call": 3,
            "roofline": {"bound": "tensor", "achieved": round(achieved, 3), "peak": peak,
                         "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                         "traffic": ncu_traffic(f"{'attn_bwd_atomic' if atomic else 'attn_bwd'} call@{w.name}",
                                                BWD_SOURCES[atomic], w.name),
                         "peak_kind": f"{peak_kind} bf16 burst; time of all three kernels"},
            "l2": l2_note, "clocks": clocks}


def bench_fp8(args, world, rank, peaks, peak_kind, w=None, steps=None, warmup=None):
    """attn_fwd_fp8 on a 128-dim forward workload with its inputs quantized
    to E4M3 per (batch, KV head); the call includes the V transpose.  FLOPs as
    for the 16-bit forward; the peak is the measured bf16 burst x 2 (the
    nominal dense FP8 : BF16 ratio of 4.5 : 2.25 PFLOP/s)."""
    from exact_tiled_attention_gb300 import attn_fwd_fp8, attn_fwd_fp8_workspace_bytes, gbattn_device_status

    w = w or PREFILL
    steps = steps or args.steps
    warmup = warmup if warmup is not None else args.warmup
    stream = torch.cuda.current_stream()
    q, k, v = make_workload(w, device="cuda")

    def quant(x):
        B, Hx, S, d = x.shape
        g = Hx // w.Hkv
        amax = x.float().reshape(B, w.Hkv, -1).abs().amax(dim=2).clamp_min(1e-12)
        ds = (amax / 448.0).contiguous()
        codes = (x.float().reshape(B, w.Hkv, g, S, d) / ds[:, :, None, None, None]).reshape(x.shape)
        return codes.to(torch.float8_e4m3fn).contiguous(), ds

    (q8, dq), (k8, dk), (v8, dv) = quant(q), quant(k), quant(v)
    del q, k, v
    o = torch.empty(q8.shape, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.B, w.H, w.Sq), dtype=torch.float32, device="cuda")
    ws = torch.empty(attn_fwd_fp8_workspace_bytes(w.B, w.Hkv, w.Sk, w.d), dtype=torch.uint8, device="cuda")
    run = lambda: attn_fwd_fp8(q8, k8, v8, dq, dk, dv, scale=w.scale, causal=w.causal, out=o, lse=lse,  # noqa: E731
                               workspace=ws, stream=stream)
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    secs = time_steps(run, steps, warmup, world, stream)
    clocks = sampler.stop()
    if gbattn_device_status() != 0:
        raise RuntimeError("a kernel reported a bounded-wait timeout")
    secs = max_over_ranks(secs, world)
    flops = prefill_flops(w)
    per_call = secs / steps
    achieved = flops / per_call / 1e12
    peak = 2.0 * peaks["bf16_tflops"]
    return {"metric": "attention fwd TFLOP/s (FP8 E4M3 inputs)", "workload": w.name + "_e4m3",
            "value": round(flops * steps * world / secs / 1e12, 3), "unit": "TFLOP/s",
            "ms_per_call": round(per_call * 1e3, 4), "steps": steps, "warmup": warmup, "dtype": "e4m3",
            "flops_per_call": flops, "kernels_per_call": 2,
            "roofline": {"bound": "tensor", "achieved": round(achieved, 3), "peak": peak, "unit": "TFLOP/s",
                         "frac": round(achieved / peak, 4),
                         "traffic": ncu_traffic(f"attn_fwd_fp8 call@{w.name}_e4m3", FP8_SOURCES, w.name),
                         "peak_kind": f"{peak_kind} bf16 burst x 2 (dense FP8 : BF16 = 2); "
                                      "V transpose included"},
            "l2": "inputs 256 MiB per call > 129 MB L2; no flush", "clocks": clocks}


# --------------------------------------------------------------------------- CPU oracle
def cpu_oracle_prefill(target_seconds: float, w=None):
    """Time the fp64 oracle on whole heads of the prefill workload (every
    query row of each sampled (b, h) against its keys), as many heads as fit
    in about target_seconds.  Returns (TFLOP/s, threads, sample description)."""
    import oracle

    w = w or PREFILL
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    q, k, v = make_workload(w, device=dev)
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]

    def run_heads(sel, n_rows=None):
        t_total, cells = 0.0, 0.0
        for (b, h) in sel:
            kvh = h // (w.H // w.Hkv)
            qh = q[b:b + 1, h:h + 1].float().cpu().numpy()
            kh = k[b:b + 1, kvh:kvh + 1].float().cpu().numpy()
            vh = v[b:b + 1, kvh:kvh + 1].float().cpu().numpy()
            n = n_rows or w.Sq
            rows = np.arange(w.Sq - n, w.Sq, dtype=np.int64)
            t0 = time.perf_counter()
            oracle.attn_fwd_rows(qh, kh, vh, w.scale, w.causal, rows)
            t_total += time.perf_counter() - t0
            vis = np.minimum(rows + 1 + (w.Sk - w.Sq), w.Sk) if w.causal else np.full(n, w.Sk)
            cells += float(np.sum(np.maximum(vis, 0)))
        return t_total, cells

    dt, cells = run_heads(heads[:1], n_rows=512)
    head_cells = float(w.Sq) * (w.Sk + 1) / 2 if w.causal else float(w.Sq) * w.Sk
    t_head = dt / cells * head_cells
    n_heads = int(min(len(heads), max(1, round(target_seconds / max(t_head, 1e-6)))))
    dt, cells = run_heads(heads[:n_heads])
    flops = 4.0 * w.d * cells
    return flops / dt / 1e12, oracle.num_threads(), (
        f"{n_heads} whole (b, h) heads of {w.B * w.H} (all {w.Sq} query rows each): "
        f"{cells:.3e} visible cells, {dt:.1f} s")


def cpu_oracle_decode(target_seconds: float):
    import oracle

    w = DECODE
    q, k, v, sl = make_workload(w, device="cuda" if torch.cuda.is_available() else "cpu")
    lens = sl.cpu().numpy()
    order = np.argsort(lens)
    b = int(order[len(order) // 2])  # a median-length sequence
    qb, kb, vb = (t[b:b + 1].float().cpu().numpy() for t in (q, k, v))
    t0 = time.perf_counter()
    oracle.attn_decode(qb, kb, vb, lens[b:b + 1], w.scale)
    dt = time.perf_counter() - t0
    reps = max(1, int(target_seconds / max(dt, 1e-3)))
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.attn_decode(qb, kb, vb, lens[b:b + 1], w.scale)
    dt = time.perf_counter() - t0
    nbytes = int(lens[b]) * w.Hkv * w.d * 2 * 2 * reps
    return nbytes / dt / 1e9, oracle.num_threads(), (
        f"sequence {b} (valid length {int(lens[b])}), all {w.H} query heads, {reps} repeats, {dt:.1f} s")


def cpu_oracle_backward(w):
    """Time the fp64 backward oracle on one KV head of batch 0 of a backward
    workload (all query heads of its group, every query row against its
    visible keys).  Returns (TFLOP/s in the 2.5 x forward convention,
    threads, sample description)."""
    import oracle
    from exact_tiled_attention_gb300.inputs import make_generator, randn

    dev = "cuda" if torch.cuda.is_available() else "cpu"
    q, k, v = make_workload(w, device=dev)
    do = randn(q.shape, q.dtype, make_generator(w.seed + 100, dev), dev)
    g = w.H // w.Hkv
    qs, dos = (t[0:1, 0:g].float().cpu().numpy() for t in (q, do))
    ks, vs = (t[0:1, 0:1].float().cpu().numpy() for t in (k, v))
    t0 = time.perf_counter()
    oracle.attn_bwd_kvheads(qs, ks, vs, dos, w.scale, w.causal, [0])
    dt = time.perf_counter() - t0
    cells = float(w.Sq) * (w.Sk + 1) / 2 if w.causal else float(w.Sq) * w.Sk
    flops = 10.0 * w.d * cells * g
    return flops / dt / 1e12, oracle.num_threads(), (
        f"{w.name}: KV head 0 of batch 0 ({g} query head(s), all {w.Sq} rows), {dt:.1f} s")


def leg_roofline(leg: dict, kernel: str) -> dict:
    """One compact row of the per-leg roofline table carried in the headline
    line's roofline object."""
    r = leg["roofline"]
    row = {"workload": leg.get("workload") or leg.get("config", {}).get("workload"), "kernel": kernel,
           "bound": r["bound"], "achieved": r["achieved"], "peak": r["peak"], "unit": r["unit"],
           "frac": r["frac"], "traffic": r["traffic"],
           "ms": leg.get("ms_per_launch") or leg.get("ms_per_call") or leg.get("ms_per_step")}
    if "cpu_baseline" in leg:
        row["cpu_baseline"] = leg["cpu_baseline"]["value"]
    return row


def reference_arm(args, world):
    """The fp64 oracle as it stands, timed on the host cores: every step is a
    bounded sample of the workload (query rows of one head for prefill, one
    sequence for decode), sized so the whole run takes about --cpu-seconds."""
    import oracle

    per_step = max(0.2, args.cpu_seconds / max(args.steps, 1))
    if args.workload != "decode":
        w = PREFILL if args.workload == "prefill" else WORKLOADS[args.workload]
        q, k, v = make_workload(w, device="cuda" if torch.cuda.is_available() else "cpu")
        qh, kh, vh = (t[0:1, 0:1].float().cpu().numpy() for t in (q, k, v))

        def step(n):
            rows = np.arange(w.Sq - n, w.Sq, dtype=np.int64)
            t0 = time.perf_counter()
            oracle.attn_fwd_rows(qh, kh, vh, w.scale, w.causal, rows)
            vis = np.clip(rows + 1 + (w.Sk - w.Sq), 0, w.Sk) if w.causal else np.full(n, w.Sk)
            return time.perf_counter() - t0, 4.0 * w.d * float(np.sum(vis))

        dt, work = step(32)
        n = int(min(w.Sq, max(8, 32 * per_step / max(dt, 1e-6))))
        unit, metric = "TFLOP/s", PREFILL_METRIC
        scale_out = 1e12
        sample = (f"{w.name}: last {n} query rows of (b=0, h=0) against its "
                  f"{'causally visible keys' if w.causal else 'keys'} (Sk = {w.Sk})")
    else:
        w = DECODE
        q, k, v, sl = make_workload(w, device="cuda" if torch.cuda.is_available() else "cpu")
        lens = sl.cpu().numpy()
        b = int(np.argsort(lens)[len(lens) // 2])
        qb, kb, vb = (t[b:b + 1].float().cpu().numpy() for t in (q, k, v))

        def step(n):
            t0 = time.perf_counter()
            for _ in range(n):
                oracle.attn_decode(qb, kb, vb, lens[b:b + 1], w.scale)
            return time.perf_counter() - t0, float(n * int(lens[b]) * w.Hkv * w.d * 2 * 2)

        dt, work = step(1)
        n = int(max(1, per_step / max(dt, 1e-6)))
        unit, metric = "GB/s", DECODE_METRIC
        scale_out = 1e9
        sample = (f"{n} decode(s) of sequence {b} (valid length {int(lens[b])}), all {w.H} query "
                  f"heads; algorithmic K/V bytes")
    for _ in range(args.warmup):
        step(max(1, n // 8))
    t_all = time.perf_counter()
    rates = []
    for _ in range(args.steps):
        dt, work = step(n)
        rates.append(work / dt / scale_out)
    wall = time.perf_counter() - t_all
    val = statistics.median(rates)
    cores = oracle.num_threads()
    return {"impl": "reference", "metric": metric, "value": val, "unit": unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(wall / max(args.steps, 1) * 1e3, 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic i.i.d. N(0,1), seeded",
            "config": {"workload": w.name, "sample_per_step": sample},
            "cpu_baseline": {"value": val, "unit": unit, "cores": cores, "kind": "oracle",
                             "sample": sample, **host_info()},
            "e2e": {"value": val, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# --------------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gbattn", "reference"], default="gbattn")
    ap.add_argument("--workload", default="prefill",
                    choices=["prefill", "decode"] + [n for n, w in WORKLOADS.items() if not w.decode])
    ap.add_argument("--fp8-only", action="store_true",
                    help="time only attn_fwd_fp8 on the headline forward workload (profiling runs)")
    ap.add_argument("--atomic", action="store_true",
                    help="with --backward-only: time attn_bwd_atomic (already the default)")
    ap.add_argument("--deterministic", action="store_true",
                    help="with --backward-only: time attn_bwd (bitwise repeatable) instead of attn_bwd_atomic")
    ap.add_argument("--backward-only", action="store_true",
                    help="time only the default backward (attn_bwd_atomic) on the headline forward workload")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-secondary", action="store_true", help="skip the second workload")
    ap.add_argument("--cta-pair", action="store_true",
                    help="with a non-causal d=128 --workload: time attn_fwd_pair (CTA pairs) alone")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the batch size of both workloads (smaller cases for ncu captures)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world, rank, local = dist_setup()
    peaks, peak_kind = load_peaks()
    if args.batch > 0:
        global PREFILL, DECODE
        PREFILL = with_batch(PREFILL, args.batch)
        DECODE = with_batch(DECODE, args.batch)

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(reference_arm(args, world)), flush=True)
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()
        return

    from exact_tiled_attention_gb300 import load_library

    load_library()  # fail loudly if the CUDA library is missing
    if args.fp8_only:
        w2 = PREFILL if args.workload == "prefill" else WORKLOADS[args.workload]
        if args.batch > 0:
            w2 = with_batch(w2, args.batch)
        line = bench_fp8(args, world, rank, peaks, peak_kind, w=w2)
        if rank == 0:
            print(json.dumps(line), flush=True)
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()
        return
    if args.backward_only:
        w2 = PREFILL if args.workload == "prefill" else WORKLOADS[args.workload]
        if args.batch > 0:
            w2 = with_batch(w2, args.batch)
        line = bench_backward(args, world, rank, peaks, peak_kind, w=w2, atomic=not args.deterministic)
        if rank == 0:
            print(json.dumps(line), flush=True)
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()
        return
    if args.workload == "prefill":
        line = bench_prefill(args, world, rank, peaks, peak_kind)
        if not args.no_secondary:
            line["decode"] = bench_decode(args, world, rank, peaks, peak_kind,
                                          steps=max(3, min(args.steps, 20)), warmup=3)
            line["prefill_other"] = [bench_prefill(args, world, rank, peaks, peak_kind, w=w2,
                                                   with_e2e=False) for w2 in OTHER_PREFILL]
            line["cta_pair"] = bench_prefill(args, world, rank, peaks, peak_kind, w=PAIR, with_e2e=False,
                                             pair=True)
            line["fp8"] = bench_fp8(args, world, rank, peaks, peak_kind, steps=max(3, min(args.steps, 20)),
                                    warmup=3)
            bw_steps = max(3, min(args.steps, 20))
            # the default backward (attention_backward: attn_bwd_atomic), then the
            # bitwise-repeatable one (attn_bwd)
            line["backward"] = [bench_backward(args, world, rank, peaks, peak_kind, w=w2, steps=bw_steps,
                                               warmup=3, atomic=True) for w2 in BACKWARD]
            line["backward_deterministic"] = [bench_backward(args, world, rank, peaks, peak_kind, w=w2,
                                                             steps=bw_steps, warmup=3) for w2 in BACKWARD]
    elif args.workload in WORKLOADS and not WORKLOADS[args.workload].decode:
        w2 = WORKLOADS[args.workload]
        if args.batch > 0:
            w2 = with_batch(w2, args.batch)
        if args.cta_pair:
            line = bench_prefill(args, world, rank, peaks, peak_kind, w=w2, with_e2e=False, pair=True)
        else:
            line = bench_prefill(args, world, rank, peaks, peak_kind, w=w2)
    else:
        line = bench_decode(args, world, rank, peaks, peak_kind)
        if not args.no_secondary:
            line["prefill"] = bench_prefill(args, world, rank, peaks, peak_kind)
    torch.cuda.synchronize()
    if rank == 0 and not args.no_cpu_baseline:
        host = host_info()

        def cpu_line(val, cores, sample, unit):
            return {"value": val, "unit": unit, "cores": cores, "kind": "oracle", "sample": sample, **host}

        if args.workload != "decode":
            line["cpu_baseline"] = cpu_line(*cpu_oracle_prefill(
                args.cpu_seconds, None if args.workload == "prefill" else WORKLOADS[args.workload]), "TFLOP/s")
        else:
            line["cpu_baseline"] = cpu_line(*cpu_oracle_decode(args.cpu_seconds), "GB/s")
        # every other leg: the oracle on a bounded sample of that leg's workload
        leg_seconds = max(1.0, args.cpu_seconds / 4)
        if isinstance(line.get("decode"), dict):
            line["decode"]["cpu_baseline"] = cpu_line(*cpu_oracle_decode(leg_seconds), "GB/s")
        if isinstance(line.get("prefill"), dict):
            line["prefill"]["cpu_baseline"] = cpu_line(*cpu_oracle_prefill(leg_seconds), "TFLOP/s")
        by_workload = {}
        for leg in line.get("prefill_other", []):
            leg["cpu_baseline"] = cpu_line(*cpu_oracle_prefill(leg_seconds, WORKLOADS[leg["workload"]]),
                                           "TFLOP/s")
            by_workload[leg["workload"]] = leg["cpu_baseline"]
        if isinstance(line.get("cta_pair"), dict) and line["cta_pair"]["workload"] in by_workload:
            line["cta_pair"]["cpu_baseline"] = by_workload[line["cta_pair"]["workload"]]
        if isinstance(line.get("fp8"), dict):
            line["fp8"]["cpu_baseline"] = dict(line["cpu_baseline"], sample=line["cpu_baseline"]["sample"]
                                               + " (the oracle takes the dequantized inputs at the same rate)")
        bwd_cpu = {}
        for legs in (line.get("backward", []), line.get("backward_deterministic", [])):
            for leg in legs:
                if leg["workload"] not in bwd_cpu:
                    bwd_cpu[leg["workload"]] = cpu_line(*cpu_oracle_backward(WORKLOADS[leg["workload"]]),
                                                        "TFLOP/s")
                leg["cpu_baseline"] = bwd_cpu[leg["workload"]]
    if "roofline" in line:
        # the per-leg roofline table, in the headline's roofline object
        rows = []
        if isinstance(line.get("decode"), dict):
            rows.append(leg_roofline(line["decode"], "decode_partial_kernel + decode_merge_kernel"))
        if isinstance(line.get("prefill"), dict):
            rows.append(leg_roofline(line["prefill"], "prefill_fwd_kernel"))
        for leg in line.get("prefill_other", []):
            rows.append(leg_roofline(leg, "prefill_fwd_kernel"))
        if isinstance(line.get("cta_pair"), dict):
            rows.append(leg_roofline(line["cta_pair"], "prefill_pair_kernel"))
        if isinstance(line.get("fp8"), dict):
            rows.append(leg_roofline(line["fp8"], "v_transpose_kernel + prefill_fp8_kernel"))
        for leg in line.get("backward", []):
            rows.append(leg_roofline(leg, "attn_bwd_atomic (3 kernels; the default backward)"))
        for leg in line.get("backward_deterministic", []):
            rows.append(leg_roofline(leg, "attn_bwd (3 kernels; bitwise repeatable)"))
        if rows:
            line["roofline"]["legs"] = rows
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
