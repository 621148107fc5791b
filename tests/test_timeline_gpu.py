"""GPU: the per-CTA timeline of the forward entry points (gbattn_timeline_set).  Each CTA of
a launch writes one record (start, end, SM, work unit); the units of one
launch cover every (batch, head, query pair) exactly once, and the output
with the timeline on still matches the fp64 oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_gb300 import (attn_fwd, attn_fwd_fp8, attn_fwd_pair, gbattn_device_status,
                                         gbattn_timeline_set)
from exact_tiled_attention_gb300.inputs import make_prefill
from tests.parity_util import assert_attn_close, host_f32

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape", [
    (2, 6, 3, 700, 700, 128, torch.bfloat16, True),    # GQA, ragged tail, causal
    (1, 4, 4, 1100, 900, 64, torch.float16, False),    # d = 64, Sq != Sk
])
def test_timeline_records_every_unit_once(shape):
    B, H, Hkv, Sq, Sk, d, dt, causal = shape
    q, k, v = make_prefill(B, H, Hkv, Sq, Sk, d, dt, 3, device="cuda")
    n_pairs = -(-Sq // 256)
    grid = B * H * n_pairs
    rec = torch.zeros(grid + 5, 4, dtype=torch.int64, device="cuda")
    try:
        gbattn_timeline_set(rec)
        o, lse = attn_fwd(q, k, v, scale=1.0 / math.sqrt(d), causal=causal)
        torch.cuda.synchronize()
    finally:
        gbattn_timeline_set(None)
    assert gbattn_device_status() == 0
    r = rec.cpu().numpy().astype(np.uint64)
    assert (r[grid:] == 0).all()                          # nothing past the grid
    r = r[:grid]
    assert (r[:, 0] > 0).all() and (r[:, 1] >= r[:, 0]).all()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert (r[:, 2] < sms).all()
    units = sorted((int(u >> np.uint64(32)), int(u & np.uint64(0xFFFFFFFF))) for u in r[:, 3])
    assert units == [(bh, p) for bh in range(B * H) for p in range(n_pairs)]
    o_ref, lse_ref = oracle.attn_fwd(host_f32(q), host_f32(k), host_f32(v), 1.0 / math.sqrt(d), causal)
    assert_attn_close(o, lse, o_ref, lse_ref, f"timeline {shape}")


def test_timeline_capacity_too_small_writes_nothing():
    q, k, v = make_prefill(1, 4, 2, 600, 600, 128, torch.bfloat16, 4, device="cuda")
    grid = 1 * 4 * 3
    rec = torch.zeros(grid - 1, 4, dtype=torch.int64, device="cuda")
    try:
        gbattn_timeline_set(rec)
        attn_fwd(q, k, v, causal=True)
        torch.cuda.synchronize()
    finally:
        gbattn_timeline_set(None)
    assert gbattn_device_status() == 0
    assert int(rec.abs().sum()) == 0
    # and off again: a later launch writes nothing either
    attn_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert int(rec.abs().sum()) == 0


def test_timeline_fp8_records_every_unit_once():
    B, H, Hkv, Sq, Sk, d = 1, 4, 2, 600, 500, 128
    g = torch.Generator(device="cpu").manual_seed(9)
    q, k, v = (torch.randn(B, h, s, d, generator=g).clamp(-4, 4).to(torch.float8_e4m3fn).cuda()
               for h, s in ((H, Sq), (Hkv, Sk), (Hkv, Sk)))
    n_pairs = -(-Sq // 256)
    grid = B * H * n_pairs
    rec = torch.zeros(grid, 4, dtype=torch.int64, device="cuda")
    try:
        gbattn_timeline_set(rec)
        o, _ = attn_fwd_fp8(q, k, v, causal=True)
        torch.cuda.synchronize()
    finally:
        gbattn_timeline_set(None)
    assert gbattn_device_status() == 0
    r = rec.cpu().numpy().astype(np.uint64)
    assert (r[:, 0] > 0).all() and (r[:, 1] >= r[:, 0]).all()
    units = sorted((int(u >> np.uint64(32)), int(u & np.uint64(0xFFFFFFFF))) for u in r[:, 3])
    assert units == [(bh, p) for bh in range(B * H) for p in range(n_pairs)]
    assert torch.isfinite(o.float()).all()


def test_timeline_pair_records_every_cluster_unit_twice():
    B, H, Hkv, Sq, Sk, d = 1, 4, 2, 1100, 700, 128
    q, k, v = make_prefill(B, H, Hkv, Sq, Sk, d, torch.bfloat16, 6, device="cuda")
    n_quads = -(-Sq // 512)
    grid = 2 * B * H * n_quads
    rec = torch.zeros(grid, 4, dtype=torch.int64, device="cuda")
    try:
        gbattn_timeline_set(rec)
        o, lse = attn_fwd_pair(q, k, v, scale=1.0 / math.sqrt(d))
        torch.cuda.synchronize()
    finally:
        gbattn_timeline_set(None)
    assert gbattn_device_status() == 0
    r = rec.cpu().numpy().astype(np.uint64)
    assert (r[:, 0] > 0).all() and (r[:, 1] >= r[:, 0]).all()
    assert (r[0::2, 3] == r[1::2, 3]).all()                       # the two CTAs of a cluster
    units = sorted((int(u >> np.uint64(32)), int(u & np.uint64(0xFFFFFFFF))) for u in r[0::2, 3])
    assert units == [(bh, u) for bh in range(B * H) for u in range(n_quads)]
    o_ref, lse_ref = oracle.attn_fwd(host_f32(q), host_f32(k), host_f32(v), 1.0 / math.sqrt(d), False)
    assert_attn_close(o, lse, o_ref, lse_ref, "timeline pair")
