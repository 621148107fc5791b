"""Long sequences: the key loops, causal tile counts and row offsets at
65,536 tokens per head (forward), 32,768 (backward) and a 262,144-slot decode
cache.  Forward and decode rows are compared with the oracle one by one; the
backward, whose oracle cost grows with Sq*Sk per head, is checked through
properties that hold at any size and against the other backward path."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_gb300 import (attn_bwd, attn_bwd_atomic, attn_decode_splitkv, attn_fwd, attn_fwd_pair,
                                         gbattn_device_status)
from exact_tiled_attention_gb300.inputs import make_generator, make_prefill, randn
from tests.parity_util import assert_attn_close, host_f32

pytestmark = pytest.mark.gpu

S = 65536


def _rows(H, Sq):
    picks = [0, 1, 127, 128, 20000, Sq // 2 - 1, Sq // 2, Sq - 129, Sq - 1]
    return np.array([h * Sq + i for h in range(H) for i in picks], dtype=np.int64)


@pytest.mark.parametrize("pair", [False, True])
def test_forward_65536_sampled_rows(pair):
    H, Hkv, d = 2, 1, 128
    q, k, v = make_prefill(1, H, Hkv, S, S, d, torch.bfloat16, 71, device="cuda")
    scale = 1.0 / math.sqrt(d)
    causal = not pair  # the CTA-pair kernel is non-causal only
    if pair:
        o, lse = attn_fwd_pair(q, k, v, scale=scale)
    else:
        o, lse = attn_fwd(q, k, v, scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert gbattn_device_status() == 0
    rows = _rows(H, S)
    o_ref, lse_ref = oracle.attn_fwd_rows(host_f32(q), host_f32(k), host_f32(v), scale, causal, rows)
    o_got = o.reshape(-1, d)[torch.from_numpy(rows).cuda()]
    lse_got = lse.reshape(-1)[torch.from_numpy(rows).cuda()]
    assert_attn_close(o_got, lse_got, o_ref, lse_ref, f"S={S} {'pair' if pair else 'causal'}")


@pytest.mark.parametrize("d,dt", [(128, torch.bfloat16), (64, torch.float16)])
def test_backward_32768_properties_and_paths_agree(d, dt):
    B, H, Hkv, Sq = 1, 2, 1, 32768
    q, k, v = make_prefill(B, H, Hkv, Sq, Sq, d, dt, 72, device="cuda")
    do = randn(q.shape, q.dtype, make_generator(73, "cuda"), "cuda")
    o, lse = attn_fwd(q, k, v, causal=True)
    a = attn_bwd(q, k, v, o, lse, do, causal=True)
    b = attn_bwd_atomic(q, k, v, o, lse, do, causal=True)
    torch.cuda.synchronize()
    assert gbattn_device_status() == 0
    for x in a + b:
        assert torch.isfinite(x).all()
    # rows of dS sum to zero, so the key gradients of a KV head sum to zero
    for dk in (a[1], b[1]):
        col = dk.double().sum(dim=2)
        assert (col.abs().max() / dk.double().abs().max()).item() <= 5e-2
    # two independent schedules of the same gradients
    for x, y, n in zip(a, b, ("dq", "dk", "dv")):
        err = (x.float() - y.float()).abs().max().item()
        assert err <= 2e-2 * y.float().abs().max().item(), n


def test_decode_262144_slot_cache():
    B, Hq, Hkv, Skm, d = 2, 8, 2, 262144, 128
    g = torch.Generator(device="cuda").manual_seed(74)
    q = torch.randn(B, Hq, 1, d, generator=g, device="cuda").to(torch.bfloat16)
    kc = torch.randn(B, Hkv, Skm, d, generator=g, device="cuda").to(torch.bfloat16)
    vc = torch.randn(B, Hkv, Skm, d, generator=g, device="cuda").to(torch.bfloat16)
    lens = [Skm, 100003]
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    scale = 1.0 / math.sqrt(d)
    o, lse, _ = attn_decode_splitkv(q, kc, vc, sl, scale=scale, n_split=16)
    torch.cuda.synchronize()
    assert gbattn_device_status() == 0
    o_ref, lse_ref = oracle.attn_decode(host_f32(q), host_f32(kc), host_f32(vc), np.array(lens, np.int32), scale)
    assert_attn_close(o, lse, o_ref, lse_ref, "decode 262144")
