"""GPU parity of the backward (C ABI attn_bwd) against the fp64 oracle.

The forward runs on the GPU (attn_fwd) and hands its O and LSE to attn_bwd,
as a training step would; the oracle computes dQ, dK, dV from q, k, v, dO
alone.  Small shapes are compared on every element; the full-size workloads
on every element of sampled KV heads (their whole query-head group), plus
properties that hold at any size."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_gb300 import attn_bwd, attn_fwd, gbattn_device_status
from exact_tiled_attention_gb300.inputs import WORKLOADS, make_generator, make_prefill, randn
from tests.parity_util import assert_grad_close, grad_extras, host_f32

pytestmark = pytest.mark.gpu

DT = {"fp16": torch.float16, "bf16": torch.bfloat16}


def _fwd_bwd(q, k, v, do, scale, causal):
    o, lse = attn_fwd(q, k, v, scale=scale, causal=causal)
    dq, dk, dv = attn_bwd(q, k, v, o, lse, do, scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert gbattn_device_status() == 0
    return dq, dk, dv


def _dout(shape, dtype, seed):
    return randn(shape, dtype, make_generator(seed, "cuda"), "cuda")


@pytest.mark.parametrize("shape", [
    # head dim 64: the tiny fp16 workload, ragged tails, causal, GQA
    (1, 4, 4, 128, 128, "fp16", False, 64),
    (1, 2, 2, 300, 300, "fp16", True, 64),
    (2, 4, 2, 257, 257, "bf16", True, 64),
    (1, 2, 1, 200, 77, "fp16", True, 64),
    (1, 1, 1, 1, 1, "fp16", False, 64),
    (1, 1, 1, 128, 128, "bf16", False),
    (1, 2, 2, 300, 300, "bf16", True),     # ragged tails, diagonal blocks
    (1, 2, 2, 300, 300, "fp16", False),
    (2, 4, 2, 257, 257, "bf16", True),     # GQA g = 2
    (1, 2, 2, 129, 700, "fp16", False),    # Sq != Sk
    (1, 4, 1, 512, 512, "bf16", True),     # MQA g = 4
    (1, 2, 2, 64, 1000, "bf16", True),     # causal Sq < Sk (bottom-right)
    (1, 2, 1, 200, 77, "bf16", True),      # causal Sq > Sk: rows with no key
    (1, 1, 1, 1, 1, "bf16", False),
    (2, 2, 2, 1, 333, "fp16", True),
    (1, 2, 2, 333, 1, "bf16", False),
])
def test_bwd_small_all_elements(shape):
    B, H, Hkv, Sq, Sk, dt, causal = shape[:7]
    d = shape[7] if len(shape) > 7 else 128
    q, k, v = make_prefill(B, H, Hkv, Sq, Sk, d, DT[dt], 31, device="cuda")
    do = _dout((B, H, Sq, d), DT[dt], 32)
    scale = 1.0 / math.sqrt(d)
    dq, dk, dv = _fwd_bwd(q, k, v, do, scale, causal)
    rq, rk, rv, _, _ = oracle.attn_bwd(host_f32(q), host_f32(k), host_f32(v), host_f32(do), scale, causal)
    ex = grad_extras(host_f32(q), host_f32(k), host_f32(v), host_f32(do), scale, causal)
    assert_grad_close(dq, rq, f"dq {shape}", extra=ex["dq"])
    assert_grad_close(dk, rk, f"dk {shape}", extra=ex["dk"])
    assert_grad_close(dv, rv, f"dv {shape}")


def test_bwd_key_gradient_sums_to_zero_and_constant_values():
    """sum_j dK_j = 0 per KV head (rows of dS sum to zero); with all V rows
    equal, dQ = dK = 0.  Both hold at any size."""
    B, H, Hkv, S, d = 1, 4, 2, 1000, 128
    q, k, v = make_prefill(B, H, Hkv, S, S, d, torch.bfloat16, 41, device="cuda")
    do = _dout((B, H, S, d), torch.bfloat16, 42)
    dq, dk, dv = _fwd_bwd(q, k, v, do, 1 / math.sqrt(d), True)
    col = dk.double().sum(dim=2)
    assert (col.abs().max() / dk.double().abs().max()).item() <= 5e-2
    v1 = v[:, :, :1, :].expand_as(v).contiguous()
    dq1, dk1, _ = _fwd_bwd(q, k, v1, do, 1 / math.sqrt(d), False)
    assert dq1.abs().max().item() <= 2e-2 * dq.abs().max().item()
    assert dk1.abs().max().item() <= 2e-2 * dk.abs().max().item()


@pytest.mark.parametrize("name,kv_ids", [
    ("tiny_fwd_fp16", [0, 3]),
    ("prefill_fp16_b1_h8_s4096_d64", [0, 7]),
    ("causal_bf16_b4_h16_s8192_d128", [0, 63]),
    ("gqa_causal_bf16_b2_hq32_hkv8_s4096_d128", [1, 14]),
])
def test_bwd_workload_sampled_heads(name, kv_ids):
    w = WORKLOADS[name]
    q, k, v = make_prefill(w.B, w.H, w.Hkv, w.Sq, w.Sk, w.d, w.dtype, w.seed, device="cuda")
    do = _dout((w.B, w.H, w.Sq, w.d), w.dtype, w.seed + 100)
    dq, dk, dv = _fwd_bwd(q, k, v, do, w.scale, w.causal)
    assert torch.isfinite(dq).all() and torch.isfinite(dk).all() and torch.isfinite(dv).all()
    g = w.H // w.Hkv
    rq, rk, rv = oracle.attn_bwd_kvheads(host_f32(q), host_f32(k), host_f32(v), host_f32(do), w.scale,
                                         w.causal, kv_ids)
    for r, kid in enumerate(kv_ids):
        b, kvh = divmod(kid, w.Hkv)
        grp = slice(kvh * g, (kvh + 1) * g)
        ex = grad_extras(host_f32(q[b:b + 1, grp]), host_f32(k[b:b + 1, kvh:kvh + 1]), host_f32(v[b:b + 1, kvh:kvh + 1]),
                         host_f32(do[b:b + 1, grp]), w.scale, w.causal)
        assert_grad_close(dq[b, grp], rq[r], f"{name} dq kv{kid}", extra=ex["dq"][0])
        assert_grad_close(dk[b, kvh], rk[r], f"{name} dk kv{kid}", extra=ex["dk"][0, 0])
        assert_grad_close(dv[b, kvh], rv[r], f"{name} dv kv{kid}")


def test_bwd_bitwise_repeatable():
    """Every gradient element has one writer and a fixed summation order, so
    two calls give identical bits."""
    q, k, v = make_prefill(1, 4, 2, 700, 700, 128, torch.bfloat16, 51, device="cuda")
    do = _dout(q.shape, torch.bfloat16, 52)
    o, lse = attn_fwd(q, k, v, causal=True)
    a = attn_bwd(q, k, v, o, lse, do, causal=True)
    b = attn_bwd(q, k, v, o, lse, do, causal=True)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y)
