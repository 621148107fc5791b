"""GPU parity of the CTA-pair forward (C ABI attn_fwd_pair: non-causal, d = 128,
two CTAs sharing every K/V tile through cta_group::2 MMAs) against the fp64
oracle, element by element on small shapes that span several 512-row pair
units and ragged query/key tails, on sampled rows of the full-size non-causal
workload, and against the one-CTA forward on the same inputs."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_gb300 import GbattnError, attn_fwd, attn_fwd_pair, gbattn_device_status
from exact_tiled_attention_gb300.inputs import WORKLOADS, make_prefill
from tests.parity_util import assert_attn_close, host_f32

pytestmark = pytest.mark.gpu

DT = {"fp16": torch.float16, "bf16": torch.bfloat16}


@pytest.mark.parametrize("shape", [
    (1, 2, 2, 512, 512, "bf16"),     # one pair unit, every tile full
    (1, 2, 2, 600, 700, "fp16"),     # ragged query and key tails, two units
    (2, 4, 2, 257, 384, "bf16"),     # GQA; tiles of rank 1's L beyond Sq
    (1, 3, 1, 1100, 129, "bf16"),    # MQA; key tail of one column
    (1, 2, 2, 100, 1000, "fp16"),    # fewer queries than one tile
    (1, 1, 1, 1, 1, "bf16"),         # one query, one key
    (1, 2, 2, 1024, 64, "fp16"),     # keys fit in rank 0's half of one K tile
])
def test_pair_small_all_elements(shape):
    B, H, Hkv, Sq, Sk, dt = shape
    q, k, v = make_prefill(B, H, Hkv, Sq, Sk, 128, DT[dt], 21, device="cuda")
    scale = 1.0 / math.sqrt(128)
    o, lse = attn_fwd_pair(q, k, v, scale=scale)
    torch.cuda.synchronize()
    assert gbattn_device_status() == 0
    o_ref, lse_ref = oracle.attn_fwd(host_f32(q), host_f32(k), host_f32(v), scale, False)
    assert_attn_close(o, lse, o_ref, lse_ref, f"pair {shape}")


def test_pair_matches_one_cta_forward():
    """Same definition, same operand rounding: the pair and the one-CTA
    forward agree to within the rounding of P and O."""
    q, k, v = make_prefill(2, 4, 2, 1500, 1300, 128, torch.bfloat16, 8, device="cuda")
    o1, l1 = attn_fwd(q, k, v, causal=False)
    o2, l2 = attn_fwd_pair(q, k, v)
    torch.cuda.synchronize()
    assert (o1.float() - o2.float()).abs().max().item() <= 1e-2
    assert (l1 - l2).abs().max().item() <= 1e-4


def test_pair_bitwise_repeatable():
    q, k, v = make_prefill(1, 4, 4, 2000, 2000, 128, torch.float16, 4, device="cuda")
    o1, l1 = attn_fwd_pair(q, k, v)
    o2, l2 = attn_fwd_pair(q, k, v)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_pair_unit_values_and_zero_query():
    q, k, _ = make_prefill(1, 2, 2, 900, 777, 128, torch.bfloat16, 12, device="cuda")
    o, _ = attn_fwd_pair(q, k, torch.ones_like(k))
    torch.cuda.synchronize()
    assert (o.float() - 1).abs().max().item() <= 1e-2
    g = torch.Generator(device="cuda").manual_seed(5)
    v = torch.randn(k.shape, device="cuda", generator=g).to(torch.bfloat16)
    o, lse = attn_fwd_pair(torch.zeros_like(q), k, v)
    torch.cuda.synchronize()
    ref = v.double().mean(dim=2, keepdim=True).expand_as(o)
    assert (o.double() - ref).abs().max().item() <= 2e-2
    assert (lse.double() - math.log(777)).abs().max().item() <= 1e-3


def test_pair_rejects_other_head_dims():
    q, k, v = make_prefill(1, 2, 2, 64, 64, 64, torch.bfloat16, 1, device="cuda")
    with pytest.raises(GbattnError):
        attn_fwd_pair(q, k, v)


def test_pair_workload_sampled_rows():
    w = WORKLOADS["noncausal_bf16_b4_h16_s8192_d128"]
    q, k, v = make_prefill(w.B, w.H, w.Hkv, w.Sq, w.Sk, w.d, w.dtype, w.seed, device="cuda")
    o, lse = attn_fwd_pair(q, k, v, scale=w.scale)
    torch.cuda.synchronize()
    assert gbattn_device_status() == 0
    assert torch.isfinite(o).all()
    rng = np.random.default_rng(w.seed)
    rows = set(rng.integers(0, w.B * w.H * w.Sq, size=256).tolist())
    for bh in range(w.B * w.H):  # rows of each of the four tiles of a pair unit, first and last rows
        for i in (0, 127, 128, 255, 256, 383, 384, 511, 512, w.Sq - 1):
            rows.add(bh * w.Sq + i)
    rows = np.array(sorted(rows), dtype=np.int64)
    o_ref, lse_ref = oracle.attn_fwd_rows(host_f32(q), host_f32(k), host_f32(v), w.scale, False, rows)
    idx = torch.from_numpy(rows).cuda()
    assert_attn_close(o.reshape(-1, w.d)[idx], lse.reshape(-1)[idx], o_ref, lse_ref, w.name)
