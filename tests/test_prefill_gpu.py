"""GPU parity of the prefill forward (C ABI attn_fwd) against the fp64 oracle.

Small shapes are compared on every output element; the full-size workloads
(launched exactly as the bench launches them) are compared on sampled rows
plus the first and last rows of every head, and through properties that hold
at any size (Q = 0 gives prefix means, V = 1 gives 1, repeat runs are
bit-identical)."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_gb300 import attn_fwd, gbattn_device_status
from exact_tiled_attention_gb300.inputs import WORKLOADS, make_prefill
from tests.parity_util import assert_attn_close, host_f32

pytestmark = pytest.mark.gpu

DT = {"fp16": torch.float16, "bf16": torch.bfloat16}


def _run_and_compare(B, H, Hkv, Sq, Sk, d, dt, causal, seed):
    q, k, v = make_prefill(B, H, Hkv, Sq, Sk, d, DT[dt], seed, device="cuda")
    scale = 1.0 / math.sqrt(d)
    o, lse = attn_fwd(q, k, v, scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert gbattn_device_status() == 0
    o_ref, lse_ref = oracle.attn_fwd(host_f32(q), host_f32(k), host_f32(v), scale, causal)
    return assert_attn_close(o, lse, o_ref, lse_ref, f"{(B, H, Hkv, Sq, Sk, d, dt, causal)}")


@pytest.mark.parametrize("shape", [
    # tiny exact-attention forward workload
    (1, 4, 4, 128, 128, 64, "fp16", False),
    # ragged query/key tails, several tiles, both head dims, both dtypes
    (1, 2, 2, 300, 300, 64, "bf16", True),
    (1, 2, 2, 300, 300, 64, "fp16", False),
    (2, 4, 2, 257, 257, 128, "bf16", True),
    (1, 2, 2, 129, 700, 128, "fp16", False),
    (1, 3, 1, 512, 512, 128, "bf16", True),
    (1, 2, 2, 640, 640, 128, "fp16", True),
    (2, 4, 2, 700, 700, 64, "fp16", True),   # d = 64: several query pairs, GQA g = 2, diagonal tiles
    (1, 3, 3, 1100, 900, 64, "bf16", False), # d = 64: Sq != Sk, ragged key tail
    # rectangular causal, bottom-right: Sq < Sk and Sq > Sk (rows with no key)
    (1, 2, 2, 64, 1000, 128, "bf16", True),
    (1, 2, 1, 200, 77, 64, "bf16", True),
    # Sq - Sk = 200: the first query tile of the first pair sees no key while
    # the second does (tile L starts without waiting for tile H)
    (1, 2, 2, 400, 200, 128, "bf16", True),
    (1, 2, 2, 400, 200, 64, "fp16", True),
    # degenerate sizes
    (1, 1, 1, 1, 1, 64, "bf16", False),
    (1, 1, 1, 1, 1, 128, "fp16", True),
    (2, 2, 2, 1, 333, 128, "bf16", False),
    (1, 2, 2, 333, 1, 64, "fp16", False),
])
def test_prefill_small_all_elements(shape):
    _run_and_compare(*shape, seed=11)


def test_prefill_bitwise_repeatable():
    q, k, v = make_prefill(1, 4, 2, 1000, 1000, 128, torch.bfloat16, 5, device="cuda")
    o1, l1 = attn_fwd(q, k, v, causal=True)
    o2, l2 = attn_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_zero_query_gives_prefix_mean(causal, d):
    """Q = 0: every score is 0, so O_i is the mean of the visible V rows and
    LSE_i = log(#visible) -- checks the GPU path without the oracle."""
    B, H, Hkv, S = 1, 4, 2, 777
    g = torch.Generator(device="cuda").manual_seed(3)
    q = torch.zeros(B, H, S, d, device="cuda", dtype=torch.bfloat16)
    k = torch.randn(B, Hkv, S, d, device="cuda", generator=g).to(torch.bfloat16)
    v = torch.randn(B, Hkv, S, d, device="cuda", generator=g).to(torch.bfloat16)
    o, lse = attn_fwd(q, k, v, causal=causal)
    torch.cuda.synchronize()
    vv = v.double().repeat_interleave(H // Hkv, dim=1)
    if causal:
        ref = vv.cumsum(dim=2) / torch.arange(1, S + 1, device="cuda", dtype=torch.float64).view(1, 1, S, 1)
        lref = torch.log(torch.arange(1, S + 1, device="cuda", dtype=torch.float64)).expand(B, H, S)
    else:
        ref = vv.mean(dim=2, keepdim=True).expand(B, H, S, d)
        lref = torch.full((B, H, S), math.log(S), device="cuda", dtype=torch.float64)
    assert (o.double() - ref).abs().max().item() <= 2e-2
    assert (lse.double() - lref).abs().max().item() <= 1e-3


def test_unit_values_give_unit_output():
    q, k, _ = make_prefill(2, 2, 2, 600, 600, 128, torch.float16, 9, device="cuda")
    v = torch.ones_like(k)
    for causal in (False, True):
        o, _ = attn_fwd(q, k, v, causal=causal)
        torch.cuda.synchronize()
        assert (o.float() - 1).abs().max().item() <= 1e-2


def _sample_rows(w, n_random, seed):
    rng = np.random.default_rng(seed)
    rows = set(rng.integers(0, w.B * w.H * w.Sq, size=n_random).tolist())
    for bh in range(w.B * w.H):  # first, last and tile-boundary rows of each head
        for i in (0, 127, 128, 255, 256, w.Sq - 1):
            if i < w.Sq:
                rows.add(bh * w.Sq + i)
    return np.array(sorted(rows), dtype=np.int64)


@pytest.mark.parametrize("name", ["tiny_fwd_fp16", "prefill_fp16_b1_h8_s4096_d64",
                                  "causal_bf16_b4_h16_s8192_d128",
                                  "gqa_causal_bf16_b2_hq32_hkv8_s4096_d128",
                                  "noncausal_bf16_b4_h16_s8192_d128"])
def test_workload_sampled_rows(name):
    w = WORKLOADS[name]
    q, k, v = make_prefill(w.B, w.H, w.Hkv, w.Sq, w.Sk, w.d, w.dtype, w.seed, device="cuda")
    o, lse = attn_fwd(q, k, v, scale=w.scale, causal=w.causal)
    torch.cuda.synchronize()
    assert gbattn_device_status() == 0
    assert torch.isfinite(o).all()
    rows = _sample_rows(w, 384, w.seed)
    o_ref, lse_ref = oracle.attn_fwd_rows(host_f32(q), host_f32(k), host_f32(v), w.scale, w.causal, rows)
    assert_attn_close(o.reshape(-1, w.d)[torch.from_numpy(rows).cuda()], lse.reshape(-1)[torch.from_numpy(rows).cuda()],
                      o_ref, lse_ref, name)
