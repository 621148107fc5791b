"""GPU checks that need no oracle, and the stream argument.

One-hot dominant rows (a closed form): with Q_i = c * K_{pi(i)} of
the query head's own KV head (h // (H / Hkv), M4.4 "FlashAttention-2 Work
Partitioning and the Decode Boundary" 0x06A) and pi(i) a visible key of row
i, the score of key pi(i) exceeds every other visible one by more than 30
(checked in the test), so O_i is
V_{pi(i)} and LSE_i is that score; a wrong head map or causal index moves
the output to another row of V."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_gb300 import (attn_bwd, attn_decode_splitkv, attn_fwd, attn_fwd_pair,
                                         gbattn_device_status)
from exact_tiled_attention_gb300.inputs import make_generator, make_prefill, randn
from tests.parity_util import assert_attn_close, assert_grad_close, grad_extras, host_f32

pytestmark = pytest.mark.gpu


def _one_hot_inputs(B, H, Hkv, S, d, causal, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    k = torch.randn(B, Hkv, S, d, generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn(B, Hkv, S, d, generator=g, device="cuda").to(torch.bfloat16)
    i = torch.arange(S, device="cuda")
    pi = (7 * i + 3) % (i + 1) if causal else (5 * i + 11) % S  # a visible key of row i
    kvh = torch.arange(H, device="cuda") // (H // Hkv)
    q = 16.0 * k[:, kvh][:, :, pi]  # power-of-two multiple: exact in bf16
    return q.contiguous(), k, v, pi, kvh


@pytest.mark.parametrize("causal,pair", [(True, False), (False, False), (False, True)])
def test_one_hot_rows_pick_their_value_row(causal, pair):
    B, H, Hkv, S, d = 2, 8, 2, 700, 128
    q, k, v, pi, kvh = _one_hot_inputs(B, H, Hkv, S, d, causal, 7)
    scale = 1.0 / math.sqrt(d)
    if pair:
        o, lse = attn_fwd_pair(q, k, v, scale=scale)
    else:
        o, lse = attn_fwd(q, k, v, scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert gbattn_device_status() == 0
    v_sel = v[:, kvh][:, :, pi].float()
    assert (o.float() - v_sel).abs().max().item() <= 2e-2
    s = scale * q.float() @ k[:, kvh].float().transpose(-1, -2)
    if causal:
        s = s.masked_fill(torch.ones(S, S, dtype=torch.bool, device="cuda").triu(1), float("-inf"))
    s_top = s.gather(-1, pi.view(1, 1, S, 1).expand(B, H, S, 1)).squeeze(-1)
    s_second = s.scatter(-1, pi.view(1, 1, S, 1).expand(B, H, S, 1), float("-inf")).amax(-1)
    gap = (s_top - s_second)[..., 1:] if causal else s_top - s_second  # row 0 sees one key
    assert gap.min().item() > 30.0
    assert (lse - s_top).abs().max().item() <= 1e-2


def test_calls_on_a_side_stream():
    """Every entry point runs on the stream it is given; results read after
    that stream synchronises match the oracle."""
    side = torch.cuda.Stream()
    q, k, v = make_prefill(1, 4, 2, 333, 333, 128, torch.bfloat16, 17, device="cuda")
    do = randn(q.shape, q.dtype, make_generator(18, "cuda"), "cuda")
    torch.cuda.synchronize()
    with torch.cuda.stream(side):
        o, lse = attn_fwd(q, k, v, causal=True, stream=side)
        dq, dk, dv = attn_bwd(q, k, v, o, lse, do, causal=True, stream=side)
    side.synchronize()
    assert gbattn_device_status() == 0
    scale = 1.0 / math.sqrt(128)
    o_ref, lse_ref = oracle.attn_fwd(host_f32(q), host_f32(k), host_f32(v), scale, True)
    assert_attn_close(o, lse, o_ref, lse_ref, "forward on a side stream")
    rq, rk, rv, _, _ = oracle.attn_bwd(host_f32(q), host_f32(k), host_f32(v), host_f32(do), scale, True)
    ex = grad_extras(host_f32(q), host_f32(k), host_f32(v), host_f32(do), scale, True)
    assert_grad_close(dq, rq, "dq on a side stream", extra=ex["dq"])
    assert_grad_close(dk, rk, "dk on a side stream", extra=ex["dk"])
    assert_grad_close(dv, rv, "dv on a side stream")
    g = torch.Generator(device="cuda").manual_seed(19)
    qd = torch.randn(2, 8, 1, 128, generator=g, device="cuda").to(torch.bfloat16)
    kc = torch.randn(2, 2, 500, 128, generator=g, device="cuda").to(torch.bfloat16)
    vc = torch.randn(2, 2, 500, 128, generator=g, device="cuda").to(torch.bfloat16)
    lens = [500, 123]
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    with torch.cuda.stream(side):
        od, lsed, _ = attn_decode_splitkv(qd, kc, vc, sl, n_split=4, stream=side)
    side.synchronize()
    o_ref, lse_ref = oracle.attn_decode(host_f32(qd), host_f32(kc), host_f32(vc), np.array(lens, np.int32), scale)
    assert_attn_close(od, lsed, o_ref, lse_ref, "decode on a side stream")
