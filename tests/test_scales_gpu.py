"""Every GPU path with a softmax scale other than 1/sqrt(d): the scale
multiplies the fp32 dot product before masking and softmax (M4.3 "IO-Aware
Attention and FlashAttention-1" 0x02A), so a kernel that assumed 1/sqrt(d)
would fail here.  Large scales make the attention nearly one-hot, which also
drives the conditional rescale (threshold in base-2 units) on most rows."""
import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_gb300 import (attn_bwd, attn_decode_splitkv, attn_fwd, attn_fwd_fp8, attn_fwd_pair,
                                         gbattn_device_status)
from exact_tiled_attention_gb300.inputs import make_generator, make_prefill, randn
from tests.fp8_util import oracle_fp8, quantize_per_kv_head
from tests.parity_util import assert_attn_close, assert_grad_close, grad_extras, host_f32

pytestmark = pytest.mark.gpu

SCALES = [0.03, 0.6, 2.0]


@pytest.mark.parametrize("scale", SCALES)
@pytest.mark.parametrize("d,dt,causal", [(128, torch.bfloat16, True), (64, torch.float16, False)])
def test_forward_scales(scale, d, dt, causal):
    q, k, v = make_prefill(1, 4, 2, 300, 333, d, dt, 41, device="cuda")
    o, lse = attn_fwd(q, k, v, scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert gbattn_device_status() == 0
    o_ref, lse_ref = oracle.attn_fwd(host_f32(q), host_f32(k), host_f32(v), scale, causal)
    assert_attn_close(o, lse, o_ref, lse_ref, f"forward scale {scale} d {d}")


@pytest.mark.parametrize("scale", SCALES)
def test_pair_scales(scale):
    q, k, v = make_prefill(1, 2, 2, 600, 450, 128, torch.bfloat16, 42, device="cuda")
    o, lse = attn_fwd_pair(q, k, v, scale=scale)
    torch.cuda.synchronize()
    assert gbattn_device_status() == 0
    o_ref, lse_ref = oracle.attn_fwd(host_f32(q), host_f32(k), host_f32(v), scale, False)
    assert_attn_close(o, lse, o_ref, lse_ref, f"pair scale {scale}")


@pytest.mark.parametrize("scale", [0.05, 0.9])
@pytest.mark.parametrize("d,dt,causal", [(128, torch.bfloat16, True), (64, torch.float16, False)])
def test_backward_scales(scale, d, dt, causal):
    q, k, v = make_prefill(1, 4, 2, 260, 300, d, dt, 43, device="cuda")
    do = randn(q.shape, dt, make_generator(44, "cuda"), "cuda")
    o, lse = attn_fwd(q, k, v, scale=scale, causal=causal)
    dq, dk, dv = attn_bwd(q, k, v, o, lse, do, scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert gbattn_device_status() == 0
    rq, rk, rv, _, _ = oracle.attn_bwd(host_f32(q), host_f32(k), host_f32(v), host_f32(do), scale, causal)
    ex = grad_extras(host_f32(q), host_f32(k), host_f32(v), host_f32(do), scale, causal)
    assert_grad_close(dq, rq, f"dq scale {scale} d {d}", extra=ex["dq"])
    assert_grad_close(dk, rk, f"dk scale {scale} d {d}", extra=ex["dk"])
    assert_grad_close(dv, rv, f"dv scale {scale} d {d}")


@pytest.mark.parametrize("scale", SCALES)
def test_decode_scales(scale):
    g = torch.Generator(device="cuda").manual_seed(45)
    q = torch.randn(2, 8, 1, 128, generator=g, device="cuda").to(torch.bfloat16)
    k = torch.randn(2, 2, 700, 128, generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn(2, 2, 700, 128, generator=g, device="cuda").to(torch.bfloat16)
    lens = [700, 333]
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    o, lse, _ = attn_decode_splitkv(q, k, v, sl, scale=scale, n_split=5)
    torch.cuda.synchronize()
    assert gbattn_device_status() == 0
    o_ref, lse_ref = oracle.attn_decode(host_f32(q), host_f32(k), host_f32(v), np.array(lens, np.int32), scale)
    assert_attn_close(o, lse, o_ref, lse_ref, f"decode scale {scale}")


@pytest.mark.parametrize("scale", [0.03, 0.4])
def test_fp8_scales(scale):
    q, k, v = make_prefill(1, 4, 2, 300, 300, 128, torch.bfloat16, 46, device="cuda")
    q8, dq = quantize_per_kv_head(q, 2)
    k8, dk = quantize_per_kv_head(k, 2)
    v8, dv = quantize_per_kv_head(v, 2)
    o, lse = attn_fwd_fp8(q8, k8, v8, dq, dk, dv, scale=scale, causal=True)
    torch.cuda.synchronize()
    assert gbattn_device_status() == 0
    o_ref, lse_ref = oracle_fp8(q8, k8, v8, dq, dk, dv, scale, True)
    o = o.float().cpu().numpy()
    lse = lse.cpu().numpy()
    vmax = float((v8.float().abs().amax(dim=(2, 3)) * dv).max())
    # the bounds of the FP8 parity tests: the E4M3 rounding of P moves each
    # weight by at most 2^-4 relative, plus bf16 rounding of O
    assert np.isfinite(o).all()
    assert np.abs(o - o_ref).max() <= 2.0 ** -4 * vmax + 2.0 ** -8 * np.abs(o_ref).max()
    assert np.abs(lse - lse_ref).max() <= 1e-3
