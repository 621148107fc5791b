"""GPU parity of the FP8 (E4M3) forward (C ABI attn_fwd_fp8) against the
fp64 oracle on the dequantized inputs, and its accuracy against unquantized
inputs at the synthetic coordinate of M4.6 0x06 ("What The Paper Actually
Reports": N(0,1) + N(0,100) Bernoulli(0.001) entries)."""
import math

import numpy as np
import pytest
import torch

from exact_tiled_attention_gb300 import attn_fwd_fp8, gbattn_device_status
from exact_tiled_attention_gb300.inputs import make_generator, make_prefill
from tests.fp8_util import oracle_fp8, quantize_per_kv_head
import oracle

pytestmark = pytest.mark.gpu


def _run(q, k, v, causal):
    Hkv = k.shape[1]
    q8, dq = quantize_per_kv_head(q, Hkv)
    k8, dk = quantize_per_kv_head(k, Hkv)
    v8, dv = quantize_per_kv_head(v, Hkv)
    scale = 1.0 / math.sqrt(q.shape[-1])
    o, lse = attn_fwd_fp8(q8, k8, v8, dq, dk, dv, scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert gbattn_device_status() == 0
    o_ref, lse_ref = oracle_fp8(q8, k8, v8, dq, dk, dv, scale, causal)
    vmax = float((v8.float().abs().amax(dim=(2, 3)) * dv).max())
    return o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, vmax


@pytest.mark.parametrize("shape", [
    (1, 4, 4, 128, 128, False),
    (1, 2, 2, 300, 300, True),
    (2, 4, 2, 257, 257, True),
    (1, 2, 2, 129, 700, False),
    (1, 2, 1, 200, 77, True),
    (1, 2, 2, 400, 200, True),  # the first query tile of the first pair sees no key
    (1, 1, 1, 1, 1, False),
])
def test_fp8_forward_vs_dequantized_oracle(shape):
    B, H, Hkv, Sq, Sk, causal = shape
    q, k, v = make_prefill(B, H, Hkv, Sq, Sk, 128, torch.bfloat16, 61, device="cuda")
    o, lse, o_ref, lse_ref, vmax = _run(q, k, v, causal)
    err = np.abs(o - o_ref)
    inf_ref = np.isneginf(lse_ref)
    assert (np.isneginf(lse) == inf_ref).all()
    lerr = np.abs(lse[~inf_ref] - lse_ref[~inf_ref]).max() if (~inf_ref).any() else 0.0
    print(f"{shape}: O max {err.max():.3e} mean {err.mean():.3e} (vmax {vmax:.2f}), LSE max {lerr:.3e}")
    assert np.isfinite(o).all()
    assert lerr <= 1e-3
    # every output is a convex combination of V rows whose weights the E4M3
    # rounding of P moves by at most 2^-4 relative, plus bf16 rounding
    assert err.max() <= 2.0 ** -4 * vmax + 2.0 ** -8 * np.abs(o_ref).max()
    assert err.mean() <= 2e-3 * vmax


def test_fp8_range_contract_near_threshold():
    """Key tile 1's scores exceed tile 0's by 3.57 log2 units, just under the
    rescale threshold 4, so the kernel keeps tile 0's reference and forms
    u = 2^(3.57 + 4) ~ 190 for tile 1: inside E4M3's 448 only because
    threshold + offset = 8 (M4.6 0x09, FP8 E4M3FN row).  A second case crosses
    the threshold (rescale).  Values are exact E4M3 codes, descales absent."""
    d, S = 128, 256
    for kval in (4.5, 5.0):
        q = torch.zeros(1, 1, 4, d)
        q[..., 0] = 8.0
        k = torch.zeros(1, 1, S, d)
        k[:, :, :128, 0] = 1.0
        k[:, :, 128:, 0] = kval
        g = make_generator(71, "cpu")
        v = torch.randn(1, 1, S, d, generator=g).clamp(-3, 3)
        q8, k8, v8 = (t.to(torch.float8_e4m3fn).cuda() for t in (q, k, v))
        scale = 1.0 / math.sqrt(d)
        o, lse = attn_fwd_fp8(q8, k8, v8, scale=scale)
        torch.cuda.synchronize()
        one = torch.ones(1, 1, device="cuda")
        o_ref, lse_ref = oracle_fp8(q8, k8, v8, one, one, one, scale, False)
        err = np.abs(o.float().cpu().numpy() - o_ref).max()
        assert err <= 2.0 ** -4 * 3 and np.abs(lse.cpu().numpy() - lse_ref).max() <= 1e-3, (kval, err)


def test_fp8_accuracy_at_page_coordinate():
    """Entries N(0,1) + N(0,100) Bernoulli(0.001) (the synthetic distribution
    of M4.6 0x06), quantized per (batch, KV head), against the fp64 oracle on
    the UNquantized values: the RMSE sits at the pages' per-tensor-scaled FP8
    figure (2.4e-2) or below, far above the 16-bit path's."""
    B, H, S, d = 1, 4, 1024, 128
    gen = make_generator(81, "cpu")

    def draw():
        x = torch.randn(B, H, S, d, generator=gen)
        spikes = torch.rand(B, H, S, d, generator=gen) < 1e-3
        return x + spikes * torch.randn(B, H, S, d, generator=gen) * 10.0

    q, k, v = draw(), draw(), draw()
    q8, dq = quantize_per_kv_head(q, H)
    k8, dk = quantize_per_kv_head(k, H)
    v8, dv = quantize_per_kv_head(v, H)
    scale = 1.0 / math.sqrt(d)
    o, _ = attn_fwd_fp8(q8.cuda(), k8.cuda(), v8.cuda(), dq.cuda(), dk.cuda(), dv.cuda(), scale=scale)
    torch.cuda.synchronize()
    o_ref, _ = oracle.attn_fwd(q.numpy(), k.numpy(), v.numpy(), scale, False)
    rmse = float(np.sqrt(np.mean((o.float().cpu().numpy() - o_ref) ** 2)))
    print(f"FP8 RMSE at the page coordinate: {rmse:.3e}")
    assert 1e-3 <= rmse <= 2.4e-2


def test_fp8_causal_workload_sampled_rows():
    """The causal [4, 16, 8192, 128] shape in E4M3, launched as the bench does,
    checked on sampled rows of every (batch, KV head) against the oracle."""
    B, H, S, d = 4, 16, 8192, 128
    q, k, v = make_prefill(B, H, H, S, S, d, torch.bfloat16, 3, device="cuda")
    q8, dq = quantize_per_kv_head(q, H)
    k8, dk = quantize_per_kv_head(k, H)
    v8, dv = quantize_per_kv_head(v, H)
    scale = 1.0 / math.sqrt(d)
    o, lse = attn_fwd_fp8(q8, k8, v8, dq, dk, dv, scale=scale, causal=True)
    torch.cuda.synchronize()
    assert gbattn_device_status() == 0 and torch.isfinite(o).all()
    rng = np.random.default_rng(3)
    qf, kf, vf = (t.float().cpu().numpy() for t in (q8, k8, v8))
    dqn, dkn, dvn = (t.double().cpu().numpy() for t in (dq, dk, dv))
    for bh in rng.choice(B * H, size=4, replace=False):
        b, h = divmod(int(bh), H)
        rows = np.unique(np.concatenate([rng.integers(0, S, 24), [0, 127, 128, S - 1]]))
        o_ref, l_ref = oracle.attn_fwd_rows(qf[b:b + 1, h:h + 1], kf[b:b + 1, h:h + 1], vf[b:b + 1, h:h + 1],
                                            scale * dqn[b, h] * dkn[b, h], True, rows)
        o_ref *= dvn[b, h]
        got = o[b, h, rows].float().cpu().numpy()
        vmax = float(np.abs(vf[b, h]).max() * dvn[b, h])
        assert np.abs(got - o_ref).max() <= 2.0 ** -4 * vmax + 2.0 ** -8 * np.abs(o_ref).max()
        assert np.abs(lse[b, h, rows].cpu().numpy() - l_ref).max() <= 1e-3
