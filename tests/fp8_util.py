"""Helpers for the FP8 (E4M3) forward tests: per-(batch, KV head) quantization
of test inputs and the fp64 oracle on the dequantized values."""
import numpy as np
import torch

import oracle

E4M3_MAX = 448.0


def quantize_per_kv_head(x, Hkv):
    """x [B, heads, S, d] (heads a multiple of Hkv) -> (E4M3 codes, descale
    [B, Hkv] fp32): one scale per (batch, KV head), shared by the heads of the
    group, so that the largest magnitude maps to 448."""
    B, Hx, S, d = x.shape
    g = Hx // Hkv
    xg = x.float().reshape(B, Hkv, g * S * d)
    amax = xg.abs().amax(dim=2).clamp_min(1e-12)
    descale = (amax / E4M3_MAX).float()
    codes = (x.float().reshape(B, Hkv, g, S, d) / descale[:, :, None, None, None]).reshape(B, Hx, S, d)
    return codes.to(torch.float8_e4m3fn).contiguous(), descale.contiguous()


def oracle_fp8(q8, k8, v8, dq, dk, dv, scale, causal):
    """Exact attention (fp64 oracle) on the dequantized inputs: per (b, KV
    head) the scores use scale * dq * dk on the E4M3 values and O is scaled
    by dv (the real values are code * descale)."""
    B, H, Sq, d = q8.shape
    Hkv = k8.shape[1]
    g = H // Hkv
    qf, kf, vf = (t.float().cpu().numpy() for t in (q8, k8, v8))
    dq, dk, dv = (t.double().cpu().numpy() for t in (dq, dk, dv))
    o = np.empty((B, H, Sq, d))
    lse = np.empty((B, H, Sq))
    for b in range(B):
        for kh in range(Hkv):
            sl = slice(kh * g, (kh + 1) * g)
            ob, lb = oracle.attn_fwd(qf[b:b + 1, sl], kf[b:b + 1, kh:kh + 1], vf[b:b + 1, kh:kh + 1],
                                     scale * dq[b, kh] * dk[b, kh], causal)
            o[b, sl] = ob[0] * dv[b, kh]
            lse[b, sl] = lb[0]
    return o, lse
