"""GPU parity of split-KV decode (C ABI attn_decode_splitkv) against the fp64
oracle: final O and LSE, and every chunk's partial state in the workspace
(compared as the chunk output o/l and the chunk LSE m + log l, which do not
depend on the retained reference the kernel kept)."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_gb300 import attn_decode_splitkv, gbattn_device_status
from exact_tiled_attention_gb300.inputs import WORKLOADS, make_decode
from tests.parity_util import LSE_MAX_ABS, O_MAX_ABS, O_MEAN_ABS, assert_attn_close, host_f32

pytestmark = pytest.mark.gpu


def _partials_from_workspace(ws, B, Hq, n, d):
    f = ws.view(torch.float32)
    n_states = B * Hq * n
    o = f[: n_states * d].view(B, Hq, n, d).double().cpu().numpy()
    ml = f[n_states * d: n_states * (d + 2)].view(B, Hq, n, 2).double().cpu().numpy()
    return o, ml[..., 0], ml[..., 1]


def _check_partials(ws, q, k, v, lens, scale, n_split):
    B, Hq, _, d = q.shape
    o_ws, m_ws, l_ws = _partials_from_workspace(ws, B, Hq, n_split, d)
    m, l, u, cnt = oracle.decode_chunk_states(host_f32(q), host_f32(k), host_f32(v), lens, scale, n_split)
    valid = cnt > 0
    assert ((l_ws > 0) == valid).all(), "empty-chunk pattern differs"
    assert np.isneginf(m_ws[~valid]).all() and (o_ws[~valid] == 0).all()
    chunk_o = o_ws[valid] / l_ws[valid][:, None]
    chunk_o_ref = u[valid] / l[valid][:, None]
    err = np.abs(chunk_o - chunk_o_ref)
    assert err.max() <= O_MAX_ABS and err.mean() <= O_MEAN_ABS
    lse_c = m_ws[valid] + np.log(l_ws[valid])
    lse_c_ref = m[valid] + np.log(l[valid])
    assert np.abs(lse_c - lse_c_ref).max() <= LSE_MAX_ABS


@pytest.mark.parametrize("cfg", [
    # B, Hq, Hkv, Sk_max, d, dtype, lens, n_split
    (3, 8, 2, 300, 128, torch.bfloat16, [1, 77, 300], 4),
    (3, 8, 2, 300, 128, torch.bfloat16, [1, 77, 300], 16),   # empty chunks for L < 16
    (2, 16, 1, 1000, 64, torch.float16, [999, 1000], 7),     # MQA, g = 16
    (2, 32, 1, 500, 128, torch.bfloat16, [130, 500], 3),     # g = 32: two head groups
    (4, 4, 4, 2049, 128, torch.float16, [2049, 64, 65, 1000], 16),
    (1, 4, 2, 64, 64, torch.bfloat16, [64], 1),
])
def test_decode_small(cfg):
    B, Hq, Hkv, Skm, d, dt, lens, n_split = cfg
    g = torch.Generator(device="cuda").manual_seed(21)
    q = torch.randn(B, Hq, 1, d, generator=g, device="cuda").to(dt)
    k = torch.randn(B, Hkv, Skm, d, generator=g, device="cuda").to(dt)
    v = torch.randn(B, Hkv, Skm, d, generator=g, device="cuda").to(dt)
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    scale = 1.0 / math.sqrt(d)
    o, lse, ws = attn_decode_splitkv(q, k, v, sl, scale=scale, n_split=n_split)
    torch.cuda.synchronize()
    assert gbattn_device_status() == 0
    lens_np = np.array(lens, np.int32)
    o_ref, lse_ref = oracle.attn_decode(host_f32(q), host_f32(k), host_f32(v), lens_np, scale)
    assert_attn_close(o, lse, o_ref, lse_ref, str(cfg))
    _check_partials(ws, q, k, v, lens_np, scale, n_split)


def test_decode_padding_is_never_read():
    """Rows past each sequence's valid length hold NaN: the result must equal
    the result over clean padding, bit for bit."""
    B, Hq, Hkv, Skm, d = 4, 8, 2, 700, 128
    g = torch.Generator(device="cuda").manual_seed(5)
    q = torch.randn(B, Hq, 1, d, generator=g, device="cuda").to(torch.bfloat16)
    k = torch.randn(B, Hkv, Skm, d, generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn(B, Hkv, Skm, d, generator=g, device="cuda").to(torch.bfloat16)
    lens = [1, 333, 699, 700]
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    o1, l1, _ = attn_decode_splitkv(q, k, v, sl, n_split=16)
    kn, vn = k.clone(), v.clone()
    for b, L in enumerate(lens):
        kn[b, :, L:] = float("nan")
        vn[b, :, L:] = float("nan")
    o2, l2, _ = attn_decode_splitkv(q, kn, vn, sl, n_split=16)
    torch.cuda.synchronize()
    assert torch.isfinite(o2).all() and torch.isfinite(l2).all()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_decode_workload_sampled_batches():
    """The 64-sequence, 32768-slot decode workload as the bench launches it;
    every head of 8 sampled sequences against the oracle, and the chunk
    partial states of those sequences."""
    w = WORKLOADS["decode_splitkv_bf16_b64_hq32_hkv8_sk32768_d128"]
    q, k, v, sl = make_decode(w.B, w.H, w.Hkv, w.Sk, w.d, w.dtype, w.len_lo, w.len_hi, w.seed,
                              device="cuda")
    o, lse, ws = attn_decode_splitkv(q, k, v, sl, scale=w.scale, n_split=w.n_split)
    torch.cuda.synchronize()
    assert gbattn_device_status() == 0
    assert torch.isfinite(o).all()
    lens = sl.cpu().numpy()
    rng = np.random.default_rng(7)
    bs = sorted(set(rng.integers(0, w.B, size=8).tolist()) | {int(np.argmin(lens)), int(np.argmax(lens))})
    for b in bs:
        qb, kb, vb = q[b:b + 1], k[b:b + 1], v[b:b + 1]
        o_ref, lse_ref = oracle.attn_decode(host_f32(qb), host_f32(kb), host_f32(vb), lens[b:b + 1], w.scale)
        assert_attn_close(o[b:b + 1], lse[b:b + 1], o_ref, lse_ref, f"batch {b}")
    # chunk partials of the first sampled sequence
    b = bs[0]
    full_ws = ws.view(torch.float32)
    n_states = w.B * w.H * w.n_split
    o_all = full_ws[: n_states * w.d].view(w.B, w.H, w.n_split, w.d)[b:b + 1]
    ml_all = full_ws[n_states * w.d: n_states * (w.d + 2)].view(w.B, w.H, w.n_split, 2)[b:b + 1]
    sub = torch.cat([o_all.reshape(-1), ml_all.reshape(-1)]).contiguous()
    _check_partials(sub.view(torch.uint8), q[b:b + 1], k[b:b + 1], v[b:b + 1], lens[b:b + 1], w.scale,
                    w.n_split)
