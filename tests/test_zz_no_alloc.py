"""attn_decode_splitkv_noalloc -- the decode entry point for callers that
cannot allocate device memory -- must give what attn_decode_splitkv gives
with a caller-provided workspace, on two calls in a row (the second with
different lengths, so stale partial states from the first call would show),
and must refuse problems larger than its fixed scratch array.

Collected last on purpose (file name), so a first failure here leaves every
other test already run; it also passes alone in a fresh process."""
import math

import numpy as np
import pytest
import torch

from exact_tiled_attention_gb300 import binding
from tests.parity_util import LSE_MAX_ABS, O_MAX_ABS, O_MEAN_ABS

pytestmark = pytest.mark.gpu


def _inputs(seed, B, Hq, Hkv, Skm, d, dt, lens):
    g = torch.Generator(device="cuda").manual_seed(seed)
    q = torch.randn(B, Hq, 1, d, generator=g, device="cuda").to(dt)
    k = torch.randn(B, Hkv, Skm, d, generator=g, device="cuda").to(dt)
    v = torch.randn(B, Hkv, Skm, d, generator=g, device="cuda").to(dt)
    return q, k, v, torch.tensor(lens, dtype=torch.int32, device="cuda")


def _noalloc_call(lib, q, k, v, sl, n_split):
    B, Hq, _, d = q.shape
    Hkv, Skm = k.shape[1], k.shape[2]
    o = torch.empty_like(q)
    lse = torch.empty(B, Hq, dtype=torch.float32, device="cuda")
    dt = 1 if q.dtype == torch.bfloat16 else 0
    rc = lib.attn_decode_splitkv_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), sl.data_ptr(),
                                         o.data_ptr(), lse.data_ptr(), B, Hq, Hkv, Skm, d,
                                         1.0 / math.sqrt(d), n_split, dt,
                                         torch.cuda.current_stream().cuda_stream)
    return rc, o, lse


def _close(o, lse, o_ref, lse_ref):
    err = (o.float() - o_ref.float()).abs()
    assert err.max().item() <= O_MAX_ABS and err.mean().item() <= O_MEAN_ABS
    assert (lse - lse_ref).abs().max().item() <= LSE_MAX_ABS


def test_noalloc_matches_workspace_entry_on_two_calls():
    lib = binding.load_library()
    # seed, B, Hq, Hkv, Sk_max, d, dtype, n_split
    cases = [
        (31, 8, 32, 8, 4096, 128, torch.bfloat16, 16),
        (32, 8, 32, 8, 4096, 128, torch.bfloat16, 16),
    ]
    rng = np.random.default_rng(3)
    for seed, B, Hq, Hkv, Skm, d, dt, n_split in cases:
        lens = rng.integers(1, Skm + 1, size=B).tolist()
        q, k, v, sl = _inputs(seed, B, Hq, Hkv, Skm, d, dt, lens)
        rc, o, lse = _noalloc_call(lib, q, k, v, sl, n_split)
        assert rc == 0, binding.error_string(rc)
        o_ref, lse_ref, _ = binding.attn_decode_splitkv(q, k, v, sl, n_split=n_split)
        torch.cuda.synchronize()
        assert binding.gbattn_device_status() == 0
        _close(o, lse, o_ref, lse_ref)


def test_noalloc_rejects_problems_larger_than_its_array():
    lib = binding.load_library()
    cap = lib.attn_decode_noalloc_scratch_bytes()
    assert cap == 32 << 20
    # B * Hq * n_split * (d + 2) * 4 bytes > 32 MiB
    B, Hq, Hkv, d, n_split = 256, 32, 8, 128, 16
    assert lib.attn_decode_workspace_bytes(B, Hq, n_split, d) > cap
    q, k, v, sl = _inputs(5, 1, Hq, Hkv, 16, d, torch.bfloat16, [16])
    rc = lib.attn_decode_splitkv_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), sl.data_ptr(),
                                         q.data_ptr(), None, B, Hq, Hkv, 16, d, 0.1, n_split, 1, None)
    assert rc == -6


def test_noalloc_at_the_64_sequence_workload_matches_the_oracle():
    """The 64-sequence, 32768-slot decode workload (17 MB of partial states,
    inside the fixed array) through the no-allocation entry point: every head
    of sampled sequences, including the shortest and longest, against the fp64
    oracle, and the whole result equal to the workspace entry point's."""
    import oracle
    from exact_tiled_attention_gb300.inputs import WORKLOADS, make_decode
    from tests.parity_util import assert_attn_close, host_f32

    w = WORKLOADS["decode_splitkv_bf16_b64_hq32_hkv8_sk32768_d128"]
    lib = binding.load_library()
    assert lib.attn_decode_workspace_bytes(w.B, w.H, w.n_split, w.d) <= lib.attn_decode_noalloc_scratch_bytes()
    q, k, v, sl = make_decode(w.B, w.H, w.Hkv, w.Sk, w.d, w.dtype, w.len_lo, w.len_hi, w.seed, device="cuda")
    rc, o, lse = _noalloc_call(lib, q, k, v, sl, w.n_split)
    assert rc == 0, binding.error_string(rc)
    torch.cuda.synchronize()
    assert binding.gbattn_device_status() == 0
    lens = sl.cpu().numpy()
    rng = np.random.default_rng(11)
    bs = sorted(set(rng.integers(0, w.B, size=6).tolist()) | {int(np.argmin(lens)), int(np.argmax(lens))})
    for b in bs:
        o_ref, lse_ref = oracle.attn_decode(host_f32(q[b:b + 1]), host_f32(k[b:b + 1]), host_f32(v[b:b + 1]),
                                            lens[b:b + 1], w.scale)
        assert_attn_close(o[b:b + 1], lse[b:b + 1], o_ref, lse_ref, f"no-alloc decode, batch {b}")
    o_ws, lse_ws, _ = binding.attn_decode_splitkv(q, k, v, sl, scale=w.scale, n_split=w.n_split)
    torch.cuda.synchronize()
    _close(o, lse, o_ws, lse_ws)
