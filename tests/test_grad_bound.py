"""The backward's error bound (tests/parity_util.py) pinned on the CPU: an
fp64 emulation of the kernels' arithmetic -- P and dS rounded to the input
dtype before their products, O stored in the dtype and D = dO . O taken from
it, every gradient rounded to the dtype -- stays inside the bound, with
margin, on causal GQA problems (including a peaked softmax, where the D term
dominates dQ); and gradients with a plausible mistake (D dropped, the scale
missing from dK, the wrong KV head) fall outside it."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_gb300.inputs import make_generator, make_prefill, randn
from tests.parity_util import GRAD_LOG, assert_grad_close, grad_extras


def _rn(x, dtype):
    return torch.from_numpy(np.ascontiguousarray(x)).to(dtype).double().numpy()


def _emulated_bwd(q, k, v, do, scale, causal, dtype, mistake=None):
    """Gradients computed the way the kernels compute them, in fp64 with the
    kernels' roundings; `mistake` plants one error."""
    B, H, Sq, d = q.shape
    Hkv, Sk = k.shape[1], k.shape[2]
    g = H // Hkv
    kv_of = (lambda h: h % Hkv) if mistake == "head_map" else (lambda h: h // g)
    dq = np.zeros(q.shape)
    dk = np.zeros(k.shape)
    dv = np.zeros(v.shape)
    for b in range(B):
        for h in range(H):
            kvh = kv_of(h)
            s = scale * q[b, h] @ k[b, kvh].T
            if causal:
                s = np.where(np.arange(Sk)[None, :] <= np.arange(Sq)[:, None] + (Sk - Sq), s, -np.inf)
            m = s.max(axis=1, keepdims=True)
            m = np.where(np.isfinite(m), m, 0.0)
            p = np.exp(s - m)
            lsum = p.sum(axis=1, keepdims=True)
            p = np.where(lsum > 0, p / np.where(lsum > 0, lsum, 1.0), 0.0)
            o_st = _rn(p @ v[b, kvh], dtype)                       # the stored output
            dd = np.zeros((Sq, 1)) if mistake == "drop_D" else (do[b, h] * o_st).sum(axis=1, keepdims=True)
            dp = do[b, h] @ v[b, kvh].T
            ds = _rn(p * (dp - dd), dtype)
            dq[b, h] = scale * ds @ k[b, kvh]
            dk[b, kvh] += (1.0 if mistake == "no_scale_dk" else scale) * ds.T @ q[b, h]
            dv[b, kvh] += _rn(p, dtype).T @ do[b, h]
    return _rn(dq, dtype), _rn(dk, dtype), _rn(dv, dtype)


CASES = [
    # B, H, Hkv, S, d, dtype, causal, scale
    (1, 4, 2, 200, 64, torch.bfloat16, True, None),
    (1, 2, 1, 160, 128, torch.float16, True, None),
    (1, 2, 2, 96, 64, torch.bfloat16, False, 0.9),   # peaked softmax: the D term dominates dQ
]


@pytest.mark.parametrize("case", CASES)
def test_emulated_kernel_arithmetic_is_inside_the_bound(case):
    B, H, Hkv, S, d, dtype, causal, scale = case
    scale = scale or 1.0 / math.sqrt(d)
    q, k, v = (t.float().numpy() for t in make_prefill(B, H, Hkv, S, S, d, dtype, 61))
    do = randn((B, H, S, d), dtype, make_generator(62, "cpu"), "cpu").float().numpy()
    rq, rk, rv, _, _ = oracle.attn_bwd(q, k, v, do, scale, causal)
    ex = grad_extras(q, k, v, do, scale, causal)
    gq, gk, gv = _emulated_bwd(q.astype(np.float64), k.astype(np.float64), v.astype(np.float64),
                               do.astype(np.float64), scale, causal, dtype)
    used = []
    used.append(assert_grad_close(gq, rq, f"emulated dq {case}", dtype=dtype, extra=ex["dq"])[1])
    used.append(assert_grad_close(gk, rk, f"emulated dk {case}", dtype=dtype, extra=ex["dk"])[1])
    used.append(assert_grad_close(gv, rv, f"emulated dv {case}", dtype=dtype)[1])
    assert max(used) < 0.75, f"the emulated arithmetic uses {max(used):.2f} of the bound"


@pytest.mark.parametrize("mistake,which", [("drop_D", 0), ("no_scale_dk", 1), ("head_map", 2)])
def test_planted_mistakes_fall_outside_the_bound(mistake, which):
    B, H, Hkv, S, d, dtype = 1, 4, 2, 200, 64, torch.bfloat16
    scale = 1.0 / math.sqrt(d)
    q, k, v = (t.float().numpy() for t in make_prefill(B, H, Hkv, S, S, d, dtype, 63))
    do = randn((B, H, S, d), dtype, make_generator(64, "cpu"), "cpu").float().numpy()
    refs = oracle.attn_bwd(q, k, v, do, scale, True)[:3]
    ex = grad_extras(q, k, v, do, scale, True)
    grads = _emulated_bwd(q.astype(np.float64), k.astype(np.float64), v.astype(np.float64), do.astype(np.float64),
                          scale, True, dtype, mistake=mistake)
    extra = [ex["dq"], ex["dk"], None][which]
    n = len(GRAD_LOG)
    with pytest.raises(AssertionError):
        assert_grad_close(grads[which], refs[which], f"planted {mistake}", dtype=dtype, extra=extra)
    del GRAD_LOG[n:]
