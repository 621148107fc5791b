"""Pins of the fp64 backward oracle (oracle.attn_bwd) to things other than
itself: a library autograd of the materialised softmax, central finite
differences of the forward oracle, the saved-output identity D_i = dO_i . O_i
that M4.4 "FlashAttention-2 Work Partitioning and the Decode Boundary" 0x06.1A
derives, and closed forms / invariants that a dropped term, a wrong sign, a
swapped index or a transposed operand would break."""
import math

import numpy as np
import pytest
import torch

import oracle


def _inputs(B, H, Hkv, Sq, Sk, d, seed, dtype=np.float32):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, H, Sq, d)).astype(dtype)
    k = rng.standard_normal((B, Hkv, Sk, d)).astype(dtype)
    v = rng.standard_normal((B, Hkv, Sk, d)).astype(dtype)
    do = rng.standard_normal((B, H, Sq, d)).astype(dtype)
    return q, k, v, do


def _autograd(q, k, v, do, scale, causal):
    """torch fp64 autograd through an explicitly materialised softmax, with
    the K/V heads expanded by repeat_interleave (its backward sums the group)
    and the bottom-right causal mask from tril."""
    B, H, Sq, d = q.shape
    Hkv, Sk = k.shape[1], k.shape[2]
    Q = torch.tensor(q, dtype=torch.float64, requires_grad=True)
    K = torch.tensor(k, dtype=torch.float64, requires_grad=True)
    V = torch.tensor(v, dtype=torch.float64, requires_grad=True)
    Kr, Vr = K.repeat_interleave(H // Hkv, dim=1), V.repeat_interleave(H // Hkv, dim=1)
    S = scale * Q @ Kr.transpose(-1, -2)
    if causal:
        vis = torch.ones(Sq, Sk, dtype=torch.bool).tril(diagonal=Sk - Sq)
        S = S.masked_fill(~vis, float("-inf"))
    P = torch.softmax(S, dim=-1)
    P = torch.nan_to_num(P, nan=0.0)  # rows with no visible key: zero payload
    O = P @ Vr
    O.backward(torch.tensor(do, dtype=torch.float64))
    return Q.grad.numpy(), K.grad.numpy(), V.grad.numpy()


@pytest.mark.parametrize("shape", [
    (1, 1, 1, 6, 6, 4, False),
    (1, 4, 2, 7, 9, 5, False),    # GQA g = 2, Sq != Sk
    (2, 4, 1, 9, 9, 8, True),     # MQA, causal square
    (1, 2, 2, 5, 11, 3, True),    # causal Sq < Sk (bottom-right)
    (1, 3, 3, 10, 4, 6, False),
])
def test_bwd_matches_library_autograd(shape):
    B, H, Hkv, Sq, Sk, d, causal = shape
    q, k, v, do = _inputs(B, H, Hkv, Sq, Sk, d, seed=sum(shape[:6]))
    scale = 1.0 / math.sqrt(d)
    dq, dk, dv, _, _ = oracle.attn_bwd(q, k, v, do, scale, causal)
    gq, gk, gv = _autograd(q, k, v, do, scale, causal)
    assert np.abs(dq - gq).max() <= 1e-12
    assert np.abs(dk - gk).max() <= 1e-12
    assert np.abs(dv - gv).max() <= 1e-12


def test_bwd_rows_without_keys():
    """Causal with Sq > Sk: rows i < Sq - Sk see no key (M4.4 0x05.1F); they
    get dQ = 0, LSE = -inf and contribute nothing to dK, dV."""
    q, k, v, do = _inputs(1, 2, 1, 8, 3, 4, seed=5)
    dq, dk, dv, D, lse = oracle.attn_bwd(q, k, v, do, 0.5, True)
    assert (dq[:, :, :5] == 0).all() and np.isneginf(lse[:, :, :5]).all() and (D[:, :, :5] == 0).all()
    gq, gk, gv = _autograd(q, k, v, do, 0.5, True)
    assert np.abs(dq - gq).max() <= 1e-12 and np.abs(dk - gk).max() <= 1e-12
    assert np.abs(dv - gv).max() <= 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_central_differences(causal):
    """<dX, E> equals the central difference of L = sum(dO * O(X)) along a
    random direction E, with O from the forward oracle (fp64 throughout)."""
    B, H, Hkv, Sq, Sk, d = 1, 4, 2, 6, 6, 4
    q, k, v, do = _inputs(B, H, Hkv, Sq, Sk, d, seed=17, dtype=np.float64)
    # The forward oracle reads binary32.  Inputs on a 2^-6 grid, directions on
    # a 2^-3 grid and the step h = 2^-12 keep X +/- hE exact in binary32
    # (|X| < 8 needs 18 significant bits).
    q, k, v = (np.clip(np.round(t * 64) / 64, -7.5, 7.5) for t in (q, k, v))
    do = do.astype(np.float32).astype(np.float64)
    scale = 0.7
    rng = np.random.default_rng(3)
    h = 2.0 ** -12

    def loss(qq, kk, vv):
        o, _ = oracle.attn_fwd(qq, kk, vv, scale, causal)
        return float(np.sum(o * do))

    grads = dict(zip("qkv", oracle.attn_bwd(q, k, v, do, scale, causal)[:3]))
    for which in "qkv":
        x = {"q": q, "k": k, "v": v}
        E = np.round(rng.standard_normal(x[which].shape) * 8) / 8
        xp, xm = dict(x), dict(x)
        xp[which] = x[which] + h * E
        xm[which] = x[which] - h * E
        for t in (xp[which], xm[which]):
            assert np.array_equal(t.astype(np.float32).astype(np.float64), t)
        fd = (loss(xp["q"], xp["k"], xp["v"]) - loss(xm["q"], xm["k"], xm["v"])) / (2 * h)
        an = float(np.sum(grads[which] * E))
        assert abs(fd - an) <= 1e-5 * max(1.0, abs(an)), (which, fd, an)


def test_row_scalar_equals_saved_output_identity():
    """M4.4 0x06.1A: sum_k P_ik dP_ik = dO_i . O_i (the oracle computes the
    left side; the forward oracle gives O)."""
    q, k, v, do = _inputs(2, 4, 2, 33, 40, 16, seed=8)
    for causal in (False, True):
        _, _, _, D, _ = oracle.attn_bwd(q, k, v, do, 0.25, causal)
        o, _ = oracle.attn_fwd(q, k, v, 0.25, causal)
        assert np.abs(D - np.sum(do.astype(np.float64) * o, axis=-1)).max() <= 1e-12


def test_constant_values_zero_query_and_key_gradients():
    """All V rows equal: O = V_0 whatever P is, so dQ = dK = 0 and every
    visible row passes its whole dO to dV: sum_j dV_j = sum_i dO_i."""
    q, k, v, do = _inputs(1, 4, 2, 12, 12, 8, seed=2)
    v[:] = v[:, :, :1, :]
    for causal in (False, True):
        dq, dk, dv, _, _ = oracle.attn_bwd(q, k, v, do, 0.35, causal)
        assert np.abs(dq).max() <= 1e-13 and np.abs(dk).max() <= 1e-13
        col = dv.sum(axis=2)                                   # [B, Hkv, d]
        ref = do.astype(np.float64).reshape(1, 2, 2, 12, 8).sum(axis=(2, 3))
        assert np.abs(col - ref).max() <= 1e-12


def test_key_gradient_sums_to_zero():
    """Each row of dS sums to zero (sum_j P_ij (dP_ij - D_i) = D_i - D_i), so
    sum_j dK_j = tau sum_i (sum_j dS_ij) Q_i = 0 per KV head; a dropped D term
    breaks this."""
    q, k, v, do = _inputs(2, 6, 3, 20, 31, 8, seed=4)
    for causal in (False, True):
        _, dk, _, _, _ = oracle.attn_bwd(q, k, v, do, 0.4, causal)
        assert np.abs(dk.sum(axis=2)).max() <= 1e-12


def test_single_key():
    """Sk = 1: P = 1, so dS = 0 (dQ = dK = 0) and dV_0 = sum_i dO_i."""
    q, k, v, do = _inputs(1, 2, 1, 9, 1, 4, seed=6)
    dq, dk, dv, _, _ = oracle.attn_bwd(q, k, v, do, 1.0, False)
    assert np.abs(dq).max() <= 1e-14 and np.abs(dk).max() <= 1e-14
    assert np.abs(dv[0, 0, 0] - do.astype(np.float64).sum(axis=(1, 2))[0]).max() <= 1e-12


def test_linear_in_output_gradient():
    q, k, v, do = _inputs(1, 2, 2, 8, 8, 4, seed=9)
    a = oracle.attn_bwd(q, k, v, do, 0.5, True)[:3]
    b = oracle.attn_bwd(q, k, v, (2 * do).astype(np.float32), 0.5, True)[:3]
    for x, y in zip(a, b):
        assert np.abs(2 * x - y).max() <= 1e-12


def test_kvhead_restriction_equals_full():
    q, k, v, do = _inputs(2, 8, 2, 10, 14, 8, seed=12)
    dq, dk, dv, _, _ = oracle.attn_bwd(q, k, v, do, 0.3, True)
    ids = [3, 0]  # (b=1, kvh=1), (b=0, kvh=0)
    sq, sk, sv = oracle.attn_bwd_kvheads(q, k, v, do, 0.3, True, ids)
    for r, kid in enumerate(ids):
        b, kvh = divmod(kid, 2)
        assert np.array_equal(sq[r], dq[b, kvh * 4:(kvh + 1) * 4])
        assert np.array_equal(sk[r], dk[b, kvh]) and np.array_equal(sv[r], dv[b, kvh])
