"""Pins for the fp64 oracle: page-printed traces, closed forms, invariants and
independent library routines.  No GPU; these run in seconds.

Every check here compares the oracle with something other than itself, so a
dropped term, a wrong sign, a wrong head/causal index or a transposed operand
in oracle/attn_oracle.c or oracle/state.py fails at least one of them.
"""
import itertools
import math
import random

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from oracle import state as st


# ---------------------------------------------------------------------------
# Page-printed worked traces
# ---------------------------------------------------------------------------

def test_two_block_trace(golden):
    """M4.4 0x02E: block states and their union, printed to 6 decimals."""
    fx = golden("two_block_trace.json")
    tol = fx["print_tolerance"]
    A = st.block_state(fx["block_A"]["scores"], fx["block_A"]["values"])
    Bs = st.block_state(fx["block_B"]["scores"], fx["block_B"]["values"])
    U = st.merge(A, Bs)
    for s, key in ((A, "A"), (Bs, "B"), (U, "union")):
        exp = fx["expected"][key]
        O, _ = st.finalize(s)
        assert abs(s.m - exp["m"]) <= tol
        assert abs(s.l - exp["l"]) <= tol
        np.testing.assert_allclose(s.u, exp["u"], atol=tol, rtol=0)
        np.testing.assert_allclose(O, exp["O"], atol=tol, rtol=0)
    assert U.n == 5


def test_three_block_trace_state_algebra(golden):
    """M4.3 0x11 / 0x09G: every fold order reaches the printed dense state."""
    fx = golden("three_block_trace.json")
    s = np.array(fx["scores"], float)
    v = np.array(fx["values"], float)
    blocks = [st.block_state(s[b], v[b]) for b in fx["blocks"]]
    first = st.merge(blocks[0], blocks[1])
    e1 = fx["expected"]["after_first_merge"]
    assert abs(first.l - e1["l"]) <= fx["print_tolerance"]
    np.testing.assert_allclose(first.u, e1["u"], atol=fx["print_tolerance"], rtol=0)
    assert abs(math.exp(blocks[0].m - first.m) - e1["alpha"]) <= fx["print_tolerance"]

    dense = fx["expected"]["dense"]
    tol = fx["dense_tolerance"]
    for order in itertools.permutations(range(3)):
        for folder in (st.fold_sequential, st.fold_balanced):
            S = folder([blocks[i] for i in order])
            O, lse = st.finalize(S)
            assert S.m == dense["m"] and S.n == 5
            assert abs(S.l - dense["l"]) <= tol
            np.testing.assert_allclose(S.u, dense["u"], atol=tol, rtol=0)
            np.testing.assert_allclose(O, dense["O"], atol=tol, rtol=0)
            assert abs(lse - dense["LSE"]) <= tol
    # The (LSE, O) log-domain merge form reaches the same row.
    L, O = -math.inf, np.zeros(2)
    for b in blocks:
        Ob, Lb = st.finalize(b)
        L, O = st.lse_merge(L, O, Lb, Ob)
    np.testing.assert_allclose(O, dense["O"], atol=tol, rtol=0)
    assert abs(L - dense["LSE"]) <= tol


def test_three_block_trace_c_oracle(golden):
    """The dense C oracle reproduces the printed row: embed the scores as
    q = [1, 0], k_j = [s_j, 0] with scale 1 and the 2-wide payloads as V."""
    fx = golden("three_block_trace.json")
    s = np.array(fx["scores"], np.float32)
    q = np.array([1, 0], np.float32).reshape(1, 1, 1, 2)
    k = np.stack([s, np.zeros_like(s)], axis=1).reshape(1, 1, 5, 2)
    v = np.array(fx["values"], np.float32).reshape(1, 1, 5, 2)
    o, lse = oracle.attn_fwd(q, k, v, 1.0, False)
    dense = fx["expected"]["dense"]
    np.testing.assert_allclose(o[0, 0, 0], dense["O"], atol=1e-12, rtol=0)
    assert abs(lse[0, 0, 0] - dense["LSE"]) <= 1e-12


def test_naive_block_softmax_trap(golden):
    """M4.3 0x09H: the global answer is 99.99101163, not 101 nor 50.5."""
    fx = golden("naive_trap.json")
    states = [st.block_state(b["scores"], b["values"]) for b in fx["blocks"]]
    O, _ = st.finalize(st.merge(*states))
    assert abs(O[0] - fx["expected_global"]) <= fx["print_tolerance"]
    local = [st.finalize(s)[0][0] for s in states]
    assert sum(local) == fx["wrong_local_sum"] and np.mean(local) == fx["wrong_local_mean"]
    # Same through the C oracle with d = 1, scale = 1.
    q = np.ones((1, 1, 1, 1), np.float32)
    k = np.array([0, 0, 10], np.float32).reshape(1, 1, 3, 1)
    v = np.array([1, 1, 100], np.float32).reshape(1, 1, 3, 1)
    o, _ = oracle.attn_fwd(q, k, v, 1.0, False)
    assert abs(o[0, 0, 0, 0] - fx["expected_global"]) <= fx["print_tolerance"]


def test_safe_softmax_no_overflow(golden):
    """M4.3 0x06B: [1000, 999, -1000] has d_safe ~= 1.367879 and no overflow."""
    fx = golden("safe_softmax.json")
    with np.errstate(over="raise", invalid="raise"):
        S = st.block_state(fx["row"], np.zeros((3, 1)))
    assert S.m == 1000.0
    assert abs(S.l - fx["expected_d_safe"]) <= fx["print_tolerance"]
    q = np.ones((1, 1, 1, 1), np.float32)
    k = np.array(fx["row"], np.float32).reshape(1, 1, 3, 1)
    v = np.array([1, 2, 3], np.float32).reshape(1, 1, 3, 1)
    o, lse = oracle.attn_fwd(q, k, v, 1.0, False)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    assert abs(lse[0, 0, 0] - (1000.0 + math.log(fx["expected_d_safe"]))) <= 1e-6


def test_equal_score_witnesses(golden):
    """M4.3 0x08G / M4.4 0x02F: with equal scores the exact output is the
    payload mean, 0.5 for both adversarial rows; fp64 gets it exactly."""
    fx = golden("adversarial_equal_scores.json")
    for case in fx["cases"]:
        n = len(case["values"])
        q = np.zeros((1, 1, 1, 1), np.float32)
        k = np.ones((1, 1, n, 1), np.float32)
        v = np.array(case["values"], np.float32).reshape(1, 1, n, 1)
        o, lse = oracle.attn_fwd(q, k, v, 0.125, False)
        assert o[0, 0, 0, 0] == case["exact_output"]
        assert abs(lse[0, 0, 0] - math.log(n)) <= 1e-15


# ---------------------------------------------------------------------------
# State algebra invariants (M4.3 0x08C-0x08F)
# ---------------------------------------------------------------------------

def test_identity_and_masked_blocks():
    rng = np.random.default_rng(0)
    S = st.block_state(rng.normal(size=5), rng.normal(size=(5, 3)))
    e = st.State.empty(3)
    with np.errstate(all="raise"):
        for r in (st.merge(e, S), st.merge(S, e)):
            assert r.valid and r.m == S.m and r.l == S.l and r.n == S.n
            np.testing.assert_array_equal(r.u, S.u)
        masked = st.block_state([-math.inf, -math.inf], rng.normal(size=(2, 3)))
        assert not masked.valid and masked.l == 0 and masked.n == 0
        both = st.merge(masked, e)
        assert not both.valid
        O, lse = st.finalize(both)
        assert lse == -math.inf and (O == 0).all()


def _random_tree_fold(states, rng):
    states = list(states)
    while len(states) > 1:
        i = rng.integers(0, len(states) - 1)
        states[i:i + 2] = [st.merge(states[i], states[i + 1])]
    return states[0]


@pytest.mark.parametrize("seed", range(5))
def test_merge_associative_any_bracketing(seed):
    """Random partitions, random bracketings and permutations agree with the
    dense row within 1e-12 (M4.3 0x08E/0x08F)."""
    rng = np.random.default_rng(seed)
    n, dv = 37, 4
    s = rng.normal(scale=3.0, size=n)
    v = rng.normal(size=(n, dv))
    dense = st.block_state(s, v)
    Od, Ld = st.finalize(dense)
    cuts = sorted(rng.choice(np.arange(1, n), size=6, replace=False))
    parts = np.split(np.arange(n), cuts)
    states = [st.block_state(s[p], v[p]) for p in parts]
    for _ in range(10):
        perm = rng.permutation(len(states))
        R = _random_tree_fold([states[i] for i in perm], rng)
        O, L = st.finalize(R)
        assert R.n == n and R.m == dense.m
        np.testing.assert_allclose(O, Od, atol=1e-12, rtol=0)
        assert abs(L - Ld) <= 1e-12


# ---------------------------------------------------------------------------
# Closed forms and special cases of the dense C oracle
# ---------------------------------------------------------------------------

def _rand(shape, rng, dtype=np.float32):
    return rng.standard_normal(shape).astype(dtype)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_query_gives_prefix_mean(causal):
    """Q = 0 makes every score 0: O_i is the mean of the visible V rows and
    LSE_i = log(#visible).  GQA: head h averages KV head h // g."""
    rng = np.random.default_rng(1)
    B, H, Hkv, S, d = 2, 4, 2, 9, 8
    q = np.zeros((B, H, S, d), np.float32)
    k = _rand((B, Hkv, S, d), rng)
    v = _rand((B, Hkv, S, d), rng)
    o, lse = oracle.attn_fwd(q, k, v, 0.3, causal)
    for b in range(B):
        for h in range(H):
            vv = v[b, h // 2].astype(np.float64)
            for i in range(S):
                n = i + 1 if causal else S
                np.testing.assert_allclose(o[b, h, i], vv[:n].mean(0), atol=1e-14, rtol=0)
                assert abs(lse[b, h, i] - math.log(n)) <= 1e-14


def test_unit_values_give_unit_output():
    """V = 1 everywhere: each probability row sums to one, so O = 1."""
    rng = np.random.default_rng(2)
    q = _rand((1, 3, 20, 16), rng) * 3
    k = _rand((1, 3, 33, 16), rng) * 3
    v = np.ones((1, 3, 33, 16), np.float32)
    for causal in (False, True):
        o, _ = oracle.attn_fwd(q, k, v, 0.25, causal)
        np.testing.assert_allclose(o, 1.0, atol=1e-13, rtol=0)


def test_one_hot_dominant_selects_row_and_kv_head():
    """Orthogonal keys and Q_i = 40 e_pi(i): O_i = V[kv(h), pi(i)] up to
    e^-40 * Sk.  Pins the head map (h // g, not h % Hkv) and the k/v index."""
    rng = np.random.default_rng(3)
    B, H, Hkv, Sq, Sk, d = 1, 4, 2, 12, 32, 32
    k = np.zeros((B, Hkv, Sk, d), np.float32)
    for kv in range(Hkv):
        k[0, kv] = np.eye(Sk, d, dtype=np.float32)
    v = _rand((B, Hkv, Sk, d), rng)
    perm = rng.integers(0, Sk, size=(H, Sq))
    q = np.zeros((B, H, Sq, d), np.float32)
    for h in range(H):
        for i in range(Sq):
            q[0, h, i, perm[h, i]] = 40.0
    o, lse = oracle.attn_fwd(q, k, v, 1.0, False)
    for h in range(H):
        for i in range(Sq):
            np.testing.assert_allclose(o[0, h, i], v[0, h // 2, perm[h, i]], atol=10 * Sk * math.exp(-40), rtol=0)
            assert abs(lse[0, h, i] - (40.0 + math.log(1 + (Sk - 1) * math.exp(-40)))) <= 1e-12
    # The wrong map h % Hkv would pick the other KV head for h = 1 and h = 2.
    assert np.abs(o[0, 1] - v[0, 1][perm[1]]).max() > 0.1


def test_causal_row_zero_sees_only_key_zero():
    rng = np.random.default_rng(4)
    q = _rand((2, 2, 7, 16), rng)
    k = _rand((2, 2, 7, 16), rng)
    v = _rand((2, 2, 7, 16), rng)
    o, lse = oracle.attn_fwd(q, k, v, 0.7, True)
    for b in range(2):
        for h in range(2):
            np.testing.assert_array_equal(o[b, h, 0], v[b, h, 0].astype(np.float64))
            s00 = 0.7 * float(np.dot(q[b, h, 0].astype(np.float64), k[b, h, 0].astype(np.float64)))
            assert abs(lse[b, h, 0] - s00) <= 1e-13


def test_lse_is_logsumexp_of_scores():
    """LSE against scipy's logsumexp of the materialised fp64 scores."""
    rng = np.random.default_rng(5)
    q = _rand((1, 2, 10, 24), rng)
    k = _rand((1, 2, 15, 24), rng)
    v = _rand((1, 2, 15, 24), rng)
    _, lse = oracle.attn_fwd(q, k, v, 0.4, False)
    S = 0.4 * np.einsum("bhid,bhjd->bhij", q.astype(np.float64), k.astype(np.float64))
    np.testing.assert_allclose(lse, scipy.special.logsumexp(S, axis=-1), atol=1e-12, rtol=0)


def _torch_materialised(q, k, v, scale, causal):
    """A second, independent implementation: library matmul + softmax in fp64
    with K/V heads expanded by repeat_interleave and the mask from tril."""
    q, k, v = (torch.from_numpy(x).double() for x in (q, k, v))
    g = q.shape[1] // k.shape[1]
    k = k.repeat_interleave(g, dim=1)
    v = v.repeat_interleave(g, dim=1)
    S = scale * q @ k.transpose(-1, -2)
    Sq, Sk = S.shape[-2:]
    if causal:
        allowed = torch.ones(Sq, Sk, dtype=torch.bool).tril(diagonal=Sk - Sq)
        S = S.masked_fill(~allowed, float("-inf"))
    P = torch.softmax(S, dim=-1)
    return (P @ v).numpy(), torch.logsumexp(S, dim=-1).numpy()


@pytest.mark.parametrize("shape", [
    (1, 2, 2, 17, 17, 8, False),
    (2, 4, 2, 13, 29, 16, True),     # GQA, rectangular bottom-right causal
    (1, 6, 2, 9, 9, 12, True),       # g = 3
    (1, 2, 1, 31, 5, 4, False),      # d < Sk < Sq: a transposed operand fails
])
def test_bruteforce_matches_torch(shape):
    B, H, Hkv, Sq, Sk, d, causal = shape
    rng = np.random.default_rng(6)
    q, k, v = _rand((B, H, Sq, d), rng), _rand((B, Hkv, Sk, d), rng), _rand((B, Hkv, Sk, d), rng)
    o, lse = oracle.attn_fwd(q, k, v, 0.37, causal)
    ot, lt = _torch_materialised(q, k, v, 0.37, causal)
    np.testing.assert_allclose(o, ot, atol=1e-12, rtol=0)
    np.testing.assert_allclose(lse, lt, atol=1e-12, rtol=0)


def test_gqa_direct_map_equals_repeat_and_wrong_map_differs():
    """M4.4 0x06C: the direct map h // g equals explicit K/V repetition
    exactly; the shape-valid wrong map h % Hkv gives a different output."""
    rng = np.random.default_rng(7)
    B, H, Hkv, S, d = 2, 6, 2, 11, 8
    q, k, v = _rand((B, H, S, d), rng), _rand((B, Hkv, S, d), rng), _rand((B, Hkv, S, d), rng)
    o, lse = oracle.attn_fwd(q, k, v, 0.5, True)
    g = H // Hkv
    kr, vr = np.repeat(k, g, axis=1), np.repeat(v, g, axis=1)
    o2, lse2 = oracle.attn_fwd(q, kr, vr, 0.5, True)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)
    wrong = [h % Hkv for h in range(H)]
    o3, _ = oracle.attn_fwd(q, k[:, wrong], v[:, wrong], 0.5, True)
    assert np.abs(o3 - o).max() > 0.05


def test_rectangular_causal_masks_bottom_right(golden):
    """M4.4 0x05.1F: Q = 0 and V_j = e_j reveal the visible set of each row:
    O_i[j] = 1/|vis(i)| exactly where j is visible.  Rows with no visible key
    follow the zero-output / LSE = -inf policy."""
    for case in golden("causal_rect_masks.json")["cases"]:
        Sq, Sk = case["Sq"], case["Sk"]
        d = Sk
        q = np.zeros((1, 1, Sq, d), np.float32)
        k = np.zeros((1, 1, Sk, d), np.float32)
        v = np.eye(Sk, d, dtype=np.float32).reshape(1, 1, Sk, d)
        o, lse = oracle.attn_fwd(q, k, v, 1.0, True)
        got = (o[0, 0] > 0).astype(int).tolist()
        assert got == case["bottom_right"]
        for i, row in enumerate(case["bottom_right"]):
            if sum(row) == 0:
                assert lse[0, 0, i] == -math.inf and (o[0, 0, i] == 0).all()
            else:
                assert abs(lse[0, 0, i] - math.log(sum(row))) <= 1e-15


# ---------------------------------------------------------------------------
# Decode oracle: split-KV partial states
# ---------------------------------------------------------------------------

def _decode_inputs(rng, B=3, Hq=4, Hkv=2, Skm=50, d=16, lens=(1, 17, 50)):
    q = _rand((B, Hq, 1, d), rng)
    k = _rand((B, Hkv, Skm, d), rng)
    v = _rand((B, Hkv, Skm, d), rng)
    return q, k, v, np.array(lens, np.int32)


@pytest.mark.parametrize("n_split", [1, 4, 16])
def test_decode_chunk_states_merge_to_unsplit(n_split):
    rng = np.random.default_rng(8)
    q, k, v, lens = _decode_inputs(rng)
    O, L = oracle.attn_decode(q, k, v, lens, 0.25)
    m, l, u, cnt = oracle.decode_chunk_states(q, k, v, lens, 0.25, n_split)
    B, Hq = q.shape[:2]
    for b in range(B):
        bounds = oracle.decode_chunk_bounds(int(lens[b]), n_split)
        assert bounds[0][0] == 0 and bounds[-1][1] == lens[b]
        assert all(bounds[c][1] == bounds[c + 1][0] for c in range(n_split - 1))
        for h in range(Hq):
            assert cnt[b, h].sum() == lens[b]
            states = []
            for c in range(n_split):
                valid = cnt[b, h, c] > 0
                assert valid == np.isfinite(m[b, h, c])
                states.append(st.State(bool(valid), m[b, h, c], l[b, h, c], u[b, h, c],
                                       int(cnt[b, h, c])))
            rng2 = random.Random(b * 31 + h)
            for fold in (st.fold_sequential, st.fold_balanced,
                         lambda s: st.fold_sequential(rng2.sample(s, len(s)))):
                Ob, Lb = st.finalize(fold(states))
                np.testing.assert_allclose(Ob, O[b, h, 0], atol=1e-12, rtol=0)
                assert abs(Lb - L[b, h]) <= 1e-12


def test_decode_equals_forward_on_valid_prefix_and_ignores_padding():
    rng = np.random.default_rng(9)
    q, k, v, lens = _decode_inputs(rng)
    O, L = oracle.attn_decode(q, k, v, lens, 0.25)
    kn, vn = k.copy(), v.copy()
    for b, Lb in enumerate(lens):
        kn[b, :, Lb:] = np.nan
        vn[b, :, Lb:] = np.nan
        of, lf = oracle.attn_fwd(q[b:b + 1], k[b:b + 1, :, :Lb], v[b:b + 1, :, :Lb], 0.25, False)
        np.testing.assert_array_equal(of[0, :, 0], O[b, :, 0])
        np.testing.assert_array_equal(lf[0, :, 0], L[b])
    O2, L2 = oracle.attn_decode(q, kn, vn, lens, 0.25)
    np.testing.assert_array_equal(O2, O)
    np.testing.assert_array_equal(L2, L)


def test_rows_subset_matches_full():
    rng = np.random.default_rng(10)
    q, k, v = _rand((2, 4, 19, 8), rng), _rand((2, 2, 23, 8), rng), _rand((2, 2, 23, 8), rng)
    o, lse = oracle.attn_fwd(q, k, v, 0.3, True)
    ids = np.array([0, 5, 18, 19, 77, 2 * 4 * 19 - 1])
    o2, l2 = oracle.attn_fwd_rows(q, k, v, 0.3, True, ids)
    np.testing.assert_array_equal(o2, o.reshape(-1, 8)[ids])
    np.testing.assert_array_equal(l2, lse.reshape(-1)[ids])
