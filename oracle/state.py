"""Online-softmax state algebra, written out in fp64 (test infrastructure only).

Nothing in the product path imports this module; tests, the smoke check and
the bench's CPU-baseline leg use it to check the CUDA kernels' partial states
and to pin the oracle against the worked traces the pages print.

Sources (page, section):
  M4.3 "IO-Aware Attention and FlashAttention-1" 0x08A  state(A) = (m, l, u, n) of an index set
  M4.3 0x08B                       binary merge with one common maximum
  M4.3 0x08C                       identity (-inf, 0, 0, 0) with a validity flag
  M4.3 0x09A / 0x09E               O = u / l,  LSE = m + log l
  M4.3 0x09E                       (LSE, O) merge via logaddexp
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np


@dataclass
class State:
    """Canonical summary of one set of allowed score positions (M4.3 0x08A).

    valid=False is the executable identity: m=-inf, l=0, u=0, n=0 (0x08C).
    """

    valid: bool
    m: float
    l: float
    u: np.ndarray
    n: int = 0

    @staticmethod
    def empty(dv: int) -> "State":
        return State(False, -math.inf, 0.0, np.zeros(dv, dtype=np.float64), 0)


def block_state(scores, values) -> State:
    """state(A) straight from its definition: m = max, l = sum exp(s - m),
    u = sum exp(s - m) v, n = |A|.  Masked positions (-inf) are not in A."""
    s = np.asarray(scores, dtype=np.float64).reshape(-1)
    v = np.asarray(values, dtype=np.float64).reshape(len(s), -1)
    keep = s != -math.inf
    s, v = s[keep], v[keep]
    if len(s) == 0:
        return State.empty(v.shape[1])
    m = float(np.max(s))
    p = np.exp(s - m)
    return State(True, m, float(np.sum(p)), p @ v, int(len(s)))


def merge(a: State, b: State) -> State:
    """a (+) b for disjoint index sets (M4.3 0x08B), with the validity branch
    of 0x08C so the identity never evaluates exp(-inf - -inf)."""
    if not a.valid:
        return b
    if not b.valid:
        return a
    m = max(a.m, b.m)
    alpha = math.exp(a.m - m)
    beta = math.exp(b.m - m)
    return State(True, m, alpha * a.l + beta * b.l, alpha * a.u + beta * b.u, a.n + b.n)


def finalize(s: State):
    """(O, LSE) of a state: O = u / l, LSE = m + log l (M4.3 0x09A, 0x09E).
    An invalid state follows the zero-payload policy: O = 0, LSE = -inf."""
    if not s.valid:
        return np.zeros_like(s.u), -math.inf
    return s.u / s.l, s.m + math.log(s.l)


def fold_sequential(states):
    acc = None
    for s in states:
        acc = s if acc is None else merge(acc, s)
    return acc


def fold_balanced(states):
    states = list(states)
    while len(states) > 1:
        nxt = [merge(states[i], states[i + 1]) for i in range(0, len(states) - 1, 2)]
        if len(states) % 2:
            nxt.append(states[-1])
        states = nxt
    return states[0]


def lse_merge(lse_a: float, o_a, lse_b: float, o_b):
    """(LSE, O) form of the merge (M4.3 0x09E): L = logaddexp(L_A, L_B),
    O = e^(L_A - L) O_A + e^(L_B - L) O_B.  -inf marks an empty part."""
    if lse_a == -math.inf:
        return lse_b, np.asarray(o_b, dtype=np.float64)
    if lse_b == -math.inf:
        return lse_a, np.asarray(o_a, dtype=np.float64)
    L = float(np.logaddexp(lse_a, lse_b))
    return L, math.exp(lse_a - L) * np.asarray(o_a) + math.exp(lse_b - L) * np.asarray(o_b)
