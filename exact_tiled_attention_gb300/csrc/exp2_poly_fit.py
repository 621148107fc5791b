"""Derives the degree-3 polynomial p(f) ~ 2^f on f in [0, 1) used by the
software exp2 in gbattn_ptx.cuh (ex2_poly3_x2).

p(f) = 1 + c1 f + c2 f^2 + c3 f^3 with p(0) = 1 exactly, chosen to minimise the
maximum RELATIVE error |p(f) / 2^f - 1| on [0, 1] (Remez exchange on the
three free coefficients, fp64).  Run it to reprint the constants:

    python exact_tiled_attention_gb300/csrc/exp2_poly_fit.py
"""
import numpy as np


def fit(iters: int = 60):
    grid = np.linspace(0.0, 1.0, 200001)
    target = np.exp2(grid)
    # start from a least-squares fit of (2^f - 1) / f on Chebyshev-like nodes
    ref = 0.5 - 0.5 * np.cos(np.pi * (np.arange(4) + 0.5) / 4)  # 4 reference points in (0, 1)
    c = np.zeros(3)
    for _ in range(iters):
        # solve p(x_i) / 2^x_i - 1 = (-1)^i E at the 4 reference points:
        # c1 x + c2 x^2 + c3 x^3 - (-1)^i E 2^x = 2^x - 1
        A = np.stack([ref, ref ** 2, ref ** 3, -((-1.0) ** np.arange(4)) * np.exp2(ref)], axis=1)
        sol = np.linalg.solve(A, np.exp2(ref) - 1.0)
        c = sol[:3]
        err = (1 + c[0] * grid + c[1] * grid ** 2 + c[2] * grid ** 3) / target - 1
        # new reference: the extrema of the error between sign changes (excluding f = 0, where err = 0)
        idx = []
        sign_changes = np.where(np.diff(np.sign(err[1:])) != 0)[0] + 1
        bounds = [1] + list(sign_changes + 1) + [len(grid)]
        for a, b in zip(bounds[:-1], bounds[1:]):
            seg = np.arange(a, b)
            if len(seg):
                idx.append(seg[np.argmax(np.abs(err[seg]))])
        if len(idx) < 4:
            break
        # keep the 4 largest alternating extrema
        idx = sorted(idx, key=lambda i: -abs(err[i]))[:4]
        ref = np.sort(grid[idx])
    err = (1 + c[0] * grid + c[1] * grid ** 2 + c[2] * grid ** 3) / target - 1
    return c, float(np.abs(err).max())


if __name__ == "__main__":
    c, e = fit()
    print("c1 = %.9ef\nc2 = %.9ef\nc3 = %.9ef\nmax relative error (fp64 evaluation) = %.3e" % (c[0], c[1], c[2], e))
