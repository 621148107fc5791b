"""Shared helpers for the GPU parity tests: tolerances and comparisons of the
CUDA path's outputs with the fp64 oracle's."""
import numpy as np
import torch

# Tolerances for fp16/bf16 inputs with fp32 accumulation: O max-abs <= 2e-2
# and mean-abs <= 2e-3, LSE max-abs <= 1e-3.  The kernel rounds P to the
# input dtype before the P.V product (8 bits of mantissa for bf16) and O to
# the output dtype; both errors are well inside these bounds for |V| ~ N(0,1).
O_MAX_ABS = 2e-2
O_MEAN_ABS = 2e-3
LSE_MAX_ABS = 1e-3


def host_f32(t: torch.Tensor) -> np.ndarray:
    """The rounded fp16/bf16 values, widened exactly to float32 on the host."""
    return t.detach().float().cpu().numpy()


def assert_attn_close(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    o = o_gpu.detach().float().cpu().numpy().astype(np.float64)
    o_ref = np.asarray(o_ref, dtype=np.float64).reshape(o.shape)
    assert np.isfinite(o).all(), f"{what}: non-finite O"
    err = np.abs(o - o_ref)
    assert err.max() <= O_MAX_ABS, f"{what}: O max-abs {err.max():.3e} > {O_MAX_ABS}"
    assert err.mean() <= O_MEAN_ABS, f"{what}: O mean-abs {err.mean():.3e} > {O_MEAN_ABS}"
    if lse_gpu is not None:
        lse = lse_gpu.detach().cpu().numpy().astype(np.float64)
        lse_ref = np.asarray(lse_ref, dtype=np.float64).reshape(lse.shape)
        inf_ref = np.isneginf(lse_ref)
        assert (np.isneginf(lse) == inf_ref).all(), f"{what}: -inf LSE pattern differs"
        if (~inf_ref).any():
            lerr = np.abs(lse[~inf_ref] - lse_ref[~inf_ref])
            assert lerr.max() <= LSE_MAX_ABS, f"{what}: LSE max-abs {lerr.max():.3e} > {LSE_MAX_ABS}"
    return float(err.max()), float(err.mean())


# Gradient tolerances (backward), relative to each gradient tensor's own scale:
# relative Frobenius error <= 1e-2 and every element within 2e-2 * max|ref|.
# The kernel rounds P and dS to the input dtype before the tensor-core
# products (relative 2^-9 for bf16, each term), takes D = dO . O from the
# forward's rounded O, and rounds dQ/dK/dV to the dtype (2^-9): each source
# alone is a ~0.1-0.2 % relative error; the bounds leave a 5x margin.
GRAD_REL_FRO = 1e-2
GRAD_MAX_REL = 2e-2
# Absolute floor for gradients whose exact value is (near) zero, e.g. dQ with a
# single visible key: the kernel's D = dO . O (fp32 FMA chain over d) and its
# dP (tensor-core fp32 sums) differ by ~d * 2^-24 * |dO||O|, so dS and dQ carry
# an absolute error of about tau * that * max|K| ~ 1e-6 even where they vanish.
GRAD_ATOL = 1e-5


def assert_grad_close(g_gpu, g_ref, what=""):
    g = g_gpu.detach().float().cpu().numpy().astype(np.float64) if isinstance(g_gpu, torch.Tensor) \
        else np.asarray(g_gpu, dtype=np.float64)
    ref = np.asarray(g_ref, dtype=np.float64).reshape(g.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite gradient"
    scale = np.abs(ref).max()
    err = np.abs(g - ref)
    fro = np.linalg.norm(g - ref) / max(np.linalg.norm(ref), 1e-300)
    fro_bound = GRAD_REL_FRO + GRAD_ATOL * np.sqrt(ref.size) / max(np.linalg.norm(ref), 1e-300)
    assert fro <= fro_bound, f"{what}: relative Frobenius error {fro:.3e} > {fro_bound:.3e}"
    assert err.max() <= GRAD_MAX_REL * scale + GRAD_ATOL, \
        f"{what}: max-abs {err.max():.3e} > {GRAD_MAX_REL} x max|ref| ({scale:.3e})"
    return float(fro), float(err.max() / max(scale, 1e-300))
