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
