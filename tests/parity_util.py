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


# Gradient tolerances (backward).  The task states none for gradients; this
# bound is derived from the arithmetic of the kernels (M4.4 0x06.1A gives the
# gradients: dV = P^T dO, dS = P o (dP - D), dQ = tau dS K, dK = tau dS^T Q,
# with the row scalar D = dO . O computed from the stored 16-bit O).
#
# With u the unit roundoff of the input dtype (bf16 2^-8, fp16 2^-11):
#
# (1) Rounded operands.  Every gradient element g = sum_t a_t b_t is formed by
#     the tensor cores from operands of which one was rounded to the dtype just
#     before the product (P for dV, dS for dQ and dK: relative error <= u each,
#     independent from term to term), accumulated in fp32 (~2^-24 per add,
#     negligible) and rounded to the dtype once (<= u |g|).  The rounding errors
#     of the summed terms are independent with mean zero, so their sum has a
#     standard deviation of about (u / sqrt(3)) * sqrt(sum_t a_t^2 b_t^2): the
#     natural scale of that gradient row, which the root mean square of the
#     reference over the row (the head dimension) estimates.  With up to three
#     such sources sigma <= u * rms_row, and the largest of ~1e8 elements stays
#     within 6 sigma: GRAD_C * u * (|ref| + rms_row) with GRAD_C = 8 covers the
#     final rounding (1) and the summed terms (6).
#
# (2) The row scalar D.  D_i = dO_i . O_i uses the stored O, which differs from
#     the exact output by its rounding (<= u |O_ik|) and the forward's own
#     rounding of P (<= u rms(O_i) per element at the same 6-sigma level), so
#     |dD_i| <= u A_i with A_i = sum_k |dO_ik| (|O_ik| + rms(O_i)).  The error
#     shifts every dS_ij of row i by P_ij dD_i, which does NOT cancel the way
#     sum_j dS_ij = 0 makes the exact dQ row cancel (rows with few visible keys,
#     or a peaked softmax, have a small dQ but the full D error):
#         dQ_ik gets  tau dD_i (P K)_ik           <= u * tau * A_i |(P K)_ik|
#         dK_jk gets  tau sum_i P_ij dD_i Q_ik    <= u * tau * (P^T (A o |Q|))_jk
#     both computed exactly by the oracle (grad_extras); GRAD_CD = 2 allows the
#     two parts of dD_i to add.  dV does not involve D.
#
#     |g - ref| <= GRAD_C * u * (|ref| + rms_row(ref)) + GRAD_CD * u * extra + GRAD_ATOL
#
# The absolute floor covers gradients that vanish exactly (dQ with a single
# visible key): the kernel's D (fp32 FMA chain) and dP (tensor-core fp32)
# differ by ~d * 2^-24 * |dO||O|, i.e. ~1e-6 after scaling.  The relative
# Frobenius error of a whole tensor is ~u * sqrt(3) (0.7 % for bf16) and is
# bounded by GRAD_REL_FRO = 1e-2.
GRAD_C = 8.0
GRAD_CD = 2.0
GRAD_REL_FRO = 1e-2
GRAD_ATOL = 1e-5
UNIT_ROUNDOFF = {torch.bfloat16: 2.0 ** -8, torch.float16: 2.0 ** -11}

# Measured margins, one record per comparison (written out by conftest when
# GBATTN_GRAD_LOG names a file).
GRAD_LOG = []


def grad_extras(q, k, v, dout, scale, causal):
    """The D-error scales of (2) above for dQ and dK, from the fp64 oracle:
    dq [B,H,Sq,d] = tau A_i |(P K)_ik| and dk [B,Hkv,Sk,d] = tau (P^T (A o |Q|))
    (summed over each KV head's query-head group).  Inputs as for the oracle
    (the rounded 16-bit values widened to fp32 numpy arrays)."""
    import oracle

    o, _ = oracle.attn_fwd(q, k, v, scale, causal)
    rms_o = np.sqrt(np.mean(o * o, axis=-1, keepdims=True))
    a = np.sum(np.abs(dout) * (np.abs(o) + rms_o), axis=-1, keepdims=True)
    pk, _ = oracle.attn_fwd(q, k, k, scale, causal)
    w = (a * np.abs(q)).astype(np.float32)
    ptw = oracle.attn_bwd(q, k, v, w, scale, causal)[2]
    return {"dq": scale * a * np.abs(pk), "dk": scale * ptw}


def assert_grad_close(g_gpu, g_ref, what="", dtype=None, extra=None):
    if isinstance(g_gpu, torch.Tensor):
        dtype = dtype or g_gpu.dtype
        g = g_gpu.detach().float().cpu().numpy().astype(np.float64)
    else:
        g = np.asarray(g_gpu, dtype=np.float64)
    u = UNIT_ROUNDOFF[dtype]
    ref = np.asarray(g_ref, dtype=np.float64).reshape(g.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite gradient"
    err = np.abs(g - ref)
    rms_row = np.sqrt(np.mean(ref * ref, axis=-1, keepdims=True))
    bound = GRAD_C * u * (np.abs(ref) + rms_row) + GRAD_ATOL
    if extra is not None:
        bound = bound + GRAD_CD * u * np.asarray(extra, dtype=np.float64).reshape(g.shape)
    nrm = np.linalg.norm(ref)
    fro = np.linalg.norm(g - ref) / nrm if nrm > 0 else 0.0
    fro_bound = GRAD_REL_FRO + (GRAD_ATOL * np.sqrt(ref.size) / nrm if nrm > 0 else 0.0)
    used = float(np.max(np.maximum(err - GRAD_ATOL, 0.0) / np.maximum(bound - GRAD_ATOL, 1e-300))) if err.size else 0.0
    GRAD_LOG.append({"what": what, "dtype": str(dtype).replace("torch.", ""), "elements": int(ref.size),
                     "rel_fro": float(fro), "bound_used": used, "d_term": extra is not None})
    if nrm > 0:
        assert fro <= fro_bound, f"{what}: relative Frobenius error {fro:.3e} > {fro_bound:.3e}"
    worst = np.unravel_index(np.argmax(err - bound), err.shape) if err.size else None
    assert (err <= bound).all(), \
        f"{what}: |err| {err[worst]:.3e} > {bound[worst]:.3e} at {worst} (ref {ref[worst]:.3e}, bound used {used:.2f})"
    return float(fro), used
