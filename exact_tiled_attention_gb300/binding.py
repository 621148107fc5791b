"""Thin Python binding of libgbattn.so (argument marshalling only).

Every step of the attention computation runs in the CUDA kernels behind the
C ABI declared in include/gbattn.h; this module only checks tensor metadata,
allocates outputs through PyTorch (device memory and streams are PyTorch's)
and forwards raw device pointers.  There is no CPU or PyTorch fallback: if the
library is missing or the current device is not sm_103, calls raise.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgbattn.so")

GBATTN_OK = 0
GBATTN_F16 = 0
GBATTN_BF16 = 1
GBATTN_EDEVICE_TIMEOUT = -8
ERRORS = {
    -1: "GBATTN_EBADSHAPE", -2: "GBATTN_EHEADS", -3: "GBATTN_EHEADDIM", -4: "GBATTN_EDTYPE",
    -5: "GBATTN_EPOINTER", -6: "GBATTN_EWORKSPACE", -7: "GBATTN_ELAUNCH",
    -8: "GBATTN_EDEVICE_TIMEOUT", -9: "GBATTN_ESPLIT", -10: "GBATTN_EUNSUPPORTED",
}
EXPORTS = ("attn_fwd", "attn_fwd_pair", "attn_decode_workspace_bytes", "attn_decode_splitkv",
           "attn_decode_splitkv_noalloc", "attn_decode_noalloc_scratch_bytes",
           "attn_bwd_workspace_bytes", "attn_bwd", "attn_bwd_atomic_workspace_bytes", "attn_bwd_atomic",
           "gbattn_exp2_paths",
           "attn_fwd_fp8_workspace_bytes", "attn_fwd_fp8", "gbattn_selftest_bounded_wait",
           "gbattn_causal_tile_counts", "gbattn_device_status", "gbattn_timeline_set",
           "gbattn_error_string", "gbattn_version")

_lock = threading.Lock()
_lib = None


class GbattnError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {ERRORS.get(code, code)} ({error_string(code)})")


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libgbattn.so (built by exact_tiled_attention_gb300._build).  Raises
    if it is missing: there is no fallback implementation."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with "
                               "`python -m exact_tiled_attention_gb300._build` (no fallback exists)")
        lib = ctypes.CDLL(path)
        vp, ci, cf, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        ll_p = ctypes.POINTER(ctypes.c_longlong)
        lib.attn_fwd.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, cf, ci, ci, vp]
        lib.attn_fwd.restype = ci
        lib.attn_fwd_pair.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, cf, ci, vp]
        lib.attn_fwd_pair.restype = ci
        lib.attn_decode_workspace_bytes.argtypes = [ci, ci, ci, ci]
        lib.attn_decode_workspace_bytes.restype = sz
        lib.attn_decode_splitkv.argtypes = [vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, cf, ci, vp, sz,
                                            ci, vp]
        lib.attn_decode_splitkv.restype = ci
        lib.attn_decode_splitkv_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, cf, ci,
                                                    ci, vp]
        lib.attn_decode_splitkv_noalloc.restype = ci
        lib.attn_decode_noalloc_scratch_bytes.argtypes = []
        lib.attn_decode_noalloc_scratch_bytes.restype = sz
        lib.attn_bwd_workspace_bytes.argtypes = [ci, ci, ci, ci]
        lib.attn_bwd_workspace_bytes.restype = sz
        lib.attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, cf, ci, vp,
                                 sz, ci, vp]
        lib.attn_bwd.restype = ci
        lib.attn_bwd_atomic_workspace_bytes.argtypes = [ci, ci, ci, ci]
        lib.attn_bwd_atomic_workspace_bytes.restype = sz
        lib.attn_bwd_atomic.argtypes = lib.attn_bwd.argtypes
        lib.attn_bwd_atomic.restype = ci
        lib.attn_fwd_fp8_workspace_bytes.argtypes = [ci, ci, ci, ci]
        lib.attn_fwd_fp8_workspace_bytes.restype = sz
        lib.attn_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, cf, ci, vp, sz, vp]
        lib.attn_fwd_fp8.restype = ci
        lib.gbattn_exp2_paths.argtypes = [vp, vp, vp, ctypes.c_longlong, vp]
        lib.gbattn_exp2_paths.restype = ci
        lib.gbattn_causal_tile_counts.argtypes = [ci, ci, ci, ci, ll_p, ll_p, ll_p, ll_p, ll_p]
        lib.gbattn_causal_tile_counts.restype = ci
        lib.gbattn_selftest_bounded_wait.argtypes = [ci, vp]
        lib.gbattn_selftest_bounded_wait.restype = ci
        lib.gbattn_timeline_set.argtypes = [vp, ctypes.c_longlong]
        lib.gbattn_timeline_set.restype = ci
        lib.gbattn_device_status.argtypes = []
        lib.gbattn_device_status.restype = ci
        lib.gbattn_error_string.argtypes = [ci]
        lib.gbattn_error_string.restype = ctypes.c_char_p
        lib.gbattn_version.argtypes = []
        lib.gbattn_version.restype = ctypes.c_char_p
        _lib = lib
        return lib


def error_string(code: int) -> str:
    try:
        return load_library().gbattn_error_string(int(code)).decode()
    except Exception:  # library not loadable: still produce a message
        return ERRORS.get(code, str(code))


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return GBATTN_F16
    if t.dtype == torch.bfloat16:
        return GBATTN_BF16
    raise TypeError(f"unsupported dtype {t.dtype}; expected float16 or bfloat16")


def _check(t: torch.Tensor, name: str, ndim: int):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (there is no CPU path)")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous ([B, heads, S, d] row-major)")


def _stream_ptr(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def attn_fwd(q, k, v, scale: float | None = None, causal: bool = False, out=None, lse=None,
             return_lse: bool = True, stream=None):
    """Exact attention forward through the C ABI `attn_fwd`.

    q [B,H,Sq,d], k/v [B,Hkv,Sk,d] (fp16 or bf16, CUDA, contiguous).
    Returns (o [B,H,Sq,d] in q's dtype, lse [B,H,Sq] fp32 or None)."""
    _check(q, "q", 4)
    _check(k, "k", 4)
    _check(v, "v", 4)
    B, H, Sq, d = q.shape
    Bk, Hkv, Sk, dk = k.shape
    if k.shape != v.shape or Bk != B or dk != d:
        raise ValueError(f"shape mismatch q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share one dtype")
    dt = _dtype_code(q)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device)
    lib = load_library()
    rc = lib.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                      lse.data_ptr() if lse is not None else None, B, H, Hkv, Sq, Sk, d, float(scale),
                      int(bool(causal)), dt, _stream_ptr(stream))
    if rc != GBATTN_OK:
        raise GbattnError(rc, "attn_fwd")
    return out, lse


def attn_fwd_pair(q, k, v, scale: float | None = None, out=None, lse=None, return_lse: bool = True, stream=None):
    """Non-causal d = 128 forward on tcgen05 CTA pairs through the C ABI
    `attn_fwd_pair`; arguments and results as attn_fwd with causal=False."""
    _check(q, "q", 4)
    _check(k, "k", 4)
    _check(v, "v", 4)
    B, H, Sq, d = q.shape
    Bk, Hkv, Sk, dk = k.shape
    if k.shape != v.shape or Bk != B or dk != d:
        raise ValueError(f"shape mismatch q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share one dtype")
    dt = _dtype_code(q)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device)
    lib = load_library()
    rc = lib.attn_fwd_pair(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                           lse.data_ptr() if lse is not None else None, B, H, Hkv, Sq, Sk, d, float(scale), dt,
                           _stream_ptr(stream))
    if rc != GBATTN_OK:
        raise GbattnError(rc, "attn_fwd_pair")
    return out, lse


def attn_decode_workspace_bytes(B: int, Hq: int, n_split: int, d: int) -> int:
    return int(load_library().attn_decode_workspace_bytes(B, Hq, n_split, d))


def _check_decode(q, k_cache, v_cache, seqlens, out, lse):
    """Metadata checks shared by both decode wrappers: tensor types and ranks,
    then every shape and dtype agreement, then device and layout.  Returns
    (B, Hq, Hkv, Sk_max, d)."""
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{n} must be a torch.Tensor")
        if t.dim() != 4:
            raise ValueError(f"{n} must have 4 dims, got shape {tuple(t.shape)}")
    if not isinstance(seqlens, torch.Tensor):
        raise TypeError("seqlens must be a torch.Tensor")
    B, Hq, one, d = q.shape
    if one != 1:
        raise ValueError("decode takes exactly one query per sequence: q [B,Hq,1,d]")
    Bk, Hkv, Sk_max, dk = k_cache.shape
    if k_cache.shape != v_cache.shape:
        raise ValueError(f"k_cache {tuple(k_cache.shape)} and v_cache {tuple(v_cache.shape)} differ")
    if Bk != B or dk != d:
        raise ValueError(f"cache batch/head dim {Bk}/{dk} do not match q's {B}/{d}")
    if not (q.dtype == k_cache.dtype == v_cache.dtype):
        raise TypeError("q and the caches must share one dtype")
    _dtype_code(q)
    if seqlens.dtype != torch.int32:
        raise TypeError(f"seqlens must be int32, got {seqlens.dtype}")
    if seqlens.dim() != 1 or seqlens.numel() != B:
        raise ValueError(f"seqlens must hold one length per sequence ({B}), got shape {tuple(seqlens.shape)}")
    if out is not None and (not isinstance(out, torch.Tensor) or out.shape != q.shape or out.dtype != q.dtype):
        raise ValueError("out must be a tensor of q's shape and dtype")
    if lse is not None and (not isinstance(lse, torch.Tensor) or tuple(lse.shape) != (B, Hq)
                            or lse.dtype != torch.float32):
        raise ValueError(f"lse must be a float32 tensor [{B}, {Hq}]")
    _check(q, "q", 4)
    _check(k_cache, "k_cache", 4)
    _check(v_cache, "v_cache", 4)
    if not seqlens.is_cuda or not seqlens.is_contiguous():
        raise ValueError("seqlens must be a contiguous CUDA tensor")
    for t, n in ((out, "out"), (lse, "lse")):
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError(f"{n} must be a contiguous CUDA tensor")
    return B, Hq, Hkv, Sk_max, d


def attn_decode_splitkv(q, k_cache, v_cache, seqlens, scale: float | None = None, n_split: int = 16,
                        workspace=None, out=None, lse=None, return_lse: bool = True, stream=None):
    """One-query split-KV decode through the C ABI `attn_decode_splitkv`.

    q [B,Hq,1,d]; k_cache/v_cache [B,Hkv,Sk_max,d]; seqlens [B] int32 (CUDA).
    workspace: optional caller-owned fp32/uint8 CUDA buffer of at least
    attn_decode_workspace_bytes(B, Hq, n_split, d) bytes (allocated here if
    omitted).  Returns (o [B,Hq,1,d], lse [B,Hq] or None, workspace)."""
    B, Hq, Hkv, Sk_max, d = _check_decode(q, k_cache, v_cache, seqlens, out, lse)
    dt = _dtype_code(q)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    lib = load_library()
    need = int(lib.attn_decode_workspace_bytes(B, Hq, n_split, d))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    rc = lib.attn_decode_splitkv(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                 seqlens.data_ptr(), out.data_ptr(),
                                 lse.data_ptr() if lse is not None else None, B, Hq, Hkv, Sk_max, d,
                                 float(scale), int(n_split), workspace.data_ptr(), ws_bytes, dt,
                                 _stream_ptr(stream))
    if rc != GBATTN_OK:
        raise GbattnError(rc, "attn_decode_splitkv")
    return out, lse, workspace


def attn_decode_splitkv_noalloc(q, k_cache, v_cache, seqlens, scale: float | None = None,
                                n_split: int = 16, out=None, lse=None, return_lse: bool = True,
                                stream=None):
    """attn_decode_splitkv without a workspace argument, for callers that
    cannot allocate device memory: the partial states go to the library's
    fixed 32 MiB device array (shared by all calls; order overlapping calls).
    Outputs are allocated here only when `out`/`lse` are not given."""
    B, Hq, Hkv, Sk_max, d = _check_decode(q, k_cache, v_cache, seqlens, out, lse)
    dt = _dtype_code(q)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    rc = load_library().attn_decode_splitkv_noalloc(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), seqlens.data_ptr(), out.data_ptr(),
        lse.data_ptr() if lse is not None else None, B, Hq, Hkv, Sk_max, d, float(scale),
        int(n_split), dt, _stream_ptr(stream))
    if rc != GBATTN_OK:
        raise GbattnError(rc, "attn_decode_splitkv_noalloc")
    return out, lse


def attention_backward(q, k, v, o, lse, dout, scale: float | None = None, causal: bool = False,
                       deterministic: bool = False, workspace=None, dq=None, dk=None, dv=None, stream=None):
    """The backward a caller should use by default: attn_bwd_atomic (the
    faster schedule in every measured case: five 128x128 products per
    (query block, key tile) pair instead of seven), or attn_bwd when
    `deterministic` asks for bitwise-repeatable dQ.  The workspace, if given,
    must be sized by the matching *_workspace_bytes function."""
    fn = attn_bwd if deterministic else attn_bwd_atomic
    return fn(q, k, v, o, lse, dout, scale=scale, causal=causal, workspace=workspace, dq=dq, dk=dk, dv=dv,
              stream=stream)


def attn_fwd_fp8_workspace_bytes(B: int, Hkv: int, Sk: int, d: int) -> int:
    return int(load_library().attn_fwd_fp8_workspace_bytes(B, Hkv, Sk, d))


def attn_fwd_fp8(q, k, v, q_descale=None, k_descale=None, v_descale=None, scale: float | None = None,
                 causal: bool = False, out=None, lse=None, return_lse: bool = True, workspace=None,
                 stream=None):
    """FP8 (E4M3) exact attention forward through the C ABI `attn_fwd_fp8`.

    q [B,H,Sq,128], k/v [B,Hkv,Sk,128] torch.float8_e4m3fn CUDA tensors;
    descales: optional fp32 CUDA tensors [B, Hkv].  Returns (o bf16, lse)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n, 4)
        if t.dtype != torch.float8_e4m3fn:
            raise TypeError(f"{n} must be torch.float8_e4m3fn")
    B, H, Sq, d = q.shape
    Bk, Hkv, Sk, dk = k.shape
    if k.shape != v.shape or Bk != B or dk != d:
        raise ValueError("shape mismatch between q, k, v")
    descales = []
    for t, n in ((q_descale, "q_descale"), (k_descale, "k_descale"), (v_descale, "v_descale")):
        if t is None:
            descales.append(None)
            continue
        if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.float32 and t.is_contiguous()
                and tuple(t.shape) == (B, Hkv)):
            raise ValueError(f"{n} must be a contiguous fp32 CUDA tensor [B, Hkv]")
        descales.append(t.data_ptr())
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    lib = load_library()
    need = int(lib.attn_fwd_fp8_workspace_bytes(B, Hkv, Sk, d))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device)
    rc = lib.attn_fwd_fp8(q.data_ptr(), k.data_ptr(), v.data_ptr(), *descales, out.data_ptr(),
                          lse.data_ptr() if lse is not None else None, B, H, Hkv, Sq, Sk, d, float(scale),
                          int(bool(causal)), workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                          _stream_ptr(stream))
    if rc != GBATTN_OK:
        raise GbattnError(rc, "attn_fwd_fp8")
    return out, lse


def attn_bwd_workspace_bytes(B: int, H: int, Sq: int, d: int) -> int:
    return int(load_library().attn_bwd_workspace_bytes(B, H, Sq, d))


def attn_bwd(q, k, v, o, lse, dout, scale: float | None = None, causal: bool = False,
             workspace=None, dq=None, dk=None, dv=None, stream=None):
    """Exact attention backward through the C ABI `attn_bwd` (two owners, no
    atomics: bitwise repeatable).

    q, o, dout [B,H,Sq,d]; k, v [B,Hkv,Sk,d] (fp16/bf16, CUDA, contiguous);
    lse [B,H,Sq] fp32 from attn_fwd.  workspace: optional caller-owned CUDA
    buffer of at least attn_bwd_workspace_bytes(B, H, Sq, d) bytes (allocated
    here if omitted).  Returns (dq, dk, dv)."""
    return _bwd_call("attn_bwd", "attn_bwd_workspace_bytes", q, k, v, o, lse, dout, scale, causal,
                     workspace, dq, dk, dv, stream)


def attn_bwd_atomic_workspace_bytes(B: int, H: int, Sq: int, d: int) -> int:
    return int(load_library().attn_bwd_atomic_workspace_bytes(B, H, Sq, d))


def attn_bwd_atomic(q, k, v, o, lse, dout, scale: float | None = None, causal: bool = False,
                    workspace=None, dq=None, dk=None, dv=None, stream=None):
    """Exact attention backward through the C ABI `attn_bwd_atomic`: one
    owner per key tile, dQ summed by fp32 atomic adds (not bitwise
    repeatable in dQ).  Head dimension 64 or 128.  Arguments and result as attn_bwd;
    the workspace is attn_bwd_atomic_workspace_bytes(B, H, Sq, d) bytes."""
    return _bwd_call("attn_bwd_atomic", "attn_bwd_atomic_workspace_bytes", q, k, v, o, lse, dout, scale,
                     causal, workspace, dq, dk, dv, stream)


def _bwd_call(fn, ws_fn, q, k, v, o, lse, dout, scale, causal, workspace, dq, dk, dv, stream):
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (dout, "dout")):
        _check(t, n, 4)
    B, H, Sq, d = q.shape
    Bk, Hkv, Sk, dk_ = k.shape
    if k.shape != v.shape or Bk != B or dk_ != d or o.shape != q.shape or dout.shape != q.shape:
        raise ValueError("shape mismatch between q, k, v, o and dout")
    if not (q.dtype == k.dtype == v.dtype == o.dtype == dout.dtype):
        raise TypeError("q, k, v, o, dout must share one dtype")
    if not isinstance(lse, torch.Tensor) or not lse.is_cuda or lse.dtype != torch.float32 or \
            tuple(lse.shape) != (B, H, Sq) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 CUDA tensor [B, H, Sq]")
    dt = _dtype_code(q)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    lib = load_library()
    need = int(getattr(lib, ws_fn)(B, H, Sq, d))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    rc = getattr(lib, fn)(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                          dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, Hkv, Sq, Sk,
                          d, float(scale), int(bool(causal)), workspace.data_ptr(), ws_bytes, dt,
                          _stream_ptr(stream))
    if rc != GBATTN_OK:
        raise GbattnError(rc, fn)
    return dq, dk, dv


def gbattn_causal_tile_counts(Sq: int, Sk: int, Br: int, Bc: int) -> dict:
    """Host planner: full / partial / skipped causal tiles and cell counts."""
    vals = [ctypes.c_longlong() for _ in range(5)]
    rc = load_library().gbattn_causal_tile_counts(Sq, Sk, Br, Bc, *[ctypes.byref(x) for x in vals])
    if rc != GBATTN_OK:
        raise GbattnError(rc, "gbattn_causal_tile_counts")
    keys = ("full", "partial", "skipped", "allowed_cells", "visited_cells")
    return {k: v.value for k, v in zip(keys, vals)}


def gbattn_exp2_paths(x, stream=None):
    """Diagnostic: (software polynomial 2^x, hardware ex2.approx 2^x) for a
    contiguous fp32 CUDA tensor x with an even number of elements."""
    if not (isinstance(x, torch.Tensor) and x.is_cuda and x.dtype == torch.float32 and x.is_contiguous()):
        raise ValueError("x must be a contiguous fp32 CUDA tensor")
    y_poly, y_hw = torch.empty_like(x), torch.empty_like(x)
    rc = load_library().gbattn_exp2_paths(x.data_ptr(), y_poly.data_ptr(), y_hw.data_ptr(), x.numel(),
                                          _stream_ptr(stream))
    if rc != GBATTN_OK:
        raise GbattnError(rc, "gbattn_exp2_paths")
    return y_poly, y_hw


def gbattn_selftest_bounded_wait(arrive: bool, stream=None) -> None:
    """Diagnostic: one bounded mbarrier wait on the device that nothing
    satisfies unless `arrive`; read the outcome with gbattn_device_status()."""
    rc = load_library().gbattn_selftest_bounded_wait(int(bool(arrive)), _stream_ptr(stream))
    if rc != GBATTN_OK:
        raise GbattnError(rc, "gbattn_selftest_bounded_wait")


_timeline_records = None  # keeps the buffer alive while the library holds its address


def gbattn_timeline_set(records) -> None:
    """Per-CTA timeline of attn_fwd and attn_fwd_fp8 launches: `records` is an int64 CUDA tensor
    of shape [capacity, 4] (start ns, end ns, SM, unit per CTA; see the header),
    or None to turn the timeline off.  A launch with more CTAs than
    `capacity` records nothing."""
    global _timeline_records
    lib = load_library()
    if records is None:
        rc = lib.gbattn_timeline_set(None, 0)
        if rc != GBATTN_OK:
            raise GbattnError(rc, "gbattn_timeline_set")
        _timeline_records = None
        return
    if not isinstance(records, torch.Tensor) or not records.is_cuda:
        raise ValueError("timeline records must be a CUDA tensor")
    if records.dtype != torch.int64 or records.dim() != 2 or records.shape[1] != 4 or not records.is_contiguous():
        raise ValueError("timeline records must be a contiguous int64 tensor of shape [capacity, 4]")
    rc = lib.gbattn_timeline_set(ctypes.c_void_p(records.data_ptr()), int(records.shape[0]))
    if rc != GBATTN_OK:
        raise GbattnError(rc, "gbattn_timeline_set")
    _timeline_records = records


def gbattn_device_status() -> int:
    """Synchronise and read/clear the kernels' status word (0 = ok)."""
    return int(load_library().gbattn_device_status())


def gbattn_version() -> str:
    return load_library().gbattn_version().decode()
