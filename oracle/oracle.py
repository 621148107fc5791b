"""ctypes wrapper around attn_oracle.c (fp64 CPU oracle; test infrastructure).

Inputs are numpy arrays holding the already-rounded fp16/bf16 values widened
exactly to float32; all arithmetic happens in binary64 inside the C code.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build_oracle(force: bool = False) -> str:
    """Compile attn_oracle.c into oracle/liboracle.so with gcc + OpenMP.

    -ffp-contract=off keeps every multiply and add separately rounded, so the
    x86 and Arm builds give the same fp64 results.
    """
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fopenmp", "-shared", "-fPIC",
               _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build_oracle()
            lib = ctypes.CDLL(_LIB)
            f32p = ctypes.POINTER(ctypes.c_float)
            f64p = ctypes.POINTER(ctypes.c_double)
            i64p = ctypes.POINTER(ctypes.c_longlong)
            i32p = ctypes.POINTER(ctypes.c_int)
            ci, cd, cll = ctypes.c_int, ctypes.c_double, ctypes.c_longlong
            lib.oracle_attn_fwd_rows.argtypes = [f32p, f32p, f32p, ci, ci, ci, ci, ci, ci, cd, ci,
                                                 i64p, cll, f64p, f64p]
            lib.oracle_attn_fwd.argtypes = [f32p, f32p, f32p, ci, ci, ci, ci, ci, ci, cd, ci,
                                            f64p, f64p]
            lib.oracle_attn_decode_rows.argtypes = [f32p, f32p, f32p, i32p, ci, ci, ci, ci, ci, cd,
                                                    i64p, cll, f64p, f64p]
            lib.oracle_decode_chunk_states.argtypes = [f32p, f32p, f32p, i32p, ci, ci, ci, ci, ci,
                                                       cd, ci, f64p, f64p, f64p, i64p]
            lib.oracle_attn_bwd.argtypes = [f32p, f32p, f32p, f32p, ci, ci, ci, ci, ci, ci, cd, ci,
                                            f64p, f64p, f64p, f64p, f64p]
            lib.oracle_attn_bwd_kvheads.argtypes = [f32p, f32p, f32p, f32p, ci, ci, ci, ci, ci, ci, cd,
                                                    ci, i64p, cll, f64p, f64p, f64p]
            lib.oracle_num_threads.argtypes = []
            for fn in (lib.oracle_attn_fwd_rows, lib.oracle_attn_fwd, lib.oracle_attn_decode_rows,
                       lib.oracle_decode_chunk_states, lib.oracle_attn_bwd, lib.oracle_attn_bwd_kvheads,
                       lib.oracle_num_threads):
                fn.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f32(a):
    a = np.ascontiguousarray(a, dtype=np.float32)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))


def _ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def attn_fwd(q, k, v, scale: float, causal: bool):
    """O [B,H,Sq,d] and LSE [B,H,Sq] (fp64) for q [B,H,Sq,d], k/v [B,Hkv,Sk,d]."""
    B, H, Sq, d = q.shape
    _, Hkv, Sk, _ = k.shape
    q, qp = _f32(q)
    k, kp = _f32(k)
    v, vp = _f32(v)
    o = np.empty((B, H, Sq, d), dtype=np.float64)
    lse = np.empty((B, H, Sq), dtype=np.float64)
    rc = _load().oracle_attn_fwd(qp, kp, vp, B, H, Hkv, Sq, Sk, d, float(scale), int(bool(causal)),
                                 _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double))
    if rc != 0:
        raise ValueError(f"oracle_attn_fwd rejected its arguments (rc={rc})")
    return o, lse


def attn_fwd_rows(q, k, v, scale: float, causal: bool, row_ids):
    """Selected rows only; row id = (b*H + h)*Sq + i.  Returns o [n,d], lse [n]."""
    B, H, Sq, d = q.shape
    _, Hkv, Sk, _ = k.shape
    q, qp = _f32(q)
    k, kp = _f32(k)
    v, vp = _f32(v)
    ids = np.ascontiguousarray(row_ids, dtype=np.int64)
    o = np.empty((len(ids), d), dtype=np.float64)
    lse = np.empty((len(ids),), dtype=np.float64)
    rc = _load().oracle_attn_fwd_rows(qp, kp, vp, B, H, Hkv, Sq, Sk, d, float(scale),
                                      int(bool(causal)), _ptr(ids, ctypes.c_longlong), len(ids),
                                      _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double))
    if rc != 0:
        raise ValueError(f"oracle_attn_fwd_rows rejected its arguments (rc={rc})")
    return o, lse


def attn_decode_rows(q, k, v, seqlens, scale: float, row_ids):
    """Decode rows; q [B,Hq,1,d], k/v [B,Hkv,Sk_max,d]; row id = b*Hq + h."""
    B, Hq, one, d = q.shape
    assert one == 1
    _, Hkv, Skm, _ = k.shape
    q, qp = _f32(q)
    k, kp = _f32(k)
    v, vp = _f32(v)
    sl = np.ascontiguousarray(seqlens, dtype=np.int32)
    ids = np.ascontiguousarray(row_ids, dtype=np.int64)
    o = np.empty((len(ids), d), dtype=np.float64)
    lse = np.empty((len(ids),), dtype=np.float64)
    rc = _load().oracle_attn_decode_rows(qp, kp, vp, _ptr(sl, ctypes.c_int), B, Hq, Hkv, Skm, d,
                                         float(scale), _ptr(ids, ctypes.c_longlong), len(ids),
                                         _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double))
    if rc != 0:
        raise ValueError(f"oracle_attn_decode_rows rejected its arguments (rc={rc})")
    return o, lse


def attn_decode(q, k, v, seqlens, scale: float):
    """All decode rows: O [B,Hq,1,d], LSE [B,Hq]."""
    B, Hq, _, d = q.shape
    o, lse = attn_decode_rows(q, k, v, seqlens, scale, np.arange(B * Hq))
    return o.reshape(B, Hq, 1, d), lse.reshape(B, Hq)


def decode_chunk_bounds(L: int, n_split: int):
    """Chunk c covers [floor(c*L/n), floor((c+1)*L/n)) -- the reading of
    "split the KV axis into n chunks" used by the oracle."""
    return [((c * L) // n_split, ((c + 1) * L) // n_split) for c in range(n_split)]


def decode_chunk_states(q, k, v, seqlens, scale: float, n_split: int):
    """Per-chunk canonical states (natural units): m, l [B,Hq,n], u [B,Hq,n,d], count."""
    B, Hq, _, d = q.shape
    _, Hkv, Skm, _ = k.shape
    q, qp = _f32(q)
    k, kp = _f32(k)
    v, vp = _f32(v)
    sl = np.ascontiguousarray(seqlens, dtype=np.int32)
    m = np.empty((B, Hq, n_split), dtype=np.float64)
    l = np.empty((B, Hq, n_split), dtype=np.float64)
    u = np.empty((B, Hq, n_split, d), dtype=np.float64)
    cnt = np.empty((B, Hq, n_split), dtype=np.int64)
    rc = _load().oracle_decode_chunk_states(qp, kp, vp, _ptr(sl, ctypes.c_int), B, Hq, Hkv, Skm, d,
                                            float(scale), n_split, _ptr(m, ctypes.c_double),
                                            _ptr(l, ctypes.c_double), _ptr(u, ctypes.c_double),
                                            _ptr(cnt, ctypes.c_longlong))
    if rc != 0:
        raise ValueError(f"oracle_decode_chunk_states rejected its arguments (rc={rc})")
    return m, l, u, cnt


def attn_bwd(q, k, v, dout, scale: float, causal: bool):
    """Exact backward from the definition (M4.4 0x06.1A), fp64.

    q, dout [B,H,Sq,d]; k, v [B,Hkv,Sk,d].  Returns dq [B,H,Sq,d],
    dk, dv [B,Hkv,Sk,d] (summed over each KV head's query-head group),
    the row scalars D = sum_j P_ij dP_ij [B,H,Sq] and LSE [B,H,Sq]."""
    B, H, Sq, d = q.shape
    _, Hkv, Sk, _ = k.shape
    q, qp = _f32(q)
    k, kp = _f32(k)
    v, vp = _f32(v)
    do, dop = _f32(dout)
    dq = np.empty((B, H, Sq, d), dtype=np.float64)
    dk = np.empty((B, Hkv, Sk, d), dtype=np.float64)
    dv = np.empty((B, Hkv, Sk, d), dtype=np.float64)
    D = np.empty((B, H, Sq), dtype=np.float64)
    lse = np.empty((B, H, Sq), dtype=np.float64)
    c = ctypes.c_double
    rc = _load().oracle_attn_bwd(qp, kp, vp, dop, B, H, Hkv, Sq, Sk, d, float(scale), int(bool(causal)),
                                 _ptr(dq, c), _ptr(dk, c), _ptr(dv, c), _ptr(D, c), _ptr(lse, c))
    if rc != 0:
        raise ValueError(f"oracle_attn_bwd rejected its arguments (rc={rc})")
    return dq, dk, dv, D, lse


def attn_bwd_kvheads(q, k, v, dout, scale: float, causal: bool, kv_ids):
    """Backward restricted to chosen KV heads, kv id = b*Hkv + kv_head.
    Returns dq [n, g, Sq, d] (the group's query heads), dk, dv [n, Sk, d]."""
    B, H, Sq, d = q.shape
    _, Hkv, Sk, _ = k.shape
    g = H // Hkv
    q, qp = _f32(q)
    k, kp = _f32(k)
    v, vp = _f32(v)
    do, dop = _f32(dout)
    ids = np.ascontiguousarray(kv_ids, dtype=np.int64)
    n = len(ids)
    dq = np.empty((n, g, Sq, d), dtype=np.float64)
    dk = np.empty((n, Sk, d), dtype=np.float64)
    dv = np.empty((n, Sk, d), dtype=np.float64)
    c = ctypes.c_double
    rc = _load().oracle_attn_bwd_kvheads(qp, kp, vp, dop, B, H, Hkv, Sq, Sk, d, float(scale),
                                         int(bool(causal)), _ptr(ids, ctypes.c_longlong), n,
                                         _ptr(dq, c), _ptr(dk, c), _ptr(dv, c))
    if rc != 0:
        raise ValueError(f"oracle_attn_bwd_kvheads rejected its arguments (rc={rc})")
    return dq, dk, dv
