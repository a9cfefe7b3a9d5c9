"""Float64 CPU oracle for attention forward + JVP and its reverse mode.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` are the only callers.  The GPU library never
imports, links or runs anything here, and this package shares no code with it.

The arithmetic lives in ``jvp_oracle.cpp`` (plain C++17, dual numbers); this
module only compiles it with g++ and marshals numpy arrays through ctypes.
Every function is pinned by the CPU tests in ``tests/test_oracle_pins.py``.

Semantics follow the "JVP Flash Attention" project page (Description and Usage
sections): a drop-in for ``scaled_dot_product_attention(q, k, v, attn_mask)``
whose dual forward returns (O, tO) for tangents (dQ, dK, dV).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "jvp_oracle.cpp")
_LIB = os.path.join(_HERE, "_build", "libjvp_oracle.so")
_lock = threading.Lock()
_lib = None

MASK_NONE, MASK_BOOL, MASK_ADDITIVE, MASK_CAUSAL = 0, 1, 2, 3
_MASK_IDS = {"none": MASK_NONE, "bool": MASK_BOOL, "additive": MASK_ADDITIVE, "causal": MASK_CAUSAL}


def build(force: bool = False) -> str:
    """Compile the oracle shared library (g++ -O2, no architecture flags)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["g++", "-std=c++17", "-O2", "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, dp, vp, i32, f64 = (ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                                     ctypes.c_int, ctypes.c_double)
            common = [i64] * 5 + [dp] * 6 + [i32, vp] + [i64] * 4 + [f64]
            lib.oracle_fwd_dual_rows.argtypes = common + [vp, i64, dp, dp, dp, dp, i32]
            lib.oracle_fwd_dual_rows.restype = i32
            lib.oracle_fwd_dual.argtypes = common + [dp, dp, dp, dp, i32]
            lib.oracle_fwd_dual.restype = i32
            lib.oracle_bwd_dual.argtypes = common + [dp] * 8 + [i32]
            lib.oracle_bwd_dual.restype = i32
            lib.oracle_default_threads.argtypes = []
            lib.oracle_default_threads.restype = i32
            _lib = lib
    return _lib


def default_threads() -> int:
    """Worker threads the oracle uses when nthreads <= 0 (all host cores)."""
    return int(_load().oracle_default_threads())


def _f64(x):
    if x is None:
        return None
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _mask_args(mask_kind, mask, B, H, Nq, Nk):
    """Normalise a mask to (kind id, contiguous array or None, element strides)."""
    kind = _MASK_IDS[mask_kind] if isinstance(mask_kind, str) else int(mask_kind)
    if kind in (MASK_NONE, MASK_CAUSAL):
        return kind, None, (0, 0, 0, 0)
    if kind == MASK_BOOL:
        arr = np.ascontiguousarray(np.asarray(mask).astype(np.uint8))
    else:
        arr = np.ascontiguousarray(np.asarray(mask, dtype=np.float64))
    if arr.ndim != 4 or arr.shape[2:] != (Nq, Nk) or arr.shape[0] not in (1, B) or arr.shape[1] not in (1, H):
        raise ValueError(f"mask shape {arr.shape} does not broadcast to {(B, H, Nq, Nk)}")
    st = [s // arr.itemsize for s in arr.strides]
    sb = 0 if arr.shape[0] == 1 else st[0]
    sh = 0 if arr.shape[1] == 1 else st[1]
    return kind, arr, (sb, sh, st[2], st[3])


def fwd_dual(q, k, v, dq=None, dk=None, dv=None, mask_kind="none", mask=None, scale=None,
             nthreads=0):
    """Float64 forward + JVP over all rows.

    q [B,H,Nq,D], k/v [B,H,Nk,D]; tangents of the same shapes or None (zero).
    Returns (o, t_o, lse, mu) as float64 numpy arrays.
    """
    q, k, v, dq, dk, dv = map(_f64, (q, k, v, dq, dk, dv))
    B, H, Nq, D = q.shape
    Nk = k.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    kind, m, (sb, sh, sq, sk) = _mask_args(mask_kind, mask, B, H, Nq, Nk)
    o = np.empty((B, H, Nq, D))
    t_o = np.empty((B, H, Nq, D))
    lse = np.empty((B, H, Nq))
    mu = np.empty((B, H, Nq))
    rc = _load().oracle_fwd_dual(B, H, Nq, Nk, D, _ptr(q), _ptr(k), _ptr(v), _ptr(dq), _ptr(dk),
                                 _ptr(dv), kind, _ptr(m), sb, sh, sq, sk, float(scale), _ptr(o),
                                 _ptr(t_o), _ptr(lse), _ptr(mu), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_fwd_dual rejected its arguments")
    return o, t_o, lse, mu


def fwd_dual_rows(q, k, v, dq, dk, dv, row_ids, mask_kind="none", mask=None, scale=None,
                  nthreads=0):
    """Forward + JVP for selected rows only; row_ids are flat (b*H + h)*Nq + i.

    Returns compact (o [R,D], t_o [R,D], lse [R], mu [R]).
    """
    q, k, v, dq, dk, dv = map(_f64, (q, k, v, dq, dk, dv))
    B, H, Nq, D = q.shape
    Nk = k.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    kind, m, (sb, sh, sq, sk) = _mask_args(mask_kind, mask, B, H, Nq, Nk)
    ids = np.ascontiguousarray(np.asarray(row_ids, dtype=np.int64))
    R = ids.shape[0]
    o = np.empty((R, D))
    t_o = np.empty((R, D))
    lse = np.empty((R,))
    mu = np.empty((R,))
    rc = _load().oracle_fwd_dual_rows(B, H, Nq, Nk, D, _ptr(q), _ptr(k), _ptr(v), _ptr(dq),
                                      _ptr(dk), _ptr(dv), kind, _ptr(m), sb, sh, sq, sk,
                                      float(scale), _ptr(ids), R, _ptr(o), _ptr(t_o), _ptr(lse),
                                      _ptr(mu), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_fwd_dual_rows rejected its arguments")
    return o, t_o, lse, mu


def bwd_dual(q, k, v, dq, dk, dv, g_o, g_to, mask_kind="none", mask=None, scale=None,
             nthreads=0):
    """Gradients of <g_o, O> + <g_to, tO> w.r.t. (q, k, v, dq, dk, dv), float64."""
    q, k, v, dq, dk, dv, g_o, g_to = map(_f64, (q, k, v, dq, dk, dv, g_o, g_to))
    B, H, Nq, D = q.shape
    Nk = k.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    kind, m, (sb, sh, sq, sk) = _mask_args(mask_kind, mask, B, H, Nq, Nk)
    outs = [np.empty_like(q), np.empty_like(k), np.empty_like(v), np.empty_like(q),
            np.empty_like(k), np.empty_like(v)]
    rc = _load().oracle_bwd_dual(B, H, Nq, Nk, D, _ptr(q), _ptr(k), _ptr(v), _ptr(dq), _ptr(dk),
                                 _ptr(dv), kind, _ptr(m), sb, sh, sq, sk, float(scale),
                                 _ptr(g_o), _ptr(g_to), *[_ptr(x) for x in outs], int(nthreads))
    if rc != 0:
        raise ValueError("oracle_bwd_dual rejected its arguments")
    return tuple(outs)
