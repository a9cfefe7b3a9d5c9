"""Python binding of the C ABI: argument marshalling only.

Every step of the computation runs in the library's CUDA kernels; this module
allocates the output tensors with PyTorch, reads pointers, strides and the
current stream, and calls the entry points declared in ``include/jvp_attn.h``.

API shaped after the "JVP Flash Attention" project page (Usage section):
``attention(q, k, v, attn_mask=...)`` is the forward, and ``fwd_dual`` returns
the output together with its tangent for tangents (dq, dk, dv), as
``JVPAttn.fwd_dual`` does under ``torch.func.jvp``.
"""

from __future__ import annotations

import ctypes
import math
from typing import Optional, Tuple

import torch

from . import _abi

_DT = {torch.float32: _abi.JVP_F32, torch.float16: _abi.JVP_F16, torch.bfloat16: _abi.JVP_BF16}


def _strides(t: torch.Tensor) -> _abi.Strides:
    sb, sh, sn, sd = t.stride()
    return _abi.Strides(sb, sh, sn, sd)


_KV_NAMES = frozenset(("k", "v", "dk", "dv"))


def _check_inputs(tensors, names) -> int:
    """Checks dtype, device, rank and sizes; returns the key/value head count.

    Key-side tensors (k, v, dk, dv) may have fewer heads than the queries
    (grouped-query attention) as long as the query heads are a multiple.
    """
    ref = tensors[0]
    if ref.dim() != 4:
        raise ValueError(f"{names[0]} must be [B, H, N, D], got {tuple(ref.shape)}")
    if ref.dtype not in _DT:
        raise TypeError(f"unsupported dtype {ref.dtype}")
    if ref.device.type != "cuda":
        raise ValueError("tensors must be on a CUDA device")
    H = ref.shape[1]
    hkv = next((t.shape[1] for t, n in zip(tensors, names) if n in _KV_NAMES and t.dim() == 4), H)
    if hkv <= 0 and H > 0 or (hkv > 0 and H % hkv != 0):
        raise ValueError(f"query heads ({H}) must be a multiple of key/value heads ({hkv})")
    for t, n in zip(tensors, names):
        if t.dtype != ref.dtype or t.device != ref.device or t.dim() != 4:
            raise ValueError(f"{n} must be a 4-D {ref.dtype} tensor on {ref.device}")
        heads = hkv if n in _KV_NAMES else H
        if t.shape[-1] != ref.shape[-1] or t.shape[0] != ref.shape[0] or t.shape[1] != heads:
            raise ValueError(f"{n} has shape {tuple(t.shape)}, inconsistent with {tuple(ref.shape)}")
        if t.stride(-1) != 1 and t.numel() > 0:
            raise ValueError(f"{n} must have a unit innermost stride")
    return hkv


def _mask_desc(attn_mask: Optional[torch.Tensor], is_causal: bool, B, H, Nq, Nk, device):
    """Mask description (and the tensor it points into, kept alive by the caller).

    ``is_causal`` together with ``attn_mask`` keeps a key only where both do
    (an extension: scaled_dot_product_attention rejects the combination).
    """
    if attn_mask is None:
        kind = _abi.JVP_MASK_CAUSAL if is_causal else _abi.JVP_MASK_NONE
        return _abi.Mask(kind, None, 0, 0, 0, 0), None
    if attn_mask.device != device:
        raise ValueError("attn_mask must be on the same device as q")
    if attn_mask.dtype == torch.bool:
        kind, m = _abi.JVP_MASK_BOOL, attn_mask.view(torch.uint8)
        if is_causal:
            kind = _abi.JVP_MASK_BOOL_CAUSAL
    elif attn_mask.dtype == torch.float32:
        kind, m = _abi.JVP_MASK_ADDITIVE, attn_mask
        if is_causal:
            kind = _abi.JVP_MASK_ADDITIVE_CAUSAL
    else:
        raise TypeError("attn_mask must be torch.bool (keep-mask) or torch.float32 (additive)")
    while m.dim() < 4:
        m = m.unsqueeze(0)
    m = m.expand(B, H, Nq, Nk)  # broadcast dimensions get stride 0
    sb, sh, sq, sk = m.stride()
    return _abi.Mask(kind, m.data_ptr(), sb, sh, sq, sk), m


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def fwd_dual(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, dq: torch.Tensor,
             dk: torch.Tensor, dv: torch.Tensor, attn_mask: Optional[torch.Tensor] = None,
             is_causal: bool = False, scale: Optional[float] = None, return_stats: bool = False,
             out: Optional[Tuple[torch.Tensor, ...]] = None, split_kv: bool = True,
             workspace: Optional[torch.Tensor] = None):
    """Attention forward and its JVP in one fused pass.

    Returns (o, t_o), or (o, t_o, lse, mu) with ``return_stats``: lse is the
    natural-log log-sum-exp per row and mu its tangent, both float32 [B,H,Nq].
    ``out`` = (o, t_o) or (o, t_o, lse, mu) gives preallocated outputs (the
    four-tuple implies ``return_stats``).  With ``split_kv`` (the default),
    problems with fewer query tiles than SMs split their key range over
    several CTAs through ``jvp_attn_fwd_dual_ws``; the scratch it needs
    (``fwd_dual_workspace_size``) is allocated here unless ``workspace`` (a
    16-byte-aligned uint8 device tensor) is given.
    """
    lib = _abi.load()
    if attn_mask is None and out is None and workspace is None:
        plan = _fwd_plan(lib, q, k, v, dq, dk, dv, is_causal, split_kv)
        if plan is not None:
            return _fwd_dual_planned(lib, plan, q, k, v, dq, dk, dv, scale, return_stats)
    hkv = _check_inputs([q, k, v, dq, dk, dv], ["q", "k", "v", "dq", "dk", "dv"])
    B, H, Nq, D = q.shape
    Nk = k.shape[2]
    for t, n in ((v, "v"), (dk, "dk"), (dv, "dv")):
        if t.shape[2] != Nk:
            raise ValueError(f"{n} must have {Nk} rows")
    if dq.shape[2] != Nq:
        raise ValueError("dq must match q")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        o = torch.empty((B, H, Nq, D), dtype=q.dtype, device=q.device)
        t_o = torch.empty_like(o)
    else:
        o, t_o = out[0], out[1]
    if out is not None and len(out) == 4:
        lse, mu = out[2], out[3]
        for t, n in ((lse, "lse"), (mu, "mu")):
            if (t.dtype != torch.float32 or tuple(t.shape) != (B, H, Nq) or not t.is_contiguous()
                    or t.device != q.device):
                raise ValueError(f"out {n} must be a contiguous float32 [B, H, Nq] device tensor")
        return_stats = True
    else:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device) if return_stats else None
        mu = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device) if return_stats else None
    mask, _keep = _mask_desc(attn_mask, is_causal, B, H, Nq, Nk, q.device)
    ins = (_abi.Strides * 6)(*[_strides(t) for t in (q, k, v, dq, dk, dv)])
    outs = (_abi.Strides * 2)(_strides(o), _strides(t_o))
    shape = _abi.Shape(B, H, Nq, Nk, D, hkv)
    stream = torch.cuda.current_stream(q.device).cuda_stream
    with torch.cuda.device(q.device):
        need = _split_ws_bytes(lib, shape, q) if split_kv else 0
        if need > 0:
            if workspace is None:
                workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
            st = lib.jvp_attn_fwd_dual_ws(ctypes.byref(shape), _DT[q.dtype], _ptr(q), _ptr(k),
                                          _ptr(v), _ptr(dq), _ptr(dk), _ptr(dv), ins,
                                          ctypes.byref(mask), float(scale), _ptr(o), _ptr(t_o),
                                          outs, _ptr(lse), _ptr(mu), _ptr(workspace),
                                          workspace.numel() * workspace.element_size(),
                                          ctypes.c_void_p(stream))
        else:
            st = lib.jvp_attn_fwd_dual(ctypes.byref(shape), _DT[q.dtype], _ptr(q), _ptr(k),
                                       _ptr(v), _ptr(dq), _ptr(dk), _ptr(dv), ins,
                                       ctypes.byref(mask), float(scale), _ptr(o), _ptr(t_o),
                                       outs, _ptr(lse), _ptr(mu), ctypes.c_void_p(stream))
    _abi.check(st)
    if return_stats:
        return o, t_o, lse, mu
    return o, t_o


# Validated call descriptions for repeated fwd_dual calls on tensors of the
# same dtypes, devices, shapes and strides (no mask tensor, fresh outputs):
# the ctypes records are built once and only the pointers change per call.
_FWD_PLANS = {}
_FWD_PLANS_MAX = 256


class _FwdPlan:
    __slots__ = ("shape", "ins", "outs", "mask", "dt", "need", "oshape", "sshape", "scale",
                 "dtype", "device", "dev_index")


def _fwd_plan(lib, q, k, v, dq, dk, dv, is_causal, split_kv):
    ts = (q, k, v, dq, dk, dv)
    key = (tuple((t.dtype, t.device, t.shape, t.stride()) for t in ts), bool(is_causal),
           bool(split_kv))
    plan = _FWD_PLANS.get(key)
    if plan is not None:
        return plan
    hkv = _check_inputs(list(ts), ["q", "k", "v", "dq", "dk", "dv"])
    B, H, Nq, D = q.shape
    Nk = k.shape[2]
    if v.shape[2] != Nk or dk.shape[2] != Nk or dv.shape[2] != Nk or dq.shape[2] != Nq:
        return None  # the general path reports the mismatch
    plan = _FwdPlan()
    plan.shape = _abi.Shape(B, H, Nq, Nk, D, hkv)
    plan.ins = (_abi.Strides * 6)(*[_strides(t) for t in ts])
    # outputs are allocated contiguous [B, H, Nq, D]
    plan.outs = (_abi.Strides * 2)(*[_abi.Strides(H * Nq * D, Nq * D, D, 1)] * 2)
    plan.mask = _abi.Mask(_abi.JVP_MASK_CAUSAL if is_causal else _abi.JVP_MASK_NONE, None,
                          0, 0, 0, 0)
    plan.dt = _DT[q.dtype]
    plan.dtype, plan.device, plan.dev_index = q.dtype, q.device, q.device.index
    plan.oshape, plan.sshape = (B, H, Nq, D), (B, H, Nq)
    plan.scale = 1.0 / math.sqrt(D)
    with torch.cuda.device(q.device):
        plan.need = _split_ws_bytes(lib, plan.shape, q) if split_kv else 0
    if len(_FWD_PLANS) >= _FWD_PLANS_MAX:
        _FWD_PLANS.clear()
    _FWD_PLANS[key] = plan
    return plan


def _fwd_dual_planned(lib, plan, q, k, v, dq, dk, dv, scale, return_stats):
    dev = plan.device
    o = torch.empty(plan.oshape, dtype=plan.dtype, device=dev)
    t_o = torch.empty(plan.oshape, dtype=plan.dtype, device=dev)
    lse = mu = None
    if return_stats:
        lse = torch.empty(plan.sshape, dtype=torch.float32, device=dev)
        mu = torch.empty(plan.sshape, dtype=torch.float32, device=dev)
    sc = plan.scale if scale is None else float(scale)
    guard = torch.cuda.current_device() != plan.dev_index
    if guard:
        ctx = torch.cuda.device(dev)
        ctx.__enter__()
    try:
        stream = torch.cuda.current_stream(plan.dev_index).cuda_stream
        lp = lse.data_ptr() if lse is not None else None
        mp = mu.data_ptr() if mu is not None else None
        if plan.need > 0:
            ws = torch.empty(plan.need, dtype=torch.uint8, device=dev)
            st = lib.jvp_attn_fwd_dual_ws(ctypes.byref(plan.shape), plan.dt, q.data_ptr(),
                                          k.data_ptr(), v.data_ptr(), dq.data_ptr(),
                                          dk.data_ptr(), dv.data_ptr(), plan.ins,
                                          ctypes.byref(plan.mask), sc, o.data_ptr(),
                                          t_o.data_ptr(), plan.outs, lp, mp, ws.data_ptr(),
                                          plan.need, stream)
        else:
            st = lib.jvp_attn_fwd_dual(ctypes.byref(plan.shape), plan.dt, q.data_ptr(),
                                       k.data_ptr(), v.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                       dv.data_ptr(), plan.ins, ctypes.byref(plan.mask), sc,
                                       o.data_ptr(), t_o.data_ptr(), plan.outs, lp, mp, stream)
    finally:
        if guard:
            ctx.__exit__(None, None, None)
    _abi.check(st)
    if return_stats:
        return o, t_o, lse, mu
    return o, t_o


_split_ws_cache = {}


def _split_ws_bytes(lib, shape, q) -> int:
    """jvp_attn_fwd_dual_workspace_size, cached per device and shape."""
    key = (q.device.index, shape.B, shape.H, shape.Nq, shape.Nk, shape.D, q.dtype)
    need = _split_ws_cache.get(key)
    if need is None:
        need = int(lib.jvp_attn_fwd_dual_workspace_size(ctypes.byref(shape), _DT[q.dtype]))
        _split_ws_cache[key] = need
    return need


def fwd_dual_workspace_size(B: int, H: int, Nq: int, Nk: int, D: int,
                            dtype: torch.dtype = torch.bfloat16, Hkv: int = 0) -> int:
    """Bytes of scratch with which fwd_dual splits the key range (0: no split)."""
    shape = _abi.Shape(B, H, Nq, Nk, D, Hkv)
    return int(_abi.load().jvp_attn_fwd_dual_workspace_size(ctypes.byref(shape), _DT[dtype]))


def fwd_dual_host_workspace_size(B: int, H: int, Nq: int, Nk: int, D: int,
                                 dtype: torch.dtype = torch.bfloat16, chunks: int = 4) -> int:
    """Device staging bytes of fwd_dual_host for this shape and chunk count."""
    shape = _abi.Shape(B, H, Nq, Nk, D, 0)
    return int(_abi.load().jvp_attn_fwd_dual_host_workspace_size(ctypes.byref(shape),
                                                                 _DT[dtype], int(chunks)))


def attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
              attn_mask: Optional[torch.Tensor] = None, is_causal: bool = False,
              scale: Optional[float] = None, return_lse: bool = False,
              out: Optional[torch.Tensor] = None):
    """Attention forward only (no tangents): o, or (o, lse) with ``return_lse``."""
    lib = _abi.load()
    hkv = _check_inputs([q, k, v], ["q", "k", "v"])
    B, H, Nq, D = q.shape
    Nk = k.shape[2]
    if v.shape[2] != Nk:
        raise ValueError("v must match k")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    o = torch.empty((B, H, Nq, D), dtype=q.dtype, device=q.device) if out is None else out
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device) if return_lse else None
    mask, _keep = _mask_desc(attn_mask, is_causal, B, H, Nq, Nk, q.device)
    ins = (_abi.Strides * 3)(*[_strides(t) for t in (q, k, v)])
    outs = (_abi.Strides * 1)(_strides(o))
    shape = _abi.Shape(B, H, Nq, Nk, D, hkv)
    stream = torch.cuda.current_stream(q.device).cuda_stream
    with torch.cuda.device(q.device):
        st = lib.jvp_attn_fwd(ctypes.byref(shape), _DT[q.dtype], _ptr(q), _ptr(k), _ptr(v), ins,
                              ctypes.byref(mask), float(scale), _ptr(o), outs, _ptr(lse),
                              ctypes.c_void_p(stream))
    _abi.check(st)
    return (o, lse) if return_lse else o


def bwd_dual_workspace_size(B: int, H: int, Nq: int, Nk: int, D: int,
                            dtype: torch.dtype = torch.bfloat16, hkv: int = 0) -> int:
    """Bytes of device scratch jvp_attn_bwd_dual needs for this shape on the
    current device (``hkv``: key/value heads, 0 = H)."""
    shape = _abi.Shape(B, H, Nq, Nk, D, hkv)
    return int(_abi.load().jvp_attn_bwd_dual_workspace_size(ctypes.byref(shape), _DT[dtype]))


def bwd_dual(q, k, v, dq, dk, dv, o, t_o, lse, mu, g_o, g_to,
             attn_mask: Optional[torch.Tensor] = None, is_causal: bool = False,
             scale: Optional[float] = None, workspace: Optional[torch.Tensor] = None):
    """Gradients of <g_o, O> + <g_to, tO> with respect to (q, k, v, dq, dk, dv).

    o, t_o, lse, mu are the outputs of ``fwd_dual(..., return_stats=True)`` on
    the same inputs.  ``workspace`` (uint8, on q's device) is allocated here if
    not given; its size is ``bwd_dual_workspace_size``.
    """
    lib = _abi.load()
    hkv = _check_inputs([q, k, v, dq, dk, dv, o, t_o, g_o, g_to],
                        ["q", "k", "v", "dq", "dk", "dv", "o", "t_o", "g_o", "g_to"])
    B, H, Nq, D = q.shape
    Nk = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    for t, n in ((lse, "lse"), (mu, "mu")):
        if t.dtype != torch.float32 or tuple(t.shape) != (B, H, Nq) or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous float32 [B, H, Nq] tensor")
    outs = [torch.empty_like(x) for x in (q, k, v, dq, dk, dv)]
    need = bwd_dual_workspace_size(B, H, Nq, Nk, D, q.dtype, hkv)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    mask, _keep = _mask_desc(attn_mask, is_causal, B, H, Nq, Nk, q.device)
    ins = (_abi.Strides * 10)(*[_strides(t) for t in (q, k, v, dq, dk, dv, o, t_o, g_o, g_to)])
    ost = (_abi.Strides * 6)(*[_strides(t) for t in outs])
    shape = _abi.Shape(B, H, Nq, Nk, D, hkv)
    stream = torch.cuda.current_stream(q.device).cuda_stream
    with torch.cuda.device(q.device):
        st = lib.jvp_attn_bwd_dual(ctypes.byref(shape), _DT[q.dtype], _ptr(q), _ptr(k), _ptr(v),
                                   _ptr(dq), _ptr(dk), _ptr(dv), _ptr(o), _ptr(t_o), _ptr(lse),
                                   _ptr(mu), _ptr(g_o), _ptr(g_to), ins, ctypes.byref(mask),
                                   float(scale), *[_ptr(x) for x in outs], ost, _ptr(workspace),
                                   workspace.numel() * workspace.element_size(),
                                   ctypes.c_void_p(stream))
    _abi.check(st)
    return tuple(outs)


def bwd_workspace_size(B: int, H: int, Nq: int, Nk: int, D: int,
                       dtype: torch.dtype = torch.bfloat16, hkv: int = 0) -> int:
    """Bytes of device scratch jvp_attn_bwd needs for this shape on the
    current device (``hkv``: key/value heads, 0 = H)."""
    shape = _abi.Shape(B, H, Nq, Nk, D, hkv)
    return int(_abi.load().jvp_attn_bwd_workspace_size(ctypes.byref(shape), _DT[dtype]))


def bwd(q, k, v, o, lse, g_o, attn_mask: Optional[torch.Tensor] = None, is_causal: bool = False,
        scale: Optional[float] = None, workspace: Optional[torch.Tensor] = None):
    """Gradients of <g_o, O> with respect to (q, k, v): the backward of
    attention without tangents.

    o, lse are the outputs of ``attention(..., return_lse=True)`` (or of
    ``fwd_dual``) on the same inputs.  ``workspace`` (uint8, on q's device) is
    allocated here if not given; its size is ``bwd_workspace_size``.
    """
    lib = _abi.load()
    hkv = _check_inputs([q, k, v, o, g_o], ["q", "k", "v", "o", "g_o"])
    B, H, Nq, D = q.shape
    Nk = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, Nq) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 [B, H, Nq] tensor")
    outs = [torch.empty_like(x) for x in (q, k, v)]
    need = bwd_workspace_size(B, H, Nq, Nk, D, q.dtype, hkv)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    mask, _keep = _mask_desc(attn_mask, is_causal, B, H, Nq, Nk, q.device)
    ins = (_abi.Strides * 5)(*[_strides(t) for t in (q, k, v, o, g_o)])
    ost = (_abi.Strides * 3)(*[_strides(t) for t in outs])
    shape = _abi.Shape(B, H, Nq, Nk, D, hkv)
    stream = torch.cuda.current_stream(q.device).cuda_stream
    with torch.cuda.device(q.device):
        st = lib.jvp_attn_bwd(ctypes.byref(shape), _DT[q.dtype], _ptr(q), _ptr(k), _ptr(v),
                              _ptr(o), _ptr(lse), _ptr(g_o), ins, ctypes.byref(mask),
                              float(scale), *[_ptr(x) for x in outs], ost, _ptr(workspace),
                              workspace.numel() * workspace.element_size(),
                              ctypes.c_void_p(stream))
    _abi.check(st)
    return tuple(outs)


def fwd_dual_host(q, k, v, dq, dk, dv, attn_mask: Optional[torch.Tensor] = None,
                  is_causal: bool = False, scale: Optional[float] = None, chunks: int = 4,
                  device=None, out: Optional[Tuple[torch.Tensor, ...]] = None,
                  return_stats: bool = False, workspace: Optional[torch.Tensor] = None):
    """fwd_dual for host-resident tensors through ``jvp_attn_fwd_dual_host``.

    q, k, v, dq, dk, dv are contiguous CPU tensors [B, H, N, D] (pinned memory
    lets the copies overlap the kernels).  The library pipelines the copies in,
    the fused kernel and the copies out over ``chunks`` groups of (batch,
    head) pairs.  Returns CPU tensors (O, tO) (plus lse, mu with
    ``return_stats``), or fills ``out``.  A mask must be shared by every
    (batch, head): [Nq, Nk] or [1, 1, Nq, Nk]; it is copied to the device.
    """
    lib = _abi.load()
    dev = torch.device(device) if device is not None else torch.device("cuda",
                                                                        torch.cuda.current_device())
    B, H, Nq, D = q.shape
    Nk = k.shape[2]
    for t in (q, k, v, dq, dk, dv):
        if t.device.type != "cpu" or not t.is_contiguous() or t.dtype != q.dtype:
            raise ValueError("fwd_dual_host takes contiguous CPU tensors of one dtype")
    if k.shape[1] != H:
        raise ValueError("fwd_dual_host needs as many key/value heads as query heads")
    if q.dtype not in _DT:
        raise TypeError(f"unsupported dtype {q.dtype}")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    mask_d = None
    if attn_mask is not None:
        m = attn_mask
        while m.dim() > 2 and m.shape[0] == 1:
            m = m[0]
        if m.dim() != 2:
            raise ValueError("fwd_dual_host needs a mask shared by all batches and heads")
        mask_d = m.to(dev, non_blocking=True)
    mask, _keep = _mask_desc(mask_d, is_causal, 1, 1, Nq, Nk, dev)
    mask.stride_b = mask.stride_h = 0
    pin = q.is_pinned()
    if out is None:
        o_h = torch.empty((B, H, Nq, D), dtype=q.dtype, pin_memory=pin)
        t_h = torch.empty((B, H, Nq, D), dtype=q.dtype, pin_memory=pin)
        lse_h = torch.empty((B, H, Nq), dtype=torch.float32, pin_memory=pin) if return_stats else None
        mu_h = torch.empty((B, H, Nq), dtype=torch.float32, pin_memory=pin) if return_stats else None
    else:
        o_h, t_h = out[0], out[1]
        lse_h, mu_h = (out[2], out[3]) if len(out) == 4 else (None, None)
    shape = _abi.Shape(B, H, Nq, Nk, D, 0)
    need = int(lib.jvp_attn_fwd_dual_host_workspace_size(ctypes.byref(shape), _DT[q.dtype],
                                                         int(chunks)))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    with torch.cuda.device(dev):
        st = lib.jvp_attn_fwd_dual_host(ctypes.byref(shape), _DT[q.dtype], _ptr(q), _ptr(k),
                                        _ptr(v), _ptr(dq), _ptr(dk), _ptr(dv), ctypes.byref(mask),
                                        float(scale), _ptr(o_h), _ptr(t_h), _ptr(lse_h),
                                        _ptr(mu_h), int(chunks), _ptr(workspace),
                                        workspace.numel() * workspace.element_size(),
                                        ctypes.c_void_p(stream))
    _abi.check(st)
    # keep the staging area and the device mask alive until the stream is done
    workspace.record_stream(torch.cuda.current_stream(dev))
    if mask_d is not None:
        mask_d.record_stream(torch.cuda.current_stream(dev))
    if return_stats or (out is not None and len(out) == 4):
        return o_h, t_h, lse_h, mu_h
    return o_h, t_h


def device_status(stream: Optional[torch.cuda.Stream] = None) -> int:
    """Synchronise the stream and return (and clear) the library's device status."""
    lib = _abi.load()
    s = (stream or torch.cuda.current_stream()).cuda_stream
    return int(lib.jvp_attn_get_device_status(ctypes.c_void_p(s)))


def last_path() -> int:
    """Kernel family of the last call on this thread: 1 tensor-core, 2 CUDA-core,
    3 tensor-core with split-KV and the merge kernel, 4 tensor-core with each
    query tile's key range split between the two CTAs of a cluster."""
    return int(_abi.load().jvp_attn_debug_last_path())


TENSOR_CORE_PATHS = (1, 3, 4)


def set_cluster_split(enable: bool) -> None:
    """Diagnostic: allow (default) or forbid the cluster key split (process-wide)."""
    _abi.check(_abi.load().jvp_attn_debug_set_cluster_split(1 if enable else 0))
