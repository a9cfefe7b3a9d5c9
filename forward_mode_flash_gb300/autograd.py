"""PyTorch autograd / torch.func integration over the C ABI.

Mirrors the "JVP Flash Attention" project page (Usage section):

* ``JVPAttn.fwd_dual(q, k, v, attn_mask=None, is_causal=False, scale=None)``
  is the call a model makes inside ``torch.func.jvp(model, (x,), (gt,))``.
  When q, k, v carry forward-mode tangents of the innermost jvp level, one
  fused ``fwd_dual`` launch computes O and tO (no separate primal pass), and
  both are returned differentiable: the reverse mode through them runs
  ``bwd_dual``, so a loss of (O, tO) trains through the JVP and the gradient
  of the tangent output is a Hessian-vector product (reverse over forward).
  Called with explicit tangents, ``JVPAttn.fwd_dual(q, k, v, dq, dk, dv)``
  returns (O, tO) from the same fused call.
* ``jvp_attention(q, k, v, attn_mask=None, is_causal=False, scale=None)`` is a
  drop-in for ``scaled_dot_product_attention``.  Under ``torch.func.jvp`` it
  takes the same fused route; elsewhere it is an autograd.Function whose
  forward-mode rule calls ``fwd_dual`` and whose backward calls the
  primal-only ``bwd`` (no tangent terms).

All arithmetic runs in the library's kernels; this module only wires them
into autograd.
"""

from __future__ import annotations

from typing import Optional

import torch
import torch.autograd.forward_ad as fwAD

from . import api

_ft = torch._C._functorch


def _zeros_if_none(t, like):
    return torch.zeros_like(like) if t is None else t


def _dense_cotangent(g, like):
    """A storage-backed contiguous cotangent for the kernels.

    Autograd passes None, or a ZeroTensor (a zero without storage, e.g. for
    O when only the tangent output enters the loss), for outputs that do not
    reach the loss."""
    if g is None or g._is_zerotensor():
        return torch.zeros_like(like)
    return g.contiguous()


def _plain(t):
    """The storage-backed tensor under torch.func's wrappers.

    Under torch.func.jvp the tensors a function sees are wrapper tensors
    without storage; the kernels need the underlying device buffers.  The
    underlying tensor is the one of the enclosing (ordinary autograd) level,
    with its autograd history.
    """
    if t is None:
        return None
    while _ft.is_functorch_wrapped_tensor(t):
        t = _ft.get_unwrapped(t)
    return t


class _FwdDual(torch.autograd.Function):
    """(O, tO) of one fused fwd_dual call; backward = reverse mode of the dual map."""

    @staticmethod
    def forward(ctx, q, k, v, dq, dk, dv, attn_mask, is_causal, scale):
        o, t_o, lse, mu = api.fwd_dual(q, k, v, dq, dk, dv, attn_mask=attn_mask,
                                       is_causal=is_causal, scale=scale, return_stats=True)
        ctx.save_for_backward(q, k, v, dq, dk, dv, o, t_o, lse, mu)
        ctx.attn_mask, ctx.is_causal, ctx.scale = attn_mask, is_causal, scale
        return o, t_o

    @staticmethod
    def backward(ctx, g_o, g_to):
        q, k, v, dq, dk, dv, o, t_o, lse, mu = ctx.saved_tensors
        g_o = _dense_cotangent(g_o, o)
        g_to = _dense_cotangent(g_to, t_o)
        grads = api.bwd_dual(q, k, v, dq, dk, dv, o, t_o, lse, mu, g_o, g_to,
                             attn_mask=ctx.attn_mask, is_causal=ctx.is_causal, scale=ctx.scale)
        return (*grads, None, None, None)


def _fused_under_jvp(q, k, v, attn_mask, is_causal, scale):
    """O as a forward-mode dual (O, tO) from one fused call, or None.

    Applies when q, k, v are torch.func wrappers of the innermost transform
    level and at least one of them carries a forward-mode tangent there (the
    body of torch.func.jvp).  The primals and tangents are unwrapped to the
    enclosing level's tensors, one _FwdDual node is recorded in that level's
    autograd graph (so O and tO are differentiable through bwd_dual), and O
    and tO are wrapped back as the dual output of this level.  Anything else
    (no transform, other transforms such as vmap at this level, jvp nested in
    another transform) returns None.
    """
    level = _ft.maybe_current_level()
    if level is None:
        return None
    xs = (q, k, v)
    if not all(_ft.is_functorch_wrapped_tensor(x) and _ft.maybe_get_level(x) == level for x in xs):
        return None
    pairs = [fwAD.unpack_dual(x) for x in xs]
    if all(t is None for _, t in pairs):
        return None

    def one_level(t):  # the enclosing level's tensor (must be a plain one)
        return _ft.get_unwrapped(t) if _ft.is_functorch_wrapped_tensor(t) else t

    ps = [one_level(p) for p, _ in pairs]
    ts = [torch.zeros_like(p) if t is None else one_level(t) for p, (_, t) in zip(ps, pairs)]
    mask = None if attn_mask is None else one_level(attn_mask)
    if any(_ft.is_functorch_wrapped_tensor(t) for t in (*ps, *ts) + ((mask,) if mask is not None else ())):
        return None  # nested transforms: the generic forward-mode rule handles them
    # Record the node at the enclosing level: functorch's dispatch is off, and
    # the single-level Function is applied directly (torch.func would otherwise
    # insist on handling the Function at this level itself).
    prev = _ft.get_single_level_autograd_function_allowed()
    _ft.set_single_level_autograd_function_allowed(True)
    try:
        with torch._C._DisableFuncTorch():
            o, t_o = super(torch.autograd.Function, _FwdDual).apply(
                *ps, *ts, mask, is_causal, scale)
    finally:
        _ft.set_single_level_autograd_function_allowed(prev)
    return fwAD.make_dual(_ft._wrap_for_grad(o, level), _ft._wrap_for_grad(t_o, level))


class JVPAttn(torch.autograd.Function):
    """Attention with a forward-mode rule backed by the fused fwd_dual kernel."""

    @staticmethod
    def forward(q, k, v, attn_mask, is_causal, scale):
        o, lse = api.attention(q, k, v, attn_mask=attn_mask, is_causal=is_causal, scale=scale,
                               return_lse=True)
        return o, lse

    @staticmethod
    def setup_context(ctx, inputs, output):
        q, k, v, attn_mask, is_causal, scale = inputs
        o, lse = output
        ctx.save_for_forward(q, k, v, o, lse)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.attn_mask, ctx.is_causal, ctx.scale = attn_mask, is_causal, scale

    @staticmethod
    def jvp(ctx, dq, dk, dv, *_):
        # Outside torch.func's dispatch, so that the output buffers the binding
        # allocates are plain device tensors too.  (Reached for forward-mode AD
        # that the fused route above does not take, e.g. torch.autograd's
        # forward_ad dual tensors; the returned tangent has no autograd history.)
        with torch._C._DisableFuncTorch():
            q, k, v, _o, lse = (_plain(t) for t in ctx.saved_tensors)
            dq, dk, dv = (_zeros_if_none(_plain(t), x) for t, x in ((dq, q), (dk, k), (dv, v)))
            _, t_o, _, mu = api.fwd_dual(q, k, v, dq, dk, dv, attn_mask=_plain(ctx.attn_mask),
                                         is_causal=ctx.is_causal, scale=ctx.scale,
                                         return_stats=True)
        return t_o, mu  # mu is the tangent of lse

    @staticmethod
    def backward(ctx, g_o, _g_lse):
        # The primal-only backward (no tangent terms); lse is an auxiliary
        # output whose cotangent is not propagated.
        q, k, v, o, lse = ctx.saved_tensors
        g = api.bwd(q, k, v, o, lse, _dense_cotangent(g_o, o), attn_mask=ctx.attn_mask,
                    is_causal=ctx.is_causal, scale=ctx.scale)
        return g[0], g[1], g[2], None, None, None

    @staticmethod
    def fwd_dual(q, k, v, dq=None, dk=None, dv=None, attn_mask: Optional[torch.Tensor] = None,
                 is_causal: bool = False, scale: Optional[float] = None):
        """Attention whose forward-mode tangent comes from one fused pass.

        ``JVPAttn.fwd_dual(q, k, v)`` (the project page's form): inside
        torch.func.jvp returns O carrying its tangent tO, both from one fused
        launch and both differentiable through bwd_dual; outside any
        transform it is ``jvp_attention(q, k, v)``.

        ``JVPAttn.fwd_dual(q, k, v, dq, dk, dv)``: (O, tO) for explicit
        tangents (None = zero) from one fused launch, differentiable through
        bwd_dual with respect to all six inputs.
        """
        if dq is None and dk is None and dv is None:
            return jvp_attention(q, k, v, attn_mask=attn_mask, is_causal=is_causal, scale=scale)
        dq, dk, dv = (_zeros_if_none(t, x) for t, x in ((dq, q), (dk, k), (dv, v)))
        return _FwdDual.apply(q, k, v, dq, dk, dv, attn_mask, is_causal, scale)


def jvp_attention(q, k, v, attn_mask: Optional[torch.Tensor] = None, is_causal: bool = False,
                  scale: Optional[float] = None) -> torch.Tensor:
    """Drop-in for scaled_dot_product_attention with a fused forward-mode rule."""
    fused = _fused_under_jvp(q, k, v, attn_mask, is_causal, scale)
    if fused is not None:
        return fused
    o, _ = JVPAttn.apply(q, k, v, attn_mask, is_causal, scale)
    return o
