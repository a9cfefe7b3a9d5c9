"""PyTorch autograd / torch.func integration over the C ABI.

Mirrors the "JVP Flash Attention" project page (Usage section):

* ``jvp_attention(q, k, v, attn_mask=None, is_causal=False, scale=None)`` is a
  drop-in for ``scaled_dot_product_attention``.  Under ``torch.func.jvp`` its
  forward-mode rule calls the fused ``fwd_dual`` kernel (O and tO in one
  pass); under reverse mode its backward calls ``bwd_dual`` with zero tangents.
* ``JVPAttn.fwd_dual(q, k, v, dq, dk, dv, ...)`` returns ``(O, tO)`` from one
  fused call and is itself differentiable: its backward is the reverse mode of
  the dual computation, which is what training through a JVP or a
  Hessian-vector product needs.

All arithmetic runs in the library's kernels; this module only wires them
into autograd.
"""

from __future__ import annotations

from typing import Optional

import torch

from . import api


def _zeros_if_none(t, like):
    return torch.zeros_like(like) if t is None else t


def _plain(t):
    """The storage-backed tensor under torch.func's wrappers.

    Under torch.func.jvp the tangents handed to a Function's jvp rule are
    wrapper tensors without storage; the kernels need the underlying device
    buffers, so the rule unwraps them and returns a plain tensor, which
    torch.func accepts as the output tangent.
    """
    if t is None:
        return None
    ft = torch._C._functorch
    while ft.is_functorch_wrapped_tensor(t):
        t = ft.get_unwrapped(t)
    return t


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
        # allocates are plain device tensors too.
        with torch._C._DisableFuncTorch():
            q, k, v, _o, lse = (_plain(t) for t in ctx.saved_tensors)
            dq, dk, dv = (_zeros_if_none(_plain(t), x) for t, x in ((dq, q), (dk, k), (dv, v)))
            _, t_o, _, mu = api.fwd_dual(q, k, v, dq, dk, dv, attn_mask=_plain(ctx.attn_mask),
                                         is_causal=ctx.is_causal, scale=ctx.scale,
                                         return_stats=True)
        return t_o, mu  # mu is the tangent of lse

    @staticmethod
    def backward(ctx, g_o, _g_lse):
        q, k, v, o, lse = ctx.saved_tensors
        zq, zk = torch.zeros_like(q), torch.zeros_like(k)
        zmu = torch.zeros_like(lse)
        g = api.bwd_dual(q, k, v, zq, zk, torch.zeros_like(v), o, torch.zeros_like(o), lse, zmu,
                         g_o.contiguous(), torch.zeros_like(o), attn_mask=ctx.attn_mask,
                         is_causal=ctx.is_causal, scale=ctx.scale)
        return g[0], g[1], g[2], None, None, None

    @staticmethod
    def fwd_dual(q, k, v, dq, dk, dv, attn_mask: Optional[torch.Tensor] = None,
                 is_causal: bool = False, scale: Optional[float] = None):
        """(O, tO) from one fused pass; differentiable through bwd_dual."""
        return _FwdDual.apply(q, k, v, dq, dk, dv, attn_mask, is_causal, scale)


class _FwdDual(torch.autograd.Function):
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
        g_o = _zeros_if_none(g_o, o).contiguous()
        g_to = _zeros_if_none(g_to, t_o).contiguous()
        grads = api.bwd_dual(q, k, v, dq, dk, dv, o, t_o, lse, mu, g_o, g_to,
                             attn_mask=ctx.attn_mask, is_causal=ctx.is_causal, scale=ctx.scale)
        return (*grads, None, None, None)


def jvp_attention(q, k, v, attn_mask: Optional[torch.Tensor] = None, is_causal: bool = False,
                  scale: Optional[float] = None) -> torch.Tensor:
    """Drop-in for scaled_dot_product_attention with a fused forward-mode rule."""
    o, _ = JVPAttn.apply(q, k, v, attn_mask, is_causal, scale)
    return o
