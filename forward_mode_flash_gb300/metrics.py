"""Work and traffic counts used to report throughput and roofline fractions.

FLOPs: the algorithmic count of the six N x N x D products of the dual
forward (Q K^T, dQ K^T, Q dK^T, P V, (P*dS) V, P dV), 2 flops per
multiply-add, i.e. 12 * B * H * Nq * Nk * D, halved for a causal mask.  This is
the count the pages' own throughput column implies (TFLOP/s x time is about
52.5 GFLOP at N = 2048 for B*H*D = 1024 in all three dtype tables of the
"JVP Flash Attention" benchmark summary), and masks do not change it.

Bytes: each input read once and each output written once, plus the mask once;
re-reads of K/V by different query tiles are served by L2 and not counted.
"""

from __future__ import annotations


def flops_fwd_dual(B: int, H: int, Nq: int, Nk: int, D: int, causal: bool = False) -> float:
    f = 12.0 * B * H * Nq * Nk * D
    return f / 2 if causal else f


def flops_fwd(B: int, H: int, Nq: int, Nk: int, D: int, causal: bool = False) -> float:
    f = 4.0 * B * H * Nq * Nk * D
    return f / 2 if causal else f


def bytes_fwd_dual(B: int, H: int, Nq: int, Nk: int, D: int, elem: int, mask: str = "none",
                   mask_batch: int = 1, stats: bool = True) -> float:
    """Algorithmic HBM bytes of one fwd_dual call ([mask_batch,1,Nq,Nk] mask)."""
    io = (2 * Nq + 4 * Nk) * B * H * D * elem + 2 * B * H * Nq * D * elem
    if stats:
        io += 8 * B * H * Nq  # lse and mu, float32
    if mask == "bool":
        io += mask_batch * Nq * Nk
    elif mask == "additive":
        io += 4 * mask_batch * Nq * Nk
    return float(io)
