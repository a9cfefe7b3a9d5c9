"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module draws random numbers and casts them; it holds none of the
attention arithmetic, so both the GPU path and the float64 oracle can be fed
from it without sharing any of the method.

Recipe (the pages measure no public dataset; their sweep is over sequence
length, mask kind and causality only): every tensor is iid N(0, 1) drawn in
float32 from ``torch.Generator().manual_seed(seed)`` in the fixed order
Q, K, V, dQ, dK, dV, mask, gO, gtO, then rounded to the working dtype.  The
boolean keep-mask is Bernoulli(keep_p) with its diagonal forced to True; the
additive mask is iid N(0, 1) float32.  Masks are [B, 1, N, N] (broadcast over
heads), the shape the pages' benchmark uses for its mask rows.
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import torch

DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16,
          "float32": torch.float32, "float16": torch.float16, "bfloat16": torch.bfloat16}


@dataclass
class Workload:
    """One attention problem: shapes, dtype, mask kind and seed."""

    name: str
    dtype: str
    B: int
    H: int
    N: int
    D: int
    mask: str = "none"  # none | bool | additive | causal
    seed: int = 0
    keep_p: float = 0.9
    extra: dict = field(default_factory=dict)
    Nk: Optional[int] = None  # key/value length; None means equal to N

    @property
    def torch_dtype(self) -> torch.dtype:
        return DTYPES[self.dtype]

    @property
    def n_keys(self) -> int:
        return self.N if self.Nk is None else self.Nk


# The five workloads the method is specified on (sizes, dtypes and masks),
# expanded so that each mask variant is its own entry.
WORKLOADS = {
    "f32_b1h2n32d16": Workload("f32_b1h2n32d16", "f32", 1, 2, 32, 16),
    "f16_b2h8n512d64": Workload("f16_b2h8n512d64", "f16", 2, 8, 512, 64),
    "f16_b2h8n512d64_causal": Workload("f16_b2h8n512d64_causal", "f16", 2, 8, 512, 64, "causal"),
    "bf16_b2h8n1024d64_bool": Workload("bf16_b2h8n1024d64_bool", "bf16", 2, 8, 1024, 64, "bool"),
    "bf16_b2h8n1024d64_additive": Workload("bf16_b2h8n1024d64_additive", "bf16", 2, 8, 1024, 64,
                                           "additive"),
    "bf16_b4h16n2048d128": Workload("bf16_b4h16n2048d128", "bf16", 4, 16, 2048, 128),
    "bf16_b4h16n2048d128_causal": Workload("bf16_b4h16n2048d128_causal", "bf16", 4, 16, 2048, 128,
                                           "causal"),
    "f16_b2h8n2048d64_causal": Workload("f16_b2h8n2048d64_causal", "f16", 2, 8, 2048, 64, "causal"),
    # the headline shape under each mask type (a [B, 1, N, N] mask per batch)
    "bf16_b4h16n2048d128_bool": Workload("bf16_b4h16n2048d128_bool", "bf16", 4, 16, 2048, 128,
                                         "bool"),
    "bf16_b4h16n2048d128_additive": Workload("bf16_b4h16n2048d128_additive", "bf16", 4, 16, 2048,
                                             128, "additive"),
}


@dataclass
class Inputs:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    dq: torch.Tensor
    dk: torch.Tensor
    dv: torch.Tensor
    mask: Optional[torch.Tensor]  # bool [B,1,N,N] or float32 [B,1,N,N] or None
    g_o: Optional[torch.Tensor] = None
    g_to: Optional[torch.Tensor] = None


def make_inputs(w: Workload, with_cotangents: bool = False, device: str = "cpu") -> Inputs:
    """Draw the inputs of workload ``w`` on the CPU, then move them to ``device``."""
    g = torch.Generator().manual_seed(w.seed)
    shape = (w.B, w.H, w.N, w.D)
    kshape = (w.B, w.H, w.n_keys, w.D)
    # draw order: Q, K, V, dQ, dK, dV
    draws = [torch.randn(sh, generator=g, dtype=torch.float32)
             for sh in (shape, kshape, kshape, shape, kshape, kshape)]
    mask = None
    if w.mask == "bool":
        keep = torch.rand((w.B, 1, w.N, w.n_keys), generator=g, dtype=torch.float32) < w.keep_p
        idx = torch.arange(min(w.N, w.n_keys))
        keep[:, :, idx, idx] = True
        mask = keep
    elif w.mask == "additive":
        mask = torch.randn((w.B, 1, w.N, w.n_keys), generator=g, dtype=torch.float32)
    g_o = g_to = None
    if with_cotangents:
        g_o = torch.randn(shape, generator=g, dtype=torch.float32)
        g_to = torch.randn(shape, generator=g, dtype=torch.float32)
    dt = w.torch_dtype
    cast = [x.to(dt).to(device) for x in draws]
    if mask is not None:
        mask = mask.to(device)
    if g_o is not None:
        g_o = g_o.to(dt).to(device)
        g_to = g_to.to(dt).to(device)
    return Inputs(*cast, mask=mask, g_o=g_o, g_to=g_to)


def small(dtype: str, B: int, H: int, N: int, D: int, mask: str = "none", seed: int = 0,
          keep_p: float = 0.9, Nk: Optional[int] = None) -> Workload:
    """An ad-hoc workload for parity cases at sizes the oracle finishes quickly.

    ``Nk`` gives keys/values a length of their own (queries keep ``N``)."""
    kv = "" if Nk is None else f"k{Nk}"
    return Workload(f"{dtype}_b{B}h{H}n{N}{kv}d{D}_{mask}_s{seed}", dtype, B, H, N, D, mask, seed,
                    keep_p, Nk=Nk)
