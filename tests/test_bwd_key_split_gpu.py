"""The backward's splits: when (batch, key/value head, key tile) CTAs would
fill less than half of the SMs and each would walk 64 or more query tiles
(grouped-query heads with few key/value heads), each key tile's query tiles
are shared by several CTAs whose fp32 partial sums of gK, g_dK, gV, g_dV a
combine kernel adds; likewise each query tile's key tiles when few
query-major CTAs would walk 64 or more key tiles (few queries, many keys),
with partial sums of gQ and g_dQ.

Checked against the float64 oracle's reverse mode (the tolerance reading of
the other backward tests: max-abs <= 2e-2 * max(1, max |reference|) per
gradient), against the unsplit kernels (run with a workspace of the base size,
8 * B * H * Nq bytes, which leaves no room for the partial sums: the two
differ only by the order of fp32 additions), and for bit-identical repeats.
"""

import numpy as np
import pytest
import torch

import oracle
from forward_mode_flash_gb300 import api as A
from forward_mode_flash_gb300 import build

pytestmark = pytest.mark.gpu
TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def np64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def make(dtype, B, H, Hkv, Nq, Nk, D, seed):
    g = torch.Generator().manual_seed(seed)
    dt = {"bf16": torch.bfloat16, "f16": torch.float16}[dtype]
    mk = lambda h, n: torch.randn(B, h, n, D, generator=g).to(dt).cuda()
    q, dq, go, gto = mk(H, Nq), mk(H, Nq), mk(H, Nq), mk(H, Nq)
    k, v, dk, dv = mk(Hkv, Nk), mk(Hkv, Nk), mk(Hkv, Nk), mk(Hkv, Nk)
    return q, k, v, dq, dk, dv, go, gto


def reference(args, causal, group, primal):
    q, k, v, dq, dk, dv, go, gto = (np64(x) for x in args)
    rep = lambda x: np.repeat(x, group, axis=1)
    if primal:
        dq, dk, dv, gto = np.zeros_like(dq), np.zeros_like(dk), np.zeros_like(dv), np.zeros_like(gto)
    r = oracle.bwd_dual(q, rep(k), rep(v), dq, rep(dk), rep(dv), go, gto,
                        "causal" if causal else "none", None)
    out = []
    for name, x in zip(("g_q", "g_k", "g_v", "g_dq", "g_dk", "g_dv"), r):
        if name in ("g_k", "g_v", "g_dk", "g_dv") and group > 1:
            B, _, N, D = x.shape
            x = x.reshape(B, -1, group, N, D).sum(axis=2)
        out.append(x)
    return out[:3] if primal else out


def run(args, causal, primal, ws):
    q, k, v, dq, dk, dv, go, gto = args
    if primal:
        o, lse = A.attention(q, k, v, is_causal=causal, return_lse=True)
        return A.bwd(q, k, v, o, lse, go, is_causal=causal, workspace=ws)
    o, t_o, lse, mu = A.fwd_dual(q, k, v, dq, dk, dv, is_causal=causal, return_stats=True,
                                 split_kv=False)
    return A.bwd_dual(q, k, v, dq, dk, dv, o, t_o, lse, mu, go, gto, is_causal=causal,
                      workspace=ws)


@pytest.mark.parametrize("primal", [False, True])
@pytest.mark.parametrize("dtype,D", [("bf16", 64), ("f16", 128), ("bf16", 32)])
@pytest.mark.parametrize("B,H,Hkv,Nq,Nk,causal", [(1, 8, 1, 512, 512, False),
                                                 (2, 16, 1, 384, 256, True),
                                                 (1, 4, 1, 1000, 300, False),
                                                 (1, 16, 1, 256, 700, True)])
def test_split_key_side_matches_oracle_and_unsplit(primal, dtype, D, B, H, Hkv, Nq, Nk, causal):
    args = make(dtype, B, H, Hkv, Nq, Nk, D, seed=Nq + Nk + D)
    need = A.bwd_dual_workspace_size(B, H, Nq, Nk, D, hkv=Hkv)
    base = 8 * B * H * Nq
    assert need > base  # these shapes split on a GB300 (152 SMs)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    got = run(args, causal, primal, ws)
    torch.cuda.synchronize()
    assert A.device_status() == 0 and A.last_path() == 1
    unsplit = run(args, causal, primal, torch.empty(base, dtype=torch.uint8, device="cuda"))
    torch.cuda.synchronize()
    ref = reference(args, causal, H // Hkv, primal)
    for x, u, r in zip(got, unsplit, ref):
        scale = max(1.0, float(np.abs(r).max()))
        assert np.abs(np64(x) - r).max() <= TOL * scale
        assert np.abs(np64(x) - np64(u)).max() <= TOL * scale
    again = run(args, causal, primal, ws)
    for x, y in zip(got, again):
        assert torch.equal(x, y)


@pytest.mark.parametrize("primal", [False, True])
@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("f16", 64), ("bf16", 16)])
@pytest.mark.parametrize("B,H,Nq,Nk,causal", [(1, 4, 100, 4096, False),
                                             (2, 2, 300, 5000, False),
                                             (1, 2, 256, 4100, True)])
def test_split_query_side_matches_oracle_and_unsplit(primal, dtype, D, B, H, Nq, Nk, causal):
    # Few queries, many keys: the query-major CTAs (B * H * ceil(Nq / 128))
    # each walk 64+ key tiles, so each query tile's key tiles are shared by
    # several CTAs and a combine kernel adds their partial g_dQ, gQ.
    args = make(dtype, B, H, H, Nq, Nk, D, seed=Nq + 3 * Nk + D)
    need = A.bwd_dual_workspace_size(B, H, Nq, Nk, D)
    base = 8 * B * H * Nq
    assert need > base  # these shapes split on a GB300 (152 SMs)
    got = run(args, causal, primal, torch.empty(need, dtype=torch.uint8, device="cuda"))
    torch.cuda.synchronize()
    assert A.device_status() == 0 and A.last_path() == 1
    unsplit = run(args, causal, primal, torch.empty(base, dtype=torch.uint8, device="cuda"))
    torch.cuda.synchronize()
    ref = reference(args, causal, 1, primal)
    for x, u, r in zip(got, unsplit, ref):
        scale = max(1.0, float(np.abs(r).max()))
        assert np.abs(np64(x) - r).max() <= TOL * scale
        assert np.abs(np64(x) - np64(u)).max() <= TOL * scale


@pytest.mark.parametrize("primal", [False, True])
@pytest.mark.parametrize("kind", ["bool", "additive"])
@pytest.mark.parametrize("B,H,Hkv,Nq,Nk", [(1, 8, 1, 512, 512), (1, 4, 4, 100, 4096)])
def test_splits_with_masks(primal, kind, B, H, Hkv, Nq, Nk):
    # Both splits under a [B, 1, Nq, Nk] mask (the first shape splits the key
    # side, the second the query side), with the causal rule on top of it.
    D = 64
    args = make("bf16", B, H, Hkv, Nq, Nk, D, seed=Nq + Nk + len(kind))
    g = torch.Generator().manual_seed(Nk)
    if kind == "bool":
        m = torch.rand(B, 1, Nq, Nk, generator=g) < 0.8
        dense = np.broadcast_to(m.numpy(), (B, H, Nq, Nk)).copy()
    else:
        m = torch.randn(B, 1, Nq, Nk, generator=g)
        dense = np.broadcast_to(m.double().numpy(), (B, H, Nq, Nk)).copy()
    above = np.triu(np.ones((Nq, Nk), dtype=bool), k=1)
    dense[..., above] = False if kind == "bool" else -np.inf
    mc = m.cuda()
    q, k, v, dq, dk, dv, go, gto = args
    need = A.bwd_dual_workspace_size(B, H, Nq, Nk, D, hkv=Hkv)
    assert need > 8 * B * H * Nq
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    if primal:
        o, lse = A.attention(q, k, v, attn_mask=mc, is_causal=True, return_lse=True)
        got = A.bwd(q, k, v, o, lse, go, attn_mask=mc, is_causal=True, workspace=ws)
    else:
        o, t_o, lse, mu = A.fwd_dual(q, k, v, dq, dk, dv, attn_mask=mc, is_causal=True,
                                     return_stats=True, split_kv=False)
        got = A.bwd_dual(q, k, v, dq, dk, dv, o, t_o, lse, mu, go, gto, attn_mask=mc,
                         is_causal=True, workspace=ws)
    torch.cuda.synchronize()
    assert A.device_status() == 0 and A.last_path() == 1
    xs = [np64(x) for x in args]
    rep = lambda x: np.repeat(x, H // Hkv, axis=1)
    if primal:
        for i in (3, 4, 5, 7):
            xs[i] = np.zeros_like(xs[i])
    r = oracle.bwd_dual(xs[0], rep(xs[1]), rep(xs[2]), xs[3], rep(xs[4]), rep(xs[5]), xs[6], xs[7],
                        kind, dense)
    for idx, (x, ref) in enumerate(zip(got, r)):
        if idx in (1, 2, 4, 5) and H // Hkv > 1:
            ref = ref.reshape(B, Hkv, H // Hkv, Nk, D).sum(axis=2)
        scale = max(1.0, float(np.abs(ref).max()))
        assert np.abs(np64(x) - ref).max() <= TOL * scale, idx
