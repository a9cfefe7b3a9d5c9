"""Mask layouts against the float64 oracle: broadcast batch / head dimensions,
rows that broadcast, keys that are not contiguous, odd key counts, ragged
query and key tiles.

At D = 128 an additive mask whose keys are contiguous, whose rows do not
broadcast and whose strides are 16-byte multiples reaches the tensor-core
kernel through a tensor map: [128 x 32] boxes copied into shared memory a
tile ahead.  Any other layout takes per-row loads.  Both must give the same
result as the oracle, to the forward tolerance (max-abs 2e-2 for fp16/bf16 on
O and tO); the layouts below cover both routes, and at D = 64 (the
register route for every layout) as a control.  Each case also runs the
forward without tangents on the same mask (two shared-memory slots at D = 128
where the layout allows the tensor map) against the oracle's O and lse.
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


def make_mask(kind, layout, B, H, Nq, Nk, g):
    """A mask tensor on the GPU in the given layout, and its dense float64 /
    bool copy [B, H, Nq, Nk] for the oracle."""
    def draw(shape):
        if kind == "additive":
            return torch.randn(*shape, generator=g)
        m = torch.rand(*shape, generator=g) < 0.85
        return m
    if layout == "full":
        base = draw((B, H, Nq, Nk))
        dev = base.cuda()
    elif layout == "batch":        # [B, 1, Nq, Nk]
        base = draw((B, 1, Nq, Nk))
        dev = base.cuda()
    elif layout == "head":         # [1, H, Nq, Nk]
        base = draw((1, H, Nq, Nk))
        dev = base.cuda()
    elif layout == "shared":       # [Nq, Nk]
        base = draw((Nq, Nk))
        dev = base.cuda()
    elif layout == "rows":         # [B, 1, 1, Nk]: one row of keys for every query
        base = draw((B, 1, 1, Nk))
        dev = base.cuda()
    elif layout == "keys_strided":  # every other column of a [Nq, 2 Nk] buffer
        wide = draw((B, 1, Nq, 2 * Nk))
        base = wide[..., ::2].contiguous()
        dev = wide.cuda()[..., ::2]
    elif layout == "transposed":    # [Nk, Nq] storage read as [Nq, Nk]
        base = draw((B, 1, Nk, Nq)).transpose(-1, -2).contiguous()
        dev = base.transpose(-1, -2).contiguous().cuda().transpose(-1, -2)
    else:
        raise ValueError(layout)
    dense = np.broadcast_to(base.numpy(), (B, H, Nq, Nk)).copy()
    if kind == "additive":
        dense = dense.astype(np.float64)
    return dev, dense


def check(dtype, D, kind, layout, B, H, Nq, Nk, causal=False, seed=0):
    g = torch.Generator().manual_seed(seed + Nq * 7 + Nk)
    dt = {"bf16": torch.bfloat16, "f16": torch.float16}[dtype]
    mk = lambda n: torch.randn(B, H, n, D, generator=g).to(dt)
    q, k, v, dq, dk, dv = mk(Nq), mk(Nk), mk(Nk), mk(Nq), mk(Nk), mk(Nk)
    m, dense = make_mask(kind, layout, B, H, Nq, Nk, g)
    if causal:
        above = np.triu(np.ones((Nq, Nk), dtype=bool), k=1)
        dense[..., above] = False if kind == "bool" else -np.inf
    o, t_o, lse, mu = A.fwd_dual(*(x.cuda() for x in (q, k, v, dq, dk, dv)), attn_mask=m,
                                 is_causal=causal, return_stats=True)
    torch.cuda.synchronize()
    assert A.device_status() == 0
    assert A.last_path() in A.TENSOR_CORE_PATHS
    ro, rt, rl, _ = oracle.fwd_dual(np64(q), np64(k), np64(v), np64(dq), np64(dk), np64(dv),
                                    kind, dense)
    eo = np.abs(np64(o) - ro).max()
    et = np.abs(np64(t_o) - rt).max()
    assert eo <= TOL and et <= TOL, (layout, eo, et)
    fin = np.isfinite(rl)
    assert np.array_equal(np.isfinite(np64(lse)), fin)
    if fin.any():
        assert np.abs(np64(lse)[fin] - rl[fin]).max() <= 1e-3
    # The forward without tangents on the same mask (its own mask routes: two
    # shared-memory slots at D = 128, registers a tile ahead at D = 64).
    po, plse = A.attention(*(x.cuda() for x in (q, k, v)), attn_mask=m, is_causal=causal,
                           return_lse=True)
    torch.cuda.synchronize()
    assert A.device_status() == 0 and A.last_path() == 1
    assert np.abs(np64(po) - ro).max() <= TOL, layout
    assert np.array_equal(np.isfinite(np64(plse)), fin)
    if fin.any():
        assert np.abs(np64(plse)[fin] - rl[fin]).max() <= 1e-3


@pytest.mark.parametrize("D", [128, 64])
@pytest.mark.parametrize("layout", ["full", "batch", "head", "shared", "rows", "keys_strided",
                                    "transposed"])
@pytest.mark.parametrize("Nq,Nk", [(256, 192), (200, 132), (130, 66)])
def test_additive_mask_layouts(D, layout, Nq, Nk):
    # Nk = 192 and 132: 16-byte rows (the shared-memory route at D = 128 for
    # contiguous keys); Nk = 66: rows of 264 bytes (per-row loads); Nq = 200
    # and 130: a ragged last query tile; Nk = 132 and 66: a ragged last key tile.
    check("bf16", D, "additive", layout, 2, 3, Nq, Nk)


@pytest.mark.parametrize("layout", ["full", "batch", "shared", "rows", "transposed"])
def test_bool_mask_layouts(layout):
    check("f16", 128, "bool", layout, 2, 2, 200, 132)
    check("bf16", 64, "bool", layout, 2, 2, 200, 132)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("Nq,Nk", [(1, 128), (1, 4), (64, 4096), (384, 384)])
def test_additive_mask_edge_lengths(dtype, Nq, Nk):
    # one query row (its row stride never used), four keys (a single 16-byte
    # row, most of the box out of range), a long key range, whole tiles
    check(dtype, 128, "additive", "batch", 1, 2, Nq, Nk)


@pytest.mark.parametrize("layout", ["batch", "full"])
def test_additive_mask_with_causal_rule(layout):
    check("bf16", 128, "additive", layout, 2, 2, 300, 300, causal=True)
    check("f16", 128, "additive", layout, 1, 2, 257, 320, causal=True)


def test_additive_mask_with_infinities_and_fully_masked_rows():
    # -inf entries exclude keys; a row of -inf is fully masked (O = tO = 0,
    # lse = -inf), at D = 128 through the shared-memory route.
    B, H, Nq, Nk, D = 1, 2, 130, 256, 128
    g = torch.Generator().manual_seed(11)
    mk = lambda n: torch.randn(B, H, n, D, generator=g).to(torch.bfloat16)
    q, k, v, dq, dk, dv = mk(Nq), mk(Nk), mk(Nk), mk(Nq), mk(Nk), mk(Nk)
    m = torch.randn(B, 1, Nq, Nk, generator=g)
    m[..., ::3] = -float("inf")
    m[:, :, 7, :] = -float("inf")
    m[:, :, 129, :] = -float("inf")
    o, t_o, lse, _ = A.fwd_dual(*(x.cuda() for x in (q, k, v, dq, dk, dv)), attn_mask=m.cuda(),
                                return_stats=True)
    torch.cuda.synchronize()
    assert A.device_status() == 0
    ro, rt, rl, _ = oracle.fwd_dual(np64(q), np64(k), np64(v), np64(dq), np64(dk), np64(dv),
                                    "additive", np.broadcast_to(m.double().numpy(),
                                                                (B, H, Nq, Nk)).copy())
    assert np.abs(np64(o) - ro).max() <= TOL and np.abs(np64(t_o) - rt).max() <= TOL
    for row in (7, 129):
        assert torch.all(o[:, :, row] == 0) and torch.all(t_o[:, :, row] == 0)
        assert torch.all(torch.isinf(lse[:, :, row])) and torch.all(lse[:, :, row] < 0)


@pytest.mark.parametrize("tangent", [False, True])
@pytest.mark.parametrize("Nq,Nk", [(200, 300), (512, 1028)])
def test_additive_mask_tile_repeats_are_bit_identical(tangent, Nq, Nk):
    # The shared-memory mask slot is refilled once every softmax warp has
    # consumed the previous tile's entries; a refill that overtook a read
    # would change some rows from one call to the next.  Forty calls, with and
    # without tangents, each equal bit for bit to the first and to the oracle.
    B, H, D = 2, 4, 128
    g = torch.Generator().manual_seed(Nk)
    mk = lambda n: torch.randn(B, H, n, D, generator=g).to(torch.bfloat16).cuda()
    q, k, v, dq, dk, dv = mk(Nq), mk(Nk), mk(Nk), mk(Nq), mk(Nk), mk(Nk)
    m = torch.randn(B, 1, Nq, Nk, generator=g).cuda()

    def call():
        if tangent:
            return A.fwd_dual(q, k, v, dq, dk, dv, attn_mask=m, split_kv=False)
        return (A.attention(q, k, v, attn_mask=m),)

    first = call()
    for _ in range(40):
        again = call()
        for a, b in zip(first, again):
            assert torch.equal(a, b)
    torch.cuda.synchronize()
    assert A.device_status() == 0
    sel = (slice(0, 1), slice(0, 2))
    ro, rt, _, _ = oracle.fwd_dual(*(np64(x[sel]) for x in (q, k, v, dq, dk, dv)), "additive",
                                   np.broadcast_to(np64(m[:1]), (1, 2, Nq, Nk)).copy())
    assert np.abs(np64(first[0][sel]) - ro).max() <= TOL
    if tangent:
        assert np.abs(np64(first[1][sel]) - rt).max() <= TOL


@pytest.mark.parametrize("name", ["bf16_b4h16n2048d128_additive", "bf16_b4h16n2048d128_bool"])
def test_headline_shape_with_masks_on_whole_heads(name):
    # The full B=4 H=16 N=2048 D=128 launch with a [B, 1, N, N] mask; every
    # element of three whole heads against the oracle.
    from forward_mode_flash_gb300 import synth
    w = synth.WORKLOADS[name]
    inp = synth.make_inputs(w)
    g = [x.cuda() for x in (inp.q, inp.k, inp.v, inp.dq, inp.dk, inp.dv)]
    o, t_o, lse, _ = A.fwd_dual(*g, attn_mask=inp.mask.cuda(), return_stats=True)
    torch.cuda.synchronize()
    assert A.device_status() == 0 and A.last_path() in A.TENSOR_CORE_PATHS
    for b, h in ((0, 0), (2, 9), (3, 15)):
        sel = (slice(b, b + 1), slice(h, h + 1))
        m = inp.mask[b:b + 1]
        m = m.numpy() if w.mask == "bool" else m.double().numpy()
        ro, rt, rl, _ = oracle.fwd_dual(*(np64(x[sel]) for x in (inp.q, inp.k, inp.v, inp.dq,
                                                                    inp.dk, inp.dv)),
                                        w.mask, m)
        assert np.abs(np64(o[sel]) - ro).max() <= TOL
        assert np.abs(np64(t_o[sel]) - rt).max() <= TOL
        assert np.abs(np64(lse[sel]) - rl).max() <= 1e-3
