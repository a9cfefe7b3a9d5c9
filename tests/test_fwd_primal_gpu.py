"""The forward without tangents (`jvp_attn_fwd`: O and the log-sum-exp of
SDPA's forward) against the float64 oracle's primal outputs.

Its tensor-core kernel hands whole key tiles to the two softmax warpgroups in
turn (warpgroup w takes the tiles t with t % 2 == w into its own accumulator;
with an additive mask each takes half of every tile), so the cases include a
single key tile (warpgroup 1 then never runs and its accumulator is never
written), odd and even tile counts, ragged last tiles, causal rows whose last
tile belongs to either warpgroup, Nq != Nk, grouped-query heads, every mask
kind, fully masked rows and bit-identical repeats.  Tolerances as for the dual
forward: max-abs 2e-2 on O (1e-4 for float32), 1e-3 on the log-sum-exp
(1e-5 for float32).
"""

import numpy as np
import pytest
import torch

import oracle
from forward_mode_flash_gb300 import api as A
from forward_mode_flash_gb300 import build, synth

pytestmark = pytest.mark.gpu
TOL = {"f32": 1e-4, "f16": 2e-2, "bf16": 2e-2}
LSE_TOL = {"f32": 1e-5, "f16": 1e-3, "bf16": 1e-3}


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def np64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def check(dt, B, H, N, D, mask, seed, Nk=None, hkv=None, expect_tc=True):
    w = synth.small(dt, B, H, N, D, mask, seed=seed, Nk=Nk)
    inp = synth.make_inputs(w)
    q, k, v = inp.q, inp.k, inp.v
    if hkv is not None:  # grouped-query heads: keep the first of every group's key/value heads
        k, v = k[:, ::H // hkv].contiguous(), v[:, ::H // hkv].contiguous()
    dev = "cuda"
    m = inp.mask.to(dev) if inp.mask is not None else None
    causal = mask == "causal"
    o, lse = A.attention(q.to(dev), k.to(dev), v.to(dev), attn_mask=m, is_causal=causal,
                         return_lse=True)
    torch.cuda.synchronize()
    assert A.device_status() == 0
    if expect_tc:
        assert A.last_path() == 1
    o2, lse2 = A.attention(q.to(dev), k.to(dev), v.to(dev), attn_mask=m, is_causal=causal,
                           return_lse=True)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    kr, vr = np64(k), np64(v)
    if hkv is not None:
        kr, vr = np.repeat(kr, H // hkv, axis=1), np.repeat(vr, H // hkv, axis=1)
    kind, mm = mask, None
    if mask == "bool":
        mm = inp.mask.numpy()
    elif mask == "additive":
        mm = inp.mask.double().numpy()
    ro, _, rl, _ = oracle.fwd_dual(np64(q), kr, vr, mask_kind=kind, mask=mm)
    assert np.abs(np64(o) - ro).max() <= TOL[dt]
    fin = np.isfinite(rl)
    got = np64(lse)
    assert np.array_equal(np.isfinite(got), fin)
    assert np.abs(got[fin] - rl[fin]).max(initial=0.0) <= LSE_TOL[dt]
    return o, lse


@pytest.mark.parametrize("mask", ["none", "causal", "bool", "additive"])
@pytest.mark.parametrize("dt,D", [("bf16", 128), ("f16", 64), ("bf16", 64), ("f16", 128)])
@pytest.mark.parametrize("N", [40, 64, 100, 128, 190, 257, 520])
def test_primal_forward_tile_counts(mask, dt, D, N):
    # 1 to 9 key tiles of 64: one warpgroup only, even and odd counts, ragged tails.
    check(dt, 2, 2, N, D, mask, seed=N + D)


@pytest.mark.parametrize("mask", ["none", "causal", "bool", "additive"])
@pytest.mark.parametrize("dt,D", [("bf16", 128), ("f16", 64)])
@pytest.mark.parametrize("Nq,Nk", [(1, 9), (13, 5), (5, 130), (200, 64), (129, 700), (700, 129)])
def test_primal_forward_query_and_key_lengths_differ(mask, dt, D, Nq, Nk):
    check(dt, 1, 3, Nq, D, mask, seed=Nq + 7 * Nk, Nk=Nk)


@pytest.mark.parametrize("mask", ["none", "causal", "bool"])
@pytest.mark.parametrize("dt,D", [("bf16", 128), ("f16", 64), ("bf16", 32), ("f16", 96)])
def test_primal_forward_grouped_query_heads_and_other_head_dims(mask, dt, D):
    check(dt, 2, 8, 300, D, mask, seed=D, hkv=2)


@pytest.mark.parametrize("mask", ["none", "causal", "bool", "additive"])
def test_primal_forward_larger_case(mask):
    check("bf16", 2, 4, 1000, 128, mask, seed=5)


def test_primal_forward_fully_masked_rows():
    # Rows whose keys are all masked give O = 0 and lse = -inf (the same
    # convention as the dual forward), whichever warpgroup's tiles they span.
    dev = "cuda"
    g = torch.Generator().manual_seed(3)
    B, H, N, D = 1, 2, 200, 128
    q, k, v = (torch.randn(B, H, N, D, generator=g).to(torch.bfloat16) for _ in range(3))
    keep = torch.rand(B, 1, N, N, generator=g) < 0.5
    keep[:, :, 7] = False          # a row with nothing kept
    keep[:, :, 9, :] = False
    keep[:, :, 9, 130] = True      # a row whose only key is in the third tile
    o, lse = A.attention(q.to(dev), k.to(dev), v.to(dev), attn_mask=keep.to(dev),
                         return_lse=True)
    torch.cuda.synchronize()
    assert A.last_path() == 1
    assert torch.all(o[:, :, 7] == 0) and torch.all(torch.isneginf(lse[:, :, 7]))
    assert torch.allclose(o[:, :, 9].float().cpu(), v[:, :, 130].float(), atol=1e-2)
    ro, _, rl, _ = oracle.fwd_dual(np64(q), np64(k), np64(v), mask_kind="bool",
                                   mask=keep.numpy())
    assert np.abs(np64(o) - ro).max() <= 2e-2


def test_primal_forward_matches_the_dual_forwards_output():
    # The same O from both entry points, up to the order of the fp32 sums.
    w = synth.small("bf16", 2, 4, 600, 128, "causal", seed=11)
    inp = synth.make_inputs(w)
    dev = "cuda"
    g = [x.to(dev) for x in (inp.q, inp.k, inp.v, inp.dq, inp.dk, inp.dv)]
    o_p, lse_p = A.attention(*g[:3], is_causal=True, return_lse=True)
    o_d, _, lse_d, _ = A.fwd_dual(*g, is_causal=True, return_stats=True, split_kv=False)
    torch.cuda.synchronize()
    assert (o_p.float() - o_d.float()).abs().max().item() <= 1.6e-2
    assert (lse_p - lse_d).abs().max().item() <= 1e-4


@pytest.mark.parametrize("mask", ["none", "causal", "bool", "additive"])
@pytest.mark.parametrize("dt,D", [("bf16", 128), ("f16", 64)])
def test_primal_forward_rescales_when_the_maximum_jumps(mask, dt, D):
    # Logits that grow by ~10 (14 in log2 units, above the 2^8 rescale
    # threshold) from one key tile to the next, so every tile moves the
    # running maximum and rescales its accumulator while the products of
    # earlier tiles may still be in flight.
    B, H, N = 2, 2, 1024
    w = synth.small(dt, B, H, N, D, mask, seed=17)
    inp = synth.make_inputs(w)
    g = torch.Generator().manual_seed(17)
    q = (torch.ones(B, H, N, D) + 0.1 * torch.randn(B, H, N, D, generator=g))
    tile = (torch.arange(N) // 64).to(torch.float32)
    k = (tile * 10.0 / D ** 0.5)[None, None, :, None] * torch.ones(B, H, N, D)
    k = k + 0.1 * torch.randn(B, H, N, D, generator=g)
    dt_t = {"bf16": torch.bfloat16, "f16": torch.float16}[dt]
    q, k = q.to(dt_t), k.to(dt_t)
    v = inp.v
    dev = "cuda"
    m = inp.mask.to(dev) if inp.mask is not None else None
    causal = mask == "causal"
    runs = [A.attention(q.to(dev), k.to(dev), v.to(dev), attn_mask=m, is_causal=causal,
                        return_lse=True) for _ in range(3)]
    torch.cuda.synchronize()
    assert A.device_status() == 0 and A.last_path() == 1
    for o, lse in runs[1:]:
        assert torch.equal(o, runs[0][0]) and torch.equal(lse, runs[0][1])
    kind, mm = mask, None
    if mask == "bool":
        mm = inp.mask.numpy()
    elif mask == "additive":
        mm = inp.mask.double().numpy()
    ro, _, rl, _ = oracle.fwd_dual(np64(q), np64(k), np64(v), mask_kind=kind, mask=mm)
    o, lse = runs[0]
    assert np.abs(np64(o) - ro).max() <= TOL[dt]
    fin = np.isfinite(rl)
    assert np.abs(np64(lse)[fin] - rl[fin]).max() <= max(1e-3, 1e-4 * float(np.abs(rl[fin]).max()))
