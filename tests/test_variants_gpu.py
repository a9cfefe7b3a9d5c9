"""GPU parity of the variants: grouped-query attention (Hkv < H) and a causal
rule on top of a bool / additive mask, forward and backward.

The oracle is the plain definition in both cases:
* grouped-query attention is ordinary attention with each key/value head
  repeated for the H / Hkv query heads that read it, and the gradient of a
  repeated tensor is the sum over its copies;
* a causal rule on top of a mask is the mask with every entry j > i
  excluded (False for a bool mask, -inf for an additive one).
Tolerances as in the other parity tests (1e-4 float32, 2e-2 fp16/bf16 on
O and tO; the backward's relative form).
"""

import numpy as np
import pytest
import torch

import oracle
from forward_mode_flash_gb300 import api as A
from forward_mode_flash_gb300 import build, synth

pytestmark = pytest.mark.gpu
TOL = {"f32": 1e-4, "f16": 2e-2, "bf16": 2e-2}


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def np64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def make(dtype, B, H, Hkv, Nq, Nk, D, mask, seed):
    """Seeded inputs; key-side tensors keep the first Hkv heads of the draw."""
    w = synth.small(dtype, B, H, Nq, D, mask, seed=seed, Nk=Nk)
    inp = synth.make_inputs(w, with_cotangents=True)
    for name in ("k", "v", "dk", "dv"):
        setattr(inp, name, getattr(inp, name)[:, :Hkv].contiguous())
    return w, inp


def oracle_mask(w, inp, causal):
    """(kind, array) for the oracle: the combined rule as a plain mask."""
    if w.mask == "none":
        return ("causal" if causal else "none"), None
    m = inp.mask.numpy() if w.mask == "bool" else inp.mask.double().numpy()
    if causal:
        Nq, Nk = m.shape[-2:]
        above = np.triu(np.ones((Nq, Nk), dtype=bool), k=1)  # j > i
        m = m.copy()
        if w.mask == "bool":
            m[..., above] = False
        else:
            m[..., above] = -np.inf
    return w.mask, m


def expand(x, group):
    return np.repeat(x, group, axis=1)


def run_fwd(w, inp, causal):
    dev = "cuda"
    g = [x.to(dev) for x in (inp.q, inp.k, inp.v, inp.dq, inp.dk, inp.dv)]
    m = inp.mask.to(dev) if inp.mask is not None else None
    o, t_o, lse, mu = A.fwd_dual(*g, attn_mask=m, is_causal=causal, return_stats=True)
    path = A.last_path()
    torch.cuda.synchronize()
    assert A.device_status() == 0
    return (o, t_o, lse, mu), path


def check_fwd(w, inp, causal):
    (o, t_o, lse, mu), path = run_fwd(w, inp, causal)
    assert path in ((2,) if w.dtype == "f32" or w.D % 8 or w.D > 128 else A.TENSOR_CORE_PATHS)
    group = inp.q.shape[1] // inp.k.shape[1]
    kind, m = oracle_mask(w, inp, causal)
    ro, rt, rl, rm = oracle.fwd_dual(np64(inp.q), expand(np64(inp.k), group),
                                     expand(np64(inp.v), group), np64(inp.dq),
                                     expand(np64(inp.dk), group), expand(np64(inp.dv), group),
                                     kind, m)
    tol = TOL[w.dtype]
    assert np.abs(np64(o) - ro).max() <= tol, w.name
    assert np.abs(np64(t_o) - rt).max() <= tol, w.name
    fin = np.isfinite(rl)
    assert np.array_equal(np.isfinite(np64(lse)), fin)
    if fin.any():
        assert np.abs(np64(lse)[fin] - rl[fin]).max() <= (1e-5 if w.dtype == "f32" else 1e-3)
    assert np.abs(np64(mu) - rm).max() <= 20 * tol


def check_bwd(w, inp, causal):
    dev = "cuda"
    (o, t_o, lse, mu), _ = run_fwd(w, inp, causal)
    g = [x.to(dev) for x in (inp.q, inp.k, inp.v, inp.dq, inp.dk, inp.dv)]
    m = inp.mask.to(dev) if inp.mask is not None else None
    grads = A.bwd_dual(*g, o, t_o, lse, mu, inp.g_o.to(dev), inp.g_to.to(dev), attn_mask=m,
                       is_causal=causal)
    path = A.last_path()
    torch.cuda.synchronize()
    assert A.device_status() == 0
    assert path == (2 if w.dtype == "f32" or w.D % 8 or w.D > 128 else 1)
    H, Hkv = inp.q.shape[1], inp.k.shape[1]
    group = H // Hkv
    kind, mm = oracle_mask(w, inp, causal)
    ref = oracle.bwd_dual(np64(inp.q), expand(np64(inp.k), group), expand(np64(inp.v), group),
                          np64(inp.dq), expand(np64(inp.dk), group), expand(np64(inp.dv), group),
                          np64(inp.g_o), np64(inp.g_to), kind, mm)
    tol = TOL[w.dtype]
    for idx, (name, got, r) in enumerate(zip(["g_q", "g_k", "g_v", "g_dq", "g_dk", "g_dv"],
                                            grads, ref)):
        if name in ("g_k", "g_v", "g_dk", "g_dv"):
            B, _, N, D = r.shape
            r = r.reshape(B, Hkv, group, N, D).sum(axis=2)
        e = np.abs(np64(got) - r).max()
        assert e <= tol * max(1.0, np.abs(r).max()), (w.name, name, e)


CASES = [("bf16", 64), ("f16", 128), ("f32", 40), ("bf16", 32)]


@pytest.mark.parametrize("dtype,D", CASES)
@pytest.mark.parametrize("H,Hkv", [(8, 2), (4, 1)])
@pytest.mark.parametrize("mask", ["none", "causal", "bool"])
@pytest.mark.parametrize("Nq,Nk", [(130, 130), (100, 257)])
def test_grouped_query_attention_forward(dtype, D, H, Hkv, mask, Nq, Nk):
    causal = mask == "causal"
    w, inp = make(dtype, 1, H, Hkv, Nq, Nk, D, "none" if causal else mask, seed=H + Nq + D)
    check_fwd(w, inp, causal)


@pytest.mark.parametrize("dtype,D", CASES)
@pytest.mark.parametrize("H,Hkv", [(8, 2), (4, 1)])
@pytest.mark.parametrize("mask", ["none", "causal", "bool"])
@pytest.mark.parametrize("Nq,Nk", [(130, 130), (100, 257)])
def test_grouped_query_attention_backward(dtype, D, H, Hkv, mask, Nq, Nk):
    causal = mask == "causal"
    w, inp = make(dtype, 1, H, Hkv, Nq, Nk, D, "none" if causal else mask, seed=H + Nq + D + 1)
    check_bwd(w, inp, causal)


@pytest.mark.parametrize("dtype,D", CASES)
@pytest.mark.parametrize("mask", ["bool", "additive"])
@pytest.mark.parametrize("Nq,Nk", [(77, 77), (200, 200), (130, 300), (300, 130)])
def test_causal_on_top_of_a_mask_forward(dtype, D, mask, Nq, Nk):
    w, inp = make(dtype, 2, 2, 2, Nq, Nk, D, mask, seed=Nq + 7 * Nk)
    check_fwd(w, inp, True)


@pytest.mark.parametrize("dtype,D", CASES)
@pytest.mark.parametrize("mask", ["bool", "additive"])
@pytest.mark.parametrize("Nq,Nk", [(77, 77), (200, 200), (130, 300), (300, 130)])
def test_causal_on_top_of_a_mask_backward(dtype, D, mask, Nq, Nk):
    w, inp = make(dtype, 2, 2, 2, Nq, Nk, D, mask, seed=Nq + 7 * Nk + 1)
    check_bwd(w, inp, True)


def test_grouped_heads_with_causal_and_bool_mask_together():
    w, inp = make("bf16", 2, 6, 3, 257, 257, 128, "bool", seed=5)
    check_fwd(w, inp, True)
    check_bwd(w, inp, True)


def test_causal_and_mask_exclude_exactly_the_union():
    # Perturbing K/V/dK/dV of keys that are excluded by the mask or lie above
    # the diagonal leaves every output bit-identical.
    w, inp = make("bf16", 1, 2, 2, 160, 160, 64, "bool", seed=9)
    inp.mask[..., 100:, 40] = False
    base, _ = run_fwd(w, inp, True)
    for t in (inp.k, inp.v, inp.dk, inp.dv):
        t[:, :, 40] += 3.0  # key 40: excluded from rows >= 100 by the mask
    pert, _ = run_fwd(w, inp, True)
    for a, b in zip(base, pert):
        assert torch.equal(a[:, :, 100:], b[:, :, 100:])
    base, _ = run_fwd(w, inp, True)
    for t in (inp.k, inp.v, inp.dk, inp.dv):
        t[:, :, 150:] -= 2.0  # keys 150..159: above the diagonal of rows < 150
    pert, _ = run_fwd(w, inp, True)
    for a, b in zip(base, pert):
        assert torch.equal(a[:, :, :150], b[:, :, :150])
