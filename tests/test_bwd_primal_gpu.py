"""GPU parity of jvp_attn_bwd (the backward of attention without tangents)
against the float64 oracle's reverse mode with zero tangents and a zero
tangent cotangent, which the CPU pins show to be the primal backward
(`test_zero_tangent_reverse_mode_is_the_primal_backward`).

Same tolerance reading as the dual backward: max-abs error <= tol *
max(1, max |reference|) per gradient, tol = 1e-4 for float32 inputs and 2e-2
for fp16/bf16.  Inputs come from `attention(..., return_lse=True)` on the
same tensors, as `jvp_attention`'s autograd backward uses them.
"""

import numpy as np
import pytest
import torch

import oracle
from forward_mode_flash_gb300 import api as A
from forward_mode_flash_gb300 import build, synth
from forward_mode_flash_gb300.autograd import jvp_attention

pytestmark = pytest.mark.gpu
TOL = {"f32": 1e-4, "f16": 2e-2, "bf16": 2e-2}


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def np64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def tc_path(w):
    return w.dtype in ("f16", "bf16") and w.D % 8 == 0 and w.D <= 128


def oracle_mask(w, inp, causal_on_mask=False):
    if w.mask in ("none", "causal"):
        return w.mask, None
    m = inp.mask.numpy() if w.mask == "bool" else inp.mask.double().numpy()
    if causal_on_mask:
        Nq, Nk = m.shape[-2:]
        above = np.triu(np.ones((Nq, Nk), dtype=bool), k=1)  # keys j > i
        m = m.copy()
        m[..., above] = False if w.mask == "bool" else -np.inf
    return w.mask, m


def reference(w, inp, k, v, causal_on_mask=False, heads=None):
    """Oracle (g_q, g_k, g_v); k, v as float64 arrays with H heads."""
    sel = slice(None) if heads is None else heads
    q = np64(inp.q)[sel]
    z = np.zeros_like(q)
    zk = np.zeros_like(k[sel])
    kind, mm = oracle_mask(w, inp, causal_on_mask)
    if mm is not None:
        mm = mm[sel]
    g = oracle.bwd_dual(q, k[sel], v[sel], z, zk, zk, np64(inp.g_o)[sel], z, kind, mm)
    return g[:3]


def run_gpu(w, inp, causal_on_mask=False):
    dev = "cuda"
    q, k, v = (x.to(dev) for x in (inp.q, inp.k, inp.v))
    m = inp.mask.to(dev) if inp.mask is not None else None
    causal = w.mask == "causal" or causal_on_mask
    o, lse = A.attention(q, k, v, attn_mask=m, is_causal=causal, return_lse=True)
    grads = A.bwd(q, k, v, o, lse, inp.g_o.to(dev), attn_mask=m, is_causal=causal)
    path = A.last_path()
    torch.cuda.synchronize()
    assert A.device_status() == 0
    assert path == (1 if tc_path(w) else 2), path
    return grads


def check(w, grads, ref, sel=None, group=1):
    tol = TOL[w.dtype]
    for name, got, r in zip(("g_q", "g_k", "g_v"), grads, ref):
        g = np64(got)
        if sel is not None:
            g = g[sel]
        if name != "g_q" and group > 1:
            B, _, N, D = r.shape
            r = r.reshape(B, -1, group, N, D).sum(axis=2)
        e = np.abs(g - r).max() if r.size else 0.0
        assert e <= tol * max(1.0, np.abs(r).max() if r.size else 0.0), (w.name, name, e)


@pytest.mark.parametrize("mask", ["none", "causal", "bool", "additive"])
@pytest.mark.parametrize("dtype,D", [("f32", 16), ("bf16", 64), ("f16", 64), ("bf16", 128),
                                     ("f16", 128), ("f16", 32), ("bf16", 16), ("f16", 80),
                                     ("bf16", 20)])
@pytest.mark.parametrize("N", [1, 33, 130, 257])
def test_primal_bwd_small(mask, dtype, D, N):
    w = synth.small(dtype, 2, 2, N, D, mask, seed=5 * N + D)
    inp = synth.make_inputs(w, with_cotangents=True)
    grads = run_gpu(w, inp)
    check(w, grads, reference(w, inp, np64(inp.k), np64(inp.v)))


@pytest.mark.parametrize("dtype,D", [("bf16", 64), ("f16", 128), ("f32", 40)])
@pytest.mark.parametrize("Nq,Nk", [(100, 300), (300, 77), (1, 129), (130, 1)])
@pytest.mark.parametrize("mask", ["none", "causal", "bool", "additive"])
def test_primal_bwd_query_and_key_lengths_differ(dtype, D, Nq, Nk, mask):
    w = synth.small(dtype, 1, 2, Nq, D, mask, seed=Nq + 5 * Nk, Nk=Nk)
    inp = synth.make_inputs(w, with_cotangents=True)
    grads = run_gpu(w, inp)
    check(w, grads, reference(w, inp, np64(inp.k), np64(inp.v)))


@pytest.mark.parametrize("dtype,D", [("bf16", 64), ("f16", 128), ("bf16", 32)])
@pytest.mark.parametrize("H,Hkv", [(8, 2), (4, 1)])
@pytest.mark.parametrize("mask", ["none", "causal", "bool"])
def test_primal_bwd_grouped_query_heads(dtype, D, H, Hkv, mask):
    # Key/value head h / (H / Hkv) serves query head h; g_k and g_v sum the
    # group's contributions.
    w = synth.small(dtype, 1, H, 130, D, mask, seed=H + D + 17, Nk=257)
    inp = synth.make_inputs(w, with_cotangents=True)
    group = H // Hkv
    inp.k, inp.v = (x[:, :Hkv].contiguous() for x in (inp.k, inp.v))
    grads = run_gpu(w, inp)
    rep = lambda x: np.repeat(np64(x), group, axis=1)
    check(w, grads, reference(w, inp, rep(inp.k), rep(inp.v)), group=group)


@pytest.mark.parametrize("dtype,D", [("bf16", 64), ("f16", 128), ("f32", 40)])
@pytest.mark.parametrize("mask", ["bool", "additive"])
def test_primal_bwd_causal_on_top_of_a_mask(dtype, D, mask):
    w = synth.small(dtype, 2, 2, 200, D, mask, seed=D + 29, Nk=300)
    inp = synth.make_inputs(w, with_cotangents=True)
    grads = run_gpu(w, inp, causal_on_mask=True)
    check(w, grads, reference(w, inp, np64(inp.k), np64(inp.v), causal_on_mask=True))


def test_primal_bwd_fully_masked_rows_give_zero_gradients():
    w = synth.small("bf16", 1, 2, 130, 64, "bool", seed=3)
    inp = synth.make_inputs(w, with_cotangents=True)
    inp.mask[:, :, 5, :] = False
    inp.mask[:, :, 70, :] = False
    grads = run_gpu(w, inp)
    assert torch.all(grads[0][:, :, 5] == 0) and torch.all(grads[0][:, :, 70] == 0)
    check(w, grads, reference(w, inp, np64(inp.k), np64(inp.v)))


@pytest.mark.parametrize("name,heads", [("f16_b2h8n2048d64_causal", None),
                                        ("bf16_b4h16n2048d128", (slice(1, 2), slice(9, 11))),
                                        ("bf16_b4h16n2048d128_causal", (slice(2, 3), slice(0, 1)))])
def test_primal_bwd_specified_shapes(name, heads):
    # Full-size launches; the oracle checks every gradient entry (of the
    # selected (batch, head) problems for the B=4 H=16 shapes).
    w = synth.WORKLOADS[name]
    inp = synth.make_inputs(w, with_cotangents=True)
    grads = run_gpu(w, inp)
    check(w, grads, reference(w, inp, np64(inp.k), np64(inp.v), heads=heads),
          sel=None if heads is None else heads)


def test_primal_bwd_workspace_is_required():
    w = synth.small("bf16", 1, 1, 64, 64, "none")
    inp = synth.make_inputs(w, with_cotangents=True)
    q, k, v = (x.cuda() for x in (inp.q, inp.k, inp.v))
    o, lse = A.attention(q, k, v, return_lse=True)
    with pytest.raises(A._abi.JvpAttnError) as ei:
        A.bwd(q, k, v, o, lse, inp.g_o.cuda(), workspace=torch.empty(8, dtype=torch.uint8,
                                                                       device="cuda"))
    assert ei.value.status == A._abi.JVP_ERR_WORKSPACE


@pytest.mark.parametrize("dtype,D,mask", [("bf16", 128, "causal"), ("f16", 64, "bool")])
def test_jvp_attention_backward_takes_the_primal_kernels(dtype, D, mask, monkeypatch):
    # Ordinary back-propagation through jvp_attention calls bwd (never the
    # dual backward) and matches the oracle.
    w = synth.small(dtype, 2, 4, 257, D, mask, seed=D + 3)
    inp = synth.make_inputs(w, with_cotangents=True)
    calls = []
    monkeypatch.setattr(A, "bwd_dual", lambda *a, **k: calls.append("bwd_dual"))
    q, k, v = (x.cuda().requires_grad_(True) for x in (inp.q, inp.k, inp.v))
    m = inp.mask.cuda() if inp.mask is not None else None
    o = jvp_attention(q, k, v, attn_mask=m, is_causal=(mask == "causal"))
    o.backward(inp.g_o.cuda())
    assert calls == [] and A.last_path() == 1
    check(w, (q.grad, k.grad, v.grad), reference(w, inp, np64(inp.k), np64(inp.v)))


@pytest.mark.parametrize("dtype,D", [("bf16", 64), ("f32", 40)])
@pytest.mark.parametrize("Nq,Nk", [(0, 70), (70, 0)])
def test_backward_with_an_empty_side(dtype, D, Nq, Nk):
    # No query rows: the key-side gradients are zero; no keys: the query-side
    # gradients are zero (and lse = -inf rows give nothing).  Both backward
    # entry points, no error.
    dt = {"bf16": torch.bfloat16, "f32": torch.float32}[dtype]
    g = torch.Generator().manual_seed(Nq + Nk)
    mk = lambda n: torch.randn(1, 2, n, D, generator=g).to("cuda", dt)
    q, dq, go, gto = mk(Nq), mk(Nq), mk(Nq), mk(Nq)
    k, v, dk, dv = mk(Nk), mk(Nk), mk(Nk), mk(Nk)
    o, t_o, lse, mu = A.fwd_dual(q, k, v, dq, dk, dv, return_stats=True)
    for grads in (A.bwd_dual(q, k, v, dq, dk, dv, o, t_o, lse, mu, go, gto),
                  A.bwd(q, k, v, o, lse, go)):
        torch.cuda.synchronize()
        assert A.device_status() == 0
        for x in grads:
            assert x.numel() == 0 or torch.all(x == 0)
