"""GPU parity of jvp_attn_bwd_dual (reverse mode of the dual computation)
against the float64 oracle's reverse mode on the same inputs.

Tolerance: max-abs error <= tol * max(1, max |reference|) per gradient, with
tol = 1e-4 for float32 inputs and 2e-2 for fp16/bf16.  The method's stated
bound (2e-2 max-abs for 16-bit inputs) is for outputs of unit-variance scale;
a gradient has the scale of its cotangents times the attention weights and
dual logits, often well above 1, and both its 16-bit rounding (relative,
2^-9 for bf16) and the fp32 sums of 16-bit products that form it err in
proportion to that scale.  So the bound is applied relative to each
gradient's own scale, and is never looser than the absolute bound when that
scale is at most 1.  The GPU computes in fp32 from its own 16-bit O and tO
(which enter delta and nu) and rounds the gradients to 16 bits.

Every comparison appends its absolute error, the reference scale and their
ratio to $JVP_PARITY_LOG (JSON lines) when that variable is set.
"""

import json
import os

import numpy as np
import pytest
import torch

import oracle
from forward_mode_flash_gb300 import api as A
from forward_mode_flash_gb300 import build, synth

pytestmark = pytest.mark.gpu
TOL = {"f32": 1e-4, "f16": 2e-2, "bf16": 2e-2}
NAMES = ["g_q", "g_k", "g_v", "g_dq", "g_dk", "g_dv"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def np64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def run(w, heads=None):
    inp = synth.make_inputs(w, with_cotangents=True)
    dev = "cuda"
    g = [x.to(dev) for x in (inp.q, inp.k, inp.v, inp.dq, inp.dk, inp.dv)]
    m = inp.mask.to(dev) if inp.mask is not None else None
    causal = w.mask == "causal"
    o, t_o, lse, mu = A.fwd_dual(*g, attn_mask=m, is_causal=causal, return_stats=True)
    grads = A.bwd_dual(*g, o, t_o, lse, mu, inp.g_o.to(dev), inp.g_to.to(dev), attn_mask=m,
                       is_causal=causal)
    path = A.last_path()
    torch.cuda.synchronize()
    # fp16/bf16 with D in {16, 32, 64, 128} take the tensor-core kernels, the rest CUDA cores
    assert path == (1 if (w.dtype in ("f16", "bf16") and w.D % 8 == 0 and w.D <= 128) else 2), path
    assert A.device_status() == 0
    sel = slice(None) if heads is None else heads
    xs = [np64(x)[sel] for x in (inp.q, inp.k, inp.v, inp.dq, inp.dk, inp.dv, inp.g_o, inp.g_to)]
    mm = None
    if w.mask == "bool":
        mm = inp.mask.numpy()[sel]
    elif w.mask == "additive":
        mm = inp.mask.double().numpy()[sel]
    ref = oracle.bwd_dual(*xs, w.mask, mm)
    errs = {}
    for name, gg, r in zip(NAMES, grads, ref):
        gv = np64(gg)[sel]
        errs[name] = (np.abs(gv - r).max(), np.abs(r).max())
    return errs


def log_errors(name, errs):
    path = os.environ.get("JVP_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            for g, (e, scale) in errs.items():
                f.write(json.dumps({"case": name, "grad": g, "abs_err": float(e),
                                    "max_abs_ref": float(scale),
                                    "err_over_scale": float(e / max(1.0, scale))}) + "\n")


def check(w, errs, tag="[bwd]"):
    tol = TOL[w.dtype]
    log_errors(w.name + tag, errs)
    for name, (e, scale) in errs.items():
        assert e <= tol * max(1.0, scale), (w.name, name, e, scale)


@pytest.mark.parametrize("mask", ["none", "causal", "bool", "additive"])
@pytest.mark.parametrize("dtype,D", [("f32", 16), ("f32", 40), ("bf16", 64), ("f16", 64),
                                     ("bf16", 128), ("f16", 128), ("f16", 32), ("bf16", 16),
                                     ("f16", 80), ("bf16", 48), ("f16", 96), ("bf16", 20)])
@pytest.mark.parametrize("N", [1, 33, 130, 257])
def test_bwd_small(mask, dtype, D, N):
    w = synth.small(dtype, 2, 2, N, D, mask, seed=N + D)
    check(w, run(w))


def test_bwd_workspace_is_required_and_sized():
    assert A.bwd_dual_workspace_size(2, 8, 2048, 2048, 64) == 8 * 2 * 8 * 2048
    w = synth.small("bf16", 1, 1, 64, 64, "none")
    inp = synth.make_inputs(w, with_cotangents=True)
    g = [x.cuda() for x in (inp.q, inp.k, inp.v, inp.dq, inp.dk, inp.dv)]
    o, t_o, lse, mu = A.fwd_dual(*g, return_stats=True)
    small_ws = torch.empty(8, dtype=torch.uint8, device="cuda")
    with pytest.raises(A._abi.JvpAttnError) as ei:
        A.bwd_dual(*g, o, t_o, lse, mu, inp.g_o.cuda(), inp.g_to.cuda(), workspace=small_ws)
    assert ei.value.status == A._abi.JVP_ERR_WORKSPACE


def test_bwd_specified_workload_f16_b2h8n2048d64_causal_every_element():
    # Full-size launch; the oracle's reverse mode checks every entry of all six
    # gradients of all 16 (batch, head) problems.
    w = synth.WORKLOADS["f16_b2h8n2048d64_causal"]
    check(w, run(w), "[bwd, every element]")


@pytest.mark.parametrize("dtype,D", [("bf16", 64), ("f16", 128), ("f32", 40)])
@pytest.mark.parametrize("Nq,Nk", [(100, 300), (300, 77), (1, 129), (130, 1)])
@pytest.mark.parametrize("mask", ["none", "causal", "bool", "additive"])
def test_bwd_query_and_key_lengths_differ(dtype, D, Nq, Nk, mask):
    w = synth.small(dtype, 1, 2, Nq, D, mask, seed=Nq + 3 * Nk, Nk=Nk)
    check(w, run(w))


@pytest.mark.parametrize("name,heads", [("bf16_b4h16n2048d128", (slice(3, 4), slice(14, 16))),
                                        ("bf16_b4h16n2048d128_causal", (slice(0, 1), slice(5, 6)))])
def test_bwd_specified_workload_d128_whole_heads(name, heads):
    # Full-size launch (value and key parts of the key-major kernel); the oracle
    # checks every gradient entry of the selected heads.
    w = synth.WORKLOADS[name]
    check(w, run(w, heads=heads), "[bwd, whole heads]")


@pytest.mark.parametrize("dtype,D,mask,N", [("bf16", 128, "causal", 4096), ("f16", 64, "none", 8192)])
def test_bwd_long_sequences_one_head(dtype, D, mask, N):
    # One (b, h) problem with many key and query tiles per CTA.
    w = synth.small(dtype, 1, 1, N, D, mask, seed=N + D)
    check(w, run(w))


@pytest.mark.parametrize("dtype,D,mask", [("bf16", 64, "causal"), ("f16", 128, "additive")])
def test_bwd_negative_scale(dtype, D, mask):
    # The backward recomputes P from the saved lse with the signed scale (no
    # running maximum), so a negative scale needs nothing special; the forward
    # that feeds it takes the tensor-core path with negated score products.
    w = synth.small(dtype, 1, 2, 130, D, mask, seed=D + 7)
    inp = synth.make_inputs(w, with_cotangents=True)
    g = [x.cuda() for x in (inp.q, inp.k, inp.v, inp.dq, inp.dk, inp.dv)]
    m = inp.mask.cuda() if inp.mask is not None else None
    causal = mask == "causal"
    o, t_o, lse, mu = A.fwd_dual(*g, attn_mask=m, is_causal=causal, scale=-0.1,
                                 return_stats=True)
    assert A.last_path() == 1
    grads = A.bwd_dual(*g, o, t_o, lse, mu, inp.g_o.cuda(), inp.g_to.cuda(), attn_mask=m,
                       is_causal=causal, scale=-0.1)
    assert A.last_path() == 1
    primal = A.bwd(*g[:3], o, lse, inp.g_o.cuda(), attn_mask=m, is_causal=causal, scale=-0.1)
    torch.cuda.synchronize()
    assert A.device_status() == 0
    xs = [np64(x) for x in (inp.q, inp.k, inp.v, inp.dq, inp.dk, inp.dv, inp.g_o, inp.g_to)]
    mm = None if inp.mask is None else inp.mask.double().numpy()
    ref = oracle.bwd_dual(*xs, w.mask, mm, scale=-0.1)
    errs = {n: (np.abs(np64(gg) - r).max(), np.abs(r).max()) for n, gg, r in zip(NAMES, grads, ref)}
    check(w, errs, "[bwd, scale < 0]")
    # the primal backward against the zero-tangent reverse mode
    z = np.zeros_like(xs[0])
    zk = np.zeros_like(xs[1])
    ref_p = oracle.bwd_dual(xs[0], xs[1], xs[2], z, zk, zk, xs[6], z, w.mask, mm, scale=-0.1)
    errs_p = {n: (np.abs(np64(gg) - r).max(), np.abs(r).max())
              for n, gg, r in zip(NAMES[:3], primal, ref_p[:3])}
    check(w, errs_p, "[bwd primal, scale < 0]")
