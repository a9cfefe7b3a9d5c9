"""torch.func / autograd integration (forward_mode_flash_gb300.autograd) on the GPU.

* torch.func.jvp of jvp_attention gives the fused kernel's (O, tO), which the
  oracle checks;
* reverse mode through JVPAttn.fwd_dual (the HVP / training-through-JVP case)
  gives the oracle's reverse mode of the dual computation;
* the plain backward of jvp_attention gives the oracle's gradients of <gO, O>.
"""

import numpy as np
import pytest
import torch

import oracle
from forward_mode_flash_gb300 import build, synth
from forward_mode_flash_gb300.autograd import JVPAttn, jvp_attention

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def np64(t):
    return t.detach().to("cpu", torch.float64).numpy()


@pytest.mark.parametrize("dtype,D,mask", [("bf16", 128, "causal"), ("f16", 64, "none"),
                                          ("f32", 32, "none")])
def test_torch_func_jvp_matches_oracle(dtype, D, mask):
    w = synth.small(dtype, 2, 2, 150, D, mask, seed=41)
    inp = synth.make_inputs(w)
    g = [x.cuda() for x in (inp.q, inp.k, inp.v, inp.dq, inp.dk, inp.dv)]
    causal = mask == "causal"
    o, t_o = torch.func.jvp(lambda q, k, v: jvp_attention(q, k, v, is_causal=causal),
                            tuple(g[:3]), tuple(g[3:]))
    ro, rt, _, _ = oracle.fwd_dual(*(np64(x) for x in g), mask)
    tol = 1e-4 if dtype == "f32" else 2e-2
    assert np.abs(np64(o) - ro).max() <= tol and np.abs(np64(t_o) - rt).max() <= tol


def test_reverse_through_fwd_dual_matches_oracle():
    w = synth.small("bf16", 1, 2, 140, 64, "causal", seed=42)
    inp = synth.make_inputs(w, with_cotangents=True)
    xs = [x.cuda().requires_grad_(True) for x in (inp.q, inp.k, inp.v, inp.dq, inp.dk, inp.dv)]
    o, t_o = JVPAttn.fwd_dual(*xs, is_causal=True)
    loss = (o.float() * inp.g_o.cuda().float()).sum() + (t_o.float() * inp.g_to.cuda().float()).sum()
    loss.backward()
    ref = oracle.bwd_dual(*(np64(x) for x in xs), np64(inp.g_o), np64(inp.g_to), "causal")
    for x, r in zip(xs, ref):
        assert np.abs(np64(x.grad) - r).max() <= 2e-2 * max(1.0, np.abs(r).max())


def test_plain_backward_matches_oracle():
    w = synth.small("f32", 1, 2, 90, 48, "none", seed=43)
    inp = synth.make_inputs(w, with_cotangents=True)
    q, k, v = (x.cuda().requires_grad_(True) for x in (inp.q, inp.k, inp.v))
    o = jvp_attention(q, k, v)
    (o * inp.g_o.cuda()).sum().backward()
    z = np.zeros_like(np64(inp.q))
    ref = oracle.bwd_dual(np64(q), np64(k), np64(v), z, z, z, np64(inp.g_o), z, "none")
    for x, r in zip((q, k, v), ref[:3]):
        assert np.abs(np64(x.grad) - r).max() <= 1e-4 * max(1.0, np.abs(r).max())
