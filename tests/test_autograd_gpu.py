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


# ----------------------------------------------------- the project page's call form
class _Count:
    """Counts the binding's kernel entry points called through the autograd glue."""

    def __init__(self, monkeypatch):
        from forward_mode_flash_gb300 import autograd as AG

        self.n = {"fwd_dual": 0, "attention": 0, "bwd_dual": 0}
        for name in self.n:
            real = getattr(AG.api, name)

            def wrapped(*a, _real=real, _name=name, **kw):
                self.n[_name] += 1
                return _real(*a, **kw)

            monkeypatch.setattr(AG.api, name, wrapped)


CALL_FORM_CASES = [("bf16", 64, "causal"), ("f16", 128, "bool"), ("f32", 40, "none"),
                   ("bf16", 128, "additive")]


def _inputs(dtype, D, mask, seed, requires_grad=False, Nk=None):
    w = synth.small(dtype, 2, 2, 150, D, mask, seed=seed, Nk=Nk)
    inp = synth.make_inputs(w, with_cotangents=True)
    xs = [x.cuda().requires_grad_(requires_grad) for x in
          (inp.q, inp.k, inp.v, inp.dq, inp.dk, inp.dv)]
    m = inp.mask.cuda() if inp.mask is not None else None
    mm = None
    if mask == "bool":
        mm = inp.mask.numpy()
    elif mask == "additive":
        mm = inp.mask.double().numpy()
    return w, inp, xs, m, mm


@pytest.mark.parametrize("dtype,D,mask", CALL_FORM_CASES)
def test_pages_call_form_is_one_fused_launch(dtype, D, mask, monkeypatch):
    # torch.func.jvp(lambda q, k, v: JVPAttn.fwd_dual(q, k, v), primals, tangents):
    # one fwd_dual launch, no separate primal pass, the oracle's (O, tO).
    w, inp, xs, m, mm = _inputs(dtype, D, mask, seed=60 + D)
    cnt = _Count(monkeypatch)
    causal = mask == "causal"
    o, t_o = torch.func.jvp(
        lambda q, k, v: JVPAttn.fwd_dual(q, k, v, attn_mask=m, is_causal=causal),
        tuple(xs[:3]), tuple(xs[3:]))
    torch.cuda.synchronize()
    assert cnt.n == {"fwd_dual": 1, "attention": 0, "bwd_dual": 0}, cnt.n
    ro, rt, _, _ = oracle.fwd_dual(*(np64(x) for x in xs), mask, mm)
    tol = 1e-4 if dtype == "f32" else 2e-2
    assert np.abs(np64(o) - ro).max() <= tol and np.abs(np64(t_o) - rt).max() <= tol
    # the drop-in takes the same fused route under torch.func.jvp
    o2, t2 = torch.func.jvp(lambda q, k, v: jvp_attention(q, k, v, attn_mask=m, is_causal=causal),
                            tuple(xs[:3]), tuple(xs[3:]))
    torch.cuda.synchronize()
    assert cnt.n["fwd_dual"] == 2 and cnt.n["attention"] == 0
    assert torch.equal(o, o2) and torch.equal(t_o, t2)


@pytest.mark.parametrize("dtype,D,mask", CALL_FORM_CASES)
def test_pages_call_form_trains_through_the_tangent(dtype, D, mask, monkeypatch):
    # The primal and tangent returned by torch.func.jvp are differentiable:
    # Loss = <gO, O> + <gtO, tO> reaches q, k, v and the tangents through one
    # bwd_dual launch, and equals the oracle's reverse mode of the dual map.
    w, inp, xs, m, mm = _inputs(dtype, D, mask, seed=70 + D, requires_grad=True)
    cnt = _Count(monkeypatch)
    causal = mask == "causal"
    o, t_o = torch.func.jvp(
        lambda q, k, v: JVPAttn.fwd_dual(q, k, v, attn_mask=m, is_causal=causal),
        tuple(xs[:3]), tuple(xs[3:]))
    assert o.requires_grad and t_o.requires_grad
    g_o, g_to = inp.g_o.cuda(), inp.g_to.cuda()
    loss = (o.float() * g_o.float()).sum() + (t_o.float() * g_to.float()).sum()
    loss.backward()
    torch.cuda.synchronize()
    assert cnt.n == {"fwd_dual": 1, "attention": 0, "bwd_dual": 1}, cnt.n
    ref = oracle.bwd_dual(*(np64(x) for x in xs), np64(g_o), np64(g_to), mask, mm)
    tol = 1e-4 if dtype == "f32" else 2e-2
    for x, r in zip(xs, ref):
        assert np.abs(np64(x.grad) - r).max() <= tol * max(1.0, np.abs(r).max())


@pytest.mark.parametrize("dtype,D,mask", [("bf16", 64, "none"), ("f16", 128, "causal"),
                                          ("f32", 24, "bool")])
def test_hessian_vector_product_reverse_over_forward(dtype, D, mask):
    # f(q, k, v) = <w, attention(q, k, v)>.  The tangent of f along
    # u = (uq, uk, uv) is grad f . u; its gradient with respect to (q, k, v)
    # is the Hessian-vector product H u (the project page's Description names
    # HVPs).  Formed here by reverse mode over torch.func.jvp of
    # JVPAttn.fwd_dual, and compared with the oracle's reverse mode of the
    # dual map with cotangents (0, w) (whose HVP identity the CPU pins fix
    # against finite differences of the gradient).
    w_, inp, xs, m, mm = _inputs(dtype, D, mask, seed=80 + D)
    q, k, v = (x.detach().requires_grad_(True) for x in xs[:3])
    u = [x.detach() for x in xs[3:]]
    wt = inp.g_to.cuda()
    causal = mask == "causal"
    f = lambda q_, k_, v_: (JVPAttn.fwd_dual(q_, k_, v_, attn_mask=m, is_causal=causal).float()
                            * wt.float()).sum()
    val, dir_deriv = torch.func.jvp(f, (q, k, v), tuple(u))
    hq, hk, hv = torch.autograd.grad(dir_deriv, (q, k, v))
    z = np.zeros(q.shape)
    ref = oracle.bwd_dual(np64(q), np64(k), np64(v), *(np64(x) for x in u), z, np64(wt), mask, mm)
    tol = 1e-4 if dtype == "f32" else 2e-2
    for got, r in zip((hq, hk, hv), ref[:3]):
        assert np.abs(np64(got) - r).max() <= tol * max(1.0, np.abs(r).max())
    # the value is f itself
    ro, _, _, _ = oracle.fwd_dual(np64(q), np64(k), np64(v), mask_kind=mask, mask=mm)
    fv = float((ro * np64(wt)).sum())
    assert abs(val.item() - fv) <= tol * max(1.0, np.abs(ro * np64(wt)).sum())


def test_training_a_model_through_torch_func_jvp():
    # The page's pattern: pred, df = torch.func.jvp(model, (x,), (gt,)) with the
    # model's attention being JVPAttn.fwd_dual, then a loss on (pred, df)
    # trained by autograd.  The weight gradients match the same model built on
    # plain float64 softmax attention (torch, CPU) to float32 accuracy.
    torch.manual_seed(0)
    B, N, C, H, D = 2, 40, 48, 2, 24
    W64 = torch.randn(3, C, H * D, dtype=torch.float64) / C ** 0.5
    x64 = torch.randn(B, N, C, dtype=torch.float64)
    gt64 = torch.randn(B, N, C, dtype=torch.float64)

    def model(W, attn):
        def m(x):
            q, k, v = ((x @ W[i]).view(B, N, H, D).transpose(1, 2) for i in range(3))
            o = attn(q, k, v)
            return torch.tanh(o.transpose(1, 2).reshape(B, N, H * D))
        return m

    def plain_attn(q, k, v):
        n = q.shape[2]
        s = (q @ k.transpose(-1, -2)) / D ** 0.5
        s = s.masked_fill(~torch.ones(n, n, dtype=torch.bool).tril(), float("-inf"))
        return torch.softmax(s, -1) @ v

    grads = []
    for dev, dt, attn in (("cuda", torch.float32,
                           lambda q, k, v: JVPAttn.fwd_dual(q, k, v, is_causal=True)),
                          ("cpu", torch.float64, plain_attn)):
        W = W64.to(dev, dt).requires_grad_(True)
        pred, df = torch.func.jvp(model(W, attn), (x64.to(dev, dt),), (gt64.to(dev, dt),))
        loss = (pred ** 2).mean() + (df ** 2).mean()
        loss.backward()
        grads.append((loss.item(), W.grad.to("cpu", torch.float64)))
    (l0, g0), (l1, g1) = grads
    assert abs(l0 - l1) <= 1e-5 * abs(l1)
    assert (g0 - g1).abs().max().item() <= 1e-4 * g1.abs().max().item()
