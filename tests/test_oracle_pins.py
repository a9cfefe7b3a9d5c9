"""Pins of the float64 oracle against facts fixed independently of its code.

Each test checks the oracle against something other than itself: central
finite differences of its own primal map, closed-form special cases, exact
invariants, brute force, and a library (torch.func) evaluation of the plain
softmax-attention expression.  Together they are chosen so that a dropped
term, a wrong sign, a wrong scale placement, a transposed operand or a wrong
mask polarity fails at least one of them.

Method: "JVP Flash Attention" project page, Description (a kernel for JVPs
and HVPs of attention) and Usage (a drop-in for scaled_dot_product_attention
with attn_mask; fwd_dual under torch.func.jvp).
"""

import math

import numpy as np
import pytest
import torch

import oracle

MASKS = ["none", "bool", "additive", "causal"]


def rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def make(B=1, H=2, N=9, D=6, mask="none", seed=0, Nk=None):
    Nk = N if Nk is None else Nk
    rng = np.random.default_rng(seed)
    q, dq = (rng.standard_normal((B, H, N, D)) for _ in range(2))
    k, v, dk, dv = (rng.standard_normal((B, H, Nk, D)) for _ in range(4))
    m = None
    if mask == "bool":
        m = rng.random((B, 1, N, Nk)) < 0.7
        for i in range(min(N, Nk)):
            m[:, :, i, i] = True
    elif mask == "additive":
        m = rng.standard_normal((B, 1, N, Nk))
    return q, k, v, dq, dk, dv, m


def primal(q, k, v, mask_kind, m, scale=None):
    return oracle.fwd_dual(q, k, v, mask_kind=mask_kind, mask=m, scale=scale)


@pytest.mark.parametrize("mask", MASKS)
def test_tangent_matches_central_finite_differences(mask):
    # tO must be the directional derivative of O: [O(x+h t) - O(x-h t)] / 2h.
    q, k, v, dq, dk, dv, m = make(B=1, H=2, N=11, D=5, mask=mask, seed=1)
    o, t_o, lse, mu = oracle.fwd_dual(q, k, v, dq, dk, dv, mask, m)
    h = 1e-5
    op, _, lp, _ = primal(q + h * dq, k + h * dk, v + h * dv, mask, m)
    om, _, lm, _ = primal(q - h * dq, k - h * dk, v - h * dv, mask, m)
    fd = (op - om) / (2 * h)
    rel = np.abs(fd - t_o).max() / np.abs(t_o).max()
    assert rel <= 1e-6, rel
    # mu is the tangent of lse.
    fd_l = (lp - lm) / (2 * h)
    assert np.abs(fd_l - mu).max() / np.abs(mu).max() <= 1e-6


@pytest.mark.parametrize("mask", MASKS)
def test_tangent_is_linear_in_the_tangents(mask):
    q, k, v, dq1, dk1, dv1, m = make(N=10, D=4, mask=mask, seed=2)
    _, _, _, dq2, dk2, dv2, _ = make(N=10, D=4, mask="none", seed=3)
    a, b = 0.7, -1.9
    _, t1, _, mu1 = oracle.fwd_dual(q, k, v, dq1, dk1, dv1, mask, m)
    _, t2, _, mu2 = oracle.fwd_dual(q, k, v, dq2, dk2, dv2, mask, m)
    _, t12, _, mu12 = oracle.fwd_dual(q, k, v, a * dq1 + b * dq2, a * dk1 + b * dk2,
                                      a * dv1 + b * dv2, mask, m)
    ref = a * t1 + b * t2
    assert np.abs(t12 - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max())
    assert np.abs(mu12 - (a * mu1 + b * mu2)).max() <= 1e-12 * max(1.0, np.abs(mu12).max())


@pytest.mark.parametrize("mask", MASKS)
def test_zero_tangent_gives_zero(mask):
    q, k, v, dq, dk, dv, m = make(N=8, D=4, mask=mask, seed=4)
    z = np.zeros_like(q)
    _, t_o, _, mu = oracle.fwd_dual(q, k, v, z, z, z, mask, m)
    assert np.all(t_o == 0.0) and np.all(mu == 0.0)
    _, t_o, _, mu = oracle.fwd_dual(q, k, v, None, None, None, mask, m)
    assert np.all(t_o == 0.0) and np.all(mu == 0.0)


def plain_softmax_weights(q, k, mask, m, scale):
    """Row-softmax weights written independently (numpy, no dual numbers)."""
    B, H, N, D = q.shape
    Nk = k.shape[2]
    s = scale * np.einsum("bhid,bhjd->bhij", q, k)
    keep = np.ones((B, H, N, Nk), dtype=bool)
    if mask == "bool":
        keep = np.broadcast_to(m, keep.shape).copy()
    elif mask == "additive":
        s = s + m
    elif mask == "causal":
        keep = np.broadcast_to(np.tril(np.ones((N, Nk), dtype=bool)), keep.shape).copy()
    s = np.where(keep, s, -np.inf)
    s = s - s.max(-1, keepdims=True)
    e = np.exp(s)
    return e / e.sum(-1, keepdims=True), keep


@pytest.mark.parametrize("mask", MASKS)
def test_dv_only_tangent_is_P_times_dV(mask):
    q, k, v, _, _, dv, m = make(N=12, D=5, mask=mask, seed=5)
    z = np.zeros_like(q)
    _, t_o, _, mu = oracle.fwd_dual(q, k, v, z, z, dv, mask, m)
    P, _ = plain_softmax_weights(q, k, mask, m, 1 / math.sqrt(5))
    assert np.abs(t_o - P @ dv).max() <= 1e-12
    assert np.all(mu == 0.0)


@pytest.mark.parametrize("mask", MASKS)
def test_tangent_V_gives_O(mask):
    # O is linear in V, so the tangent along (0, 0, V) is O itself.
    q, k, v, _, _, _, m = make(N=9, D=3, mask=mask, seed=6)
    z = np.zeros_like(q)
    o, t_o, _, _ = oracle.fwd_dual(q, k, v, z, z, v, mask, m)
    assert np.abs(t_o - o).max() <= 1e-13


@pytest.mark.parametrize("mask", MASKS)
def test_shifting_all_keys_along_one_direction_gives_zero_tangent(mask):
    # dK_j = u for all j shifts every logit of row i by scale*q_i.u: softmax is
    # invariant to a per-row shift, so tO = 0 and mu = scale*q_i.u.
    q, k, v, _, _, _, m = make(N=9, D=4, mask=mask, seed=7)
    u = np.array([0.3, -1.2, 0.5, 2.0])
    dk = np.broadcast_to(u, k.shape).copy()
    z = np.zeros_like(q)
    _, t_o, _, mu = oracle.fwd_dual(q, k, v, z, dk, z, mask, m)
    assert np.abs(t_o).max() <= 1e-13
    assert np.abs(mu - (q @ u) / 2.0).max() <= 1e-13


def test_zero_queries_average_the_kept_values():
    rng = np.random.default_rng(8)
    B, H, N, D = 2, 2, 10, 4
    k, v = rng.standard_normal((2, B, H, N, D))
    q = np.zeros((B, H, N, D))
    o, _, lse, _ = oracle.fwd_dual(q, k, v, mask_kind="none")
    assert np.abs(o - v.mean(axis=2, keepdims=True)).max() <= 1e-14
    assert np.abs(lse - math.log(N)).max() <= 1e-14
    o, _, _, _ = oracle.fwd_dual(q, k, v, mask_kind="causal")
    ref = np.cumsum(v, axis=2) / np.arange(1, N + 1)[None, None, :, None]
    assert np.abs(o - ref).max() <= 1e-14
    keep = rng.random((B, 1, N, N)) < 0.5
    keep[..., 0] = True
    o, _, _, _ = oracle.fwd_dual(q, k, v, mask_kind="bool", mask=keep)
    kb = np.broadcast_to(keep, (B, H, N, N)).astype(float)
    ref = (kb @ v) / kb.sum(-1, keepdims=True)
    assert np.abs(o - ref).max() <= 1e-14


def test_single_key():
    q, k, v, dq, dk, dv, _ = make(B=2, H=3, N=1, D=7, seed=9)
    o, t_o, lse, mu = oracle.fwd_dual(q, k, v, dq, dk, dv, scale=0.37)
    assert np.array_equal(o, v) and np.array_equal(t_o, dv)
    assert np.abs(lse - 0.37 * (q * k).sum(-1)).max() <= 1e-14
    # softmax of one logit is constant 1, so its tangent mu is the logit tangent
    assert np.abs(mu - 0.37 * ((dq * k).sum(-1) + (q * dk).sum(-1))).max() <= 1e-14


@pytest.mark.parametrize("mask", MASKS)
def test_closed_form_of_the_jvp(mask):
    # Derived closed form: dS = s (dQ K^T + Q dK^T), mu = rowsum(P*dS),
    # tO = (P*dS) V - mu O + P dV.  Evaluated here with plain numpy matrices.
    q, k, v, dq, dk, dv, m = make(B=2, H=2, N=13, D=6, mask=mask, seed=10)
    s = 0.41
    o, t_o, lse, mu = oracle.fwd_dual(q, k, v, dq, dk, dv, mask, m, scale=s)
    P, keep = plain_softmax_weights(q, k, mask, m, s)
    dS = s * (dq @ np.swapaxes(k, -1, -2) + q @ np.swapaxes(dk, -1, -2))
    dS = np.where(keep, dS, 0.0)
    mu_ref = (P * dS).sum(-1)
    O_ref = P @ v
    tO_ref = (P * dS) @ v - mu_ref[..., None] * O_ref + P @ dv
    assert np.abs(o - O_ref).max() <= 1e-12
    assert np.abs(t_o - tO_ref).max() <= 1e-12
    assert np.abs(mu - mu_ref).max() <= 1e-12


def torch_attention(q, k, v, mask, m, scale):
    """Plain float64 softmax attention in torch, as SDPA defines attn_mask."""
    s = scale * q @ k.transpose(-1, -2)
    if mask == "bool":
        s = s.masked_fill(~m, float("-inf"))
    elif mask == "additive":
        s = s + m
    elif mask == "causal":
        n, nk = s.shape[-2:]
        s = s.masked_fill(~torch.ones(n, nk, dtype=torch.bool).tril(), float("-inf"))
    return torch.softmax(s, dim=-1) @ v


@pytest.mark.parametrize("mask", MASKS)
def test_agrees_with_torch_func_jvp(mask):
    q, k, v, dq, dk, dv, m = make(B=2, H=2, N=14, D=8, mask=mask, seed=11)
    s = 1 / math.sqrt(8)
    o, t_o, _, _ = oracle.fwd_dual(q, k, v, dq, dk, dv, mask, m)
    T = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    mt = None if m is None else T(m)
    f = lambda q_, k_, v_: torch_attention(q_, k_, v_, mask, mt, s)
    o_ref, t_ref = torch.func.jvp(f, (T(q), T(k), T(v)), (T(dq), T(dk), T(dv)))
    assert np.abs(o - o_ref.numpy()).max() <= 1e-12
    assert np.abs(t_o - t_ref.numpy()).max() <= 1e-12


def test_lse_brute_force():
    q, k, v, _, _, _, m = make(B=1, H=1, N=7, D=3, mask="additive", seed=12)
    s = 0.5
    _, _, lse, _ = oracle.fwd_dual(q, k, v, mask_kind="additive", mask=m, scale=s)
    for i in range(7):
        terms = [math.exp(s * float(q[0, 0, i] @ k[0, 0, j]) + m[0, 0, i, j]) for j in range(7)]
        assert abs(lse[0, 0, i] - math.log(math.fsum(terms))) <= 1e-13


def test_fully_masked_row_and_minus_inf_bias():
    q, k, v, dq, dk, dv, _ = make(B=1, H=1, N=6, D=4, seed=13)
    keep = np.ones((1, 1, 6, 6), dtype=bool)
    keep[0, 0, 2, :] = False
    keep[0, 0, 4, 1] = False
    o, t_o, lse, mu = oracle.fwd_dual(q, k, v, dq, dk, dv, "bool", keep)
    assert np.all(o[0, 0, 2] == 0) and np.all(t_o[0, 0, 2] == 0)
    assert lse[0, 0, 2] == -np.inf and mu[0, 0, 2] == 0
    # An additive -inf excludes exactly as a False keep entry does.
    bias = np.where(keep, 0.0, -np.inf)
    o2, t2, l2, mu2 = oracle.fwd_dual(q, k, v, dq, dk, dv, "additive", bias)
    assert np.array_equal(o, o2) and np.array_equal(t_o, t2)
    assert np.array_equal(lse, l2) and np.array_equal(mu, mu2)


def test_causal_equals_lower_triangular_keep_mask_and_rows_subset():
    q, k, v, dq, dk, dv, _ = make(B=2, H=2, N=9, D=4, seed=14)
    tril = np.broadcast_to(np.tril(np.ones((9, 9), dtype=bool)), (2, 1, 9, 9))
    a = oracle.fwd_dual(q, k, v, dq, dk, dv, "causal")
    b = oracle.fwd_dual(q, k, v, dq, dk, dv, "bool", tril)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    rows = np.array([0, 5, 17, 35])
    o, t_o, lse, mu = oracle.fwd_dual_rows(q, k, v, dq, dk, dv, rows, "causal")
    flat = [x.reshape(36, -1) for x in a]
    assert np.array_equal(o, flat[0][rows]) and np.array_equal(t_o, flat[1][rows])
    assert np.array_equal(lse, flat[2][rows, 0]) and np.array_equal(mu, flat[3][rows, 0])


def test_per_head_mask_broadcast():
    q, k, v, dq, dk, dv, m = make(B=2, H=3, N=6, D=4, mask="bool", seed=15)
    full = np.broadcast_to(m, (2, 3, 6, 6)).copy()
    a = oracle.fwd_dual(q, k, v, dq, dk, dv, "bool", m)
    b = oracle.fwd_dual(q, k, v, dq, dk, dv, "bool", full)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


# ----------------------------------------------------------------- reverse mode

@pytest.mark.parametrize("mask", MASKS)
def test_backward_matches_finite_differences(mask):
    # Gradient of Loss = <gO, O> + <gtO, tO> along a random direction, against
    # a central difference of Loss computed from the forward oracle.
    q, k, v, dq, dk, dv, m = make(B=1, H=2, N=8, D=4, mask=mask, seed=16)
    rng = np.random.default_rng(17)
    g_o, g_to = rng.standard_normal((2,) + q.shape)
    grads = oracle.bwd_dual(q, k, v, dq, dk, dv, g_o, g_to, mask, m)
    xs = [q, k, v, dq, dk, dv]

    def loss(vals):
        o, t_o, _, _ = oracle.fwd_dual(*vals, mask, m)
        return float((g_o * o).sum() + (g_to * t_o).sum())

    h = 1e-5
    for idx in range(6):
        u = rng.standard_normal(xs[idx].shape)
        plus = [x + h * u if n == idx else x for n, x in enumerate(xs)]
        minus = [x - h * u if n == idx else x for n, x in enumerate(xs)]
        fd = (loss(plus) - loss(minus)) / (2 * h)
        an = float((grads[idx] * u).sum())
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (idx, fd, an)


def test_backward_identities_and_torch_double_backward():
    q, k, v, dq, dk, dv, m = make(B=1, H=2, N=10, D=6, mask="causal", seed=18)
    rng = np.random.default_rng(19)
    g_o, g_to = rng.standard_normal((2,) + q.shape)
    s = 1 / math.sqrt(6)
    grads = oracle.bwd_dual(q, k, v, dq, dk, dv, g_o, g_to, "causal")
    # tO is linear in dV with coefficient P, so d Loss / d dV = P^T gtO exactly.
    P, _ = plain_softmax_weights(q, k, "causal", None, s)
    assert np.abs(grads[5] - np.swapaxes(P, -1, -2) @ g_to).max() <= 1e-12
    # Library cross-check: reverse mode through torch.func.jvp in float64.
    T = lambda a: torch.from_numpy(np.ascontiguousarray(a)).requires_grad_(True)
    ts = [T(x) for x in (q, k, v, dq, dk, dv)]
    f = lambda q_, k_, v_: torch_attention(q_, k_, v_, "causal", None, s)
    o, t_o = torch.func.jvp(f, tuple(ts[:3]), tuple(ts[3:]))
    L = (torch.from_numpy(g_o) * o).sum() + (torch.from_numpy(g_to) * t_o).sum()
    ref = torch.autograd.grad(L, ts)
    for g, r in zip(grads, ref):
        assert np.abs(g - r.numpy()).max() <= 1e-11


# ------------------------------------------------- query and key lengths differ
# The GPU tests with Nq != Nk (cross-length parity, split-KV over long key
# ranges, the backward at Nq != Nk) rest on the oracle's key-row indexing, its
# top-left causal rule (key j kept for query i iff j <= i, whatever Nk) and the
# reverse mode's key-side offsets at unequal lengths.  These pins fix those
# paths against finite differences, a torch.func evaluation of the plain
# expression, brute force and the exact dV identity, at shapes where a slip
# between Nq and Nk (or a causal rule aligned bottom-right) changes the result.
CROSS = [(5, 13), (13, 5), (1, 9)]


@pytest.mark.parametrize("mask", MASKS)
@pytest.mark.parametrize("Nq,Nk", CROSS)
def test_cross_length_tangent_matches_central_finite_differences(mask, Nq, Nk):
    q, k, v, dq, dk, dv, m = make(B=1, H=2, N=Nq, D=5, mask=mask, seed=100 + Nq, Nk=Nk)
    o, t_o, lse, mu = oracle.fwd_dual(q, k, v, dq, dk, dv, mask, m)
    assert o.shape == (1, 2, Nq, 5) and lse.shape == (1, 2, Nq)
    h = 1e-5
    op, _, lp, _ = primal(q + h * dq, k + h * dk, v + h * dv, mask, m)
    om, _, lm, _ = primal(q - h * dq, k - h * dk, v - h * dv, mask, m)
    fd = (op - om) / (2 * h)
    assert np.abs(fd - t_o).max() / np.abs(t_o).max() <= 1e-6
    fd_l = (lp - lm) / (2 * h)
    assert np.abs(fd_l - mu).max() / max(np.abs(mu).max(), 1e-300) <= 1e-6


@pytest.mark.parametrize("mask", MASKS)
@pytest.mark.parametrize("Nq,Nk", CROSS)
def test_cross_length_agrees_with_torch_func_jvp(mask, Nq, Nk):
    q, k, v, dq, dk, dv, m = make(B=2, H=2, N=Nq, D=8, mask=mask, seed=110 + Nk, Nk=Nk)
    s = 1 / math.sqrt(8)
    o, t_o, lse, mu = oracle.fwd_dual(q, k, v, dq, dk, dv, mask, m)
    T = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    mt = None if m is None else T(m)
    f = lambda q_, k_, v_: torch_attention(q_, k_, v_, mask, mt, s)
    o_ref, t_ref = torch.func.jvp(f, (T(q), T(k), T(v)), (T(dq), T(dk), T(dv)))
    assert np.abs(o - o_ref.numpy()).max() <= 1e-12
    assert np.abs(t_o - t_ref.numpy()).max() <= 1e-12
    # lse by brute force over the kept keys of every row
    P, keep = plain_softmax_weights(q, k, mask, m, s)
    S = s * np.einsum("bhid,bhjd->bhij", q, k) + (m if mask == "additive" else 0.0)
    for b in range(2):
        for hh in range(2):
            for i in range(Nq):
                terms = [math.exp(S[b, hh, i, j]) for j in range(Nk) if keep[b, hh, i, j]]
                assert abs(lse[b, hh, i] - math.log(math.fsum(terms))) <= 1e-12


@pytest.mark.parametrize("Nq,Nk", CROSS)
def test_cross_length_causal_is_top_left_aligned(Nq, Nk):
    # Query i sees keys 0..i: with dV only on the keys j > i of every row, the
    # tangent of row i is zero; keys beyond Nq - 1 are never seen at all.
    q, k, v, _, _, _, _ = make(B=1, H=1, N=Nq, D=4, seed=120 + Nq, Nk=Nk)
    z = np.zeros_like(q)
    if Nk > Nq:
        dv = np.zeros_like(v)
        dv[:, :, Nq:] = 1.0  # only keys no query may see
        _, t_o, _, _ = oracle.fwd_dual(q, k, v, z, np.zeros_like(k), dv, "causal")
        assert np.all(t_o == 0.0)
    # row 0 keeps only key 0: O = V_0, lse = s q_0 . k_0
    o, _, lse, _ = oracle.fwd_dual(q, k, v, mask_kind="causal", scale=0.3)
    assert np.array_equal(o[0, 0, 0], v[0, 0, 0])
    assert abs(lse[0, 0, 0] - 0.3 * float(q[0, 0, 0] @ k[0, 0, 0])) <= 1e-14
    # the last row keeps min(Nq, Nk) keys: with q = 0 it averages them
    o, _, _, _ = oracle.fwd_dual(np.zeros_like(q), k, v, mask_kind="causal")
    n = min(Nq, Nk)
    assert np.abs(o[0, 0, Nq - 1] - v[0, 0, :n].mean(axis=0)).max() <= 1e-14


@pytest.mark.parametrize("mask", MASKS)
@pytest.mark.parametrize("Nq,Nk", CROSS)
def test_cross_length_backward_matches_finite_differences(mask, Nq, Nk):
    q, k, v, dq, dk, dv, m = make(B=1, H=2, N=Nq, D=4, mask=mask, seed=130 + Nq + Nk, Nk=Nk)
    rng = np.random.default_rng(131)
    g_o, g_to = rng.standard_normal((2,) + q.shape)
    grads = oracle.bwd_dual(q, k, v, dq, dk, dv, g_o, g_to, mask, m)
    xs = [q, k, v, dq, dk, dv]
    for g, x in zip(grads, xs):
        assert g.shape == x.shape

    def loss(vals):
        o, t_o, _, _ = oracle.fwd_dual(*vals, mask, m)
        return float((g_o * o).sum() + (g_to * t_o).sum())

    h = 1e-5
    for idx in range(6):
        u = rng.standard_normal(xs[idx].shape)
        plus = [x + h * u if n == idx else x for n, x in enumerate(xs)]
        minus = [x - h * u if n == idx else x for n, x in enumerate(xs)]
        fd = (loss(plus) - loss(minus)) / (2 * h)
        an = float((grads[idx] * u).sum())
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (idx, fd, an)


@pytest.mark.parametrize("mask", MASKS)
@pytest.mark.parametrize("Nq,Nk", CROSS)
def test_cross_length_backward_identity_and_torch_double_backward(mask, Nq, Nk):
    q, k, v, dq, dk, dv, m = make(B=1, H=2, N=Nq, D=6, mask=mask, seed=140 + Nk, Nk=Nk)
    rng = np.random.default_rng(141)
    g_o, g_to = rng.standard_normal((2,) + q.shape)
    s = 1 / math.sqrt(6)
    grads = oracle.bwd_dual(q, k, v, dq, dk, dv, g_o, g_to, mask, m)
    P, _ = plain_softmax_weights(q, k, mask, m, s)
    assert np.abs(grads[5] - np.swapaxes(P, -1, -2) @ g_to).max() <= 1e-12
    T = lambda a: torch.from_numpy(np.ascontiguousarray(a)).requires_grad_(True)
    ts = [T(x) for x in (q, k, v, dq, dk, dv)]
    mt = None if m is None else torch.from_numpy(np.ascontiguousarray(m))
    f = lambda q_, k_, v_: torch_attention(q_, k_, v_, mask, mt, s)
    o, t_o = torch.func.jvp(f, tuple(ts[:3]), tuple(ts[3:]))
    L = (torch.from_numpy(g_o) * o).sum() + (torch.from_numpy(g_to) * t_o).sum()
    ref = torch.autograd.grad(L, ts)
    for g, r in zip(grads, ref):
        assert np.abs(g - r.numpy()).max() <= 1e-11


# ------------------------------------------- Hessian-vector products (reverse over forward)
@pytest.mark.parametrize("mask", MASKS)
def test_reverse_mode_of_the_tangent_is_a_hessian_vector_product(mask):
    # For f(q, k, v) = <w, O>, the tangent along u = (dq, dk, dv) is <w, tO> =
    # grad f . u.  Its gradient with respect to (q, k, v) is the Hessian-vector
    # product H u (the use named in the project page's Description); with
    # respect to u it is grad f itself.  The oracle's reverse mode with
    # cotangents (gO, gtO) = (0, w) must give both: H u against a central
    # difference of grad f (itself the reverse mode with (w, 0)), grad f exactly.
    q, k, v, dq, dk, dv, m = make(B=1, H=2, N=7, D=4, mask=mask, seed=150, Nk=9)
    w = np.random.default_rng(151).standard_normal(q.shape)
    z = np.zeros_like(q)
    hvp = oracle.bwd_dual(q, k, v, dq, dk, dv, z, w, mask, m)

    def grad_f(qq, kk, vv):
        return oracle.bwd_dual(qq, kk, vv, dq, dk, dv, w, z, mask, m)[:3]

    h = 1e-5
    gp = grad_f(q + h * dq, k + h * dk, v + h * dv)
    gm = grad_f(q - h * dq, k - h * dk, v - h * dv)
    for a, b, c in zip(hvp[:3], gp, gm):
        fd = (b - c) / (2 * h)
        assert np.abs(a - fd).max() <= 1e-6 * max(1.0, np.abs(fd).max())
    g0 = grad_f(q, k, v)
    for a, b in zip(hvp[3:], g0):
        assert np.abs(a - b).max() <= 1e-12 * max(1.0, np.abs(b).max())


@pytest.mark.parametrize("mask", MASKS)
@pytest.mark.parametrize("Nq,Nk", [(9, 9), (5, 13), (13, 5)])
def test_zero_tangent_reverse_mode_is_the_primal_backward(mask, Nq, Nk):
    # The primal backward of attention (gradients of <gO, O> with respect to
    # q, k, v) is the reverse mode of the dual map with dQ = dK = dV = 0 and
    # gtO = 0; the tangent-side gradients are then those of the linear map
    # (dq, dk, dv) -> tO at the same point, which gtO = 0 makes zero.  Checked
    # against torch.autograd of a float64 softmax attention (no jvp involved)
    # and against central differences of the oracle's own O.
    q, k, v, _, _, _, m = make(B=1, H=2, N=Nq, D=6, mask=mask, seed=41 + Nq, Nk=Nk)
    rng = np.random.default_rng(42 + Nk)
    g_o = rng.standard_normal(q.shape)
    s = 1 / math.sqrt(6)
    z = [np.zeros_like(x) for x in (q, k, v)]
    grads = oracle.bwd_dual(q, k, v, *z, g_o, np.zeros_like(g_o), mask, m)
    for g in grads[3:]:
        assert np.abs(g).max() == 0.0
    T = lambda a: torch.from_numpy(np.ascontiguousarray(a)).requires_grad_(True)
    ts = [T(x) for x in (q, k, v)]
    mt = None if m is None else torch.from_numpy(m)
    o = torch_attention(*ts, mask, mt, s)
    ref = torch.autograd.grad((torch.from_numpy(g_o) * o).sum(), ts)
    for g, r in zip(grads[:3], ref):
        assert np.abs(g - r.detach().numpy()).max() <= 1e-12
    h = 1e-6
    for which in range(3):
        u = rng.standard_normal((q, k, v)[which].shape)
        xp = [x.copy() for x in (q, k, v)]
        xm = [x.copy() for x in (q, k, v)]
        xp[which] += h * u
        xm[which] -= h * u
        fd = ((primal(*xp, mask, m)[0] - primal(*xm, mask, m)[0]) * g_o).sum() / (2 * h)
        assert abs(fd - (grads[which] * u).sum()) <= 1e-6 * max(1.0, abs(fd))
