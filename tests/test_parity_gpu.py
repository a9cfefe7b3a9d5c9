"""GPU parity: the CUDA path against the float64 oracle on the same inputs.

Tolerances (max-abs on O and tO, unit-variance inputs): 1e-4 for float32
inputs, 2e-2 for fp16/bf16 inputs.  lse is checked too (1e-5 / 1e-3).
Boolean and causal masking must be exact in which keys contribute: perturbing
an excluded key's K, V, dK or dV leaves every output bit-identical.

The oracle runs on the dtype-rounded inputs upcast to float64, so the only
differences are the GPU's own rounding (fp32 accumulation, 16-bit P and
P*dS operands, 16-bit outputs).
"""

import json
import math
import os

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
    return None if t is None else t.detach().to("cpu", torch.float64).numpy()


def mask_for_oracle(w, inp):
    if w.mask == "bool":
        return "bool", inp.mask.numpy()
    if w.mask == "additive":
        return "additive", inp.mask.double().numpy()
    return w.mask, None


def run_gpu(w, inp, scale=None):
    dev = "cuda"
    g = [x.to(dev) for x in (inp.q, inp.k, inp.v, inp.dq, inp.dk, inp.dv)]
    m = inp.mask.to(dev) if inp.mask is not None else None
    o, t_o, lse, mu = A.fwd_dual(*g, attn_mask=m, is_causal=(w.mask == "causal"), scale=scale,
                                 return_stats=True)
    torch.cuda.synchronize()
    return o, t_o, lse, mu, A.last_path()


def log_error(name, **errs):
    """Append the measured errors to $JVP_PARITY_LOG (one JSON object per line)."""
    path = os.environ.get("JVP_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"case": name, **{k: float(v) for k, v in errs.items()}}) + "\n")


def compare_full(w, scale=None, expect_path=None):
    inp = synth.make_inputs(w)
    o, t_o, lse, mu, path = run_gpu(w, inp, scale)
    if expect_path is not None:
        # 1: tensor-core kernel (3: the same with split-KV and the merge kernel;
        # 4: the same with each key range split inside a 2-CTA cluster)
        ok = path in A.TENSOR_CORE_PATHS if expect_path == 1 else path == expect_path
        assert ok, f"expected path {expect_path}, got {path}"
    kind, m = mask_for_oracle(w, inp)
    ro, rt, rl, rm = oracle.fwd_dual(np64(inp.q), np64(inp.k), np64(inp.v), np64(inp.dq),
                                     np64(inp.dk), np64(inp.dv), kind, m, scale=scale)
    eo = np.abs(np64(o) - ro).max()
    et = np.abs(np64(t_o) - rt).max()
    fin = np.isfinite(rl)
    el = np.abs(np64(lse)[fin] - rl[fin]).max() if fin.any() else 0.0
    assert np.array_equal(np.isfinite(np64(lse)), fin)
    em = np.abs(np64(mu) - rm).max()
    tol = TOL[w.dtype]
    log_error(w.name, o=eo, t_o=et, lse=el, mu=em)
    assert eo <= tol and et <= tol, (w.name, eo, et)
    assert el <= LSE_TOL[w.dtype], (w.name, el)
    assert em <= 20 * tol, (w.name, em)
    return eo, et


# ------------------------------------------------------------------ small shapes
SMALL_N = [1, 17, 63, 64, 65, 127, 128, 129, 200, 333]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("N", SMALL_N)
@pytest.mark.parametrize("mask", ["none", "causal"])
def test_tensor_core_path_small(dtype, D, N, mask):
    w = synth.small(dtype, 2, 3, N, D, mask, seed=N + D)
    compare_full(w, expect_path=1)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("N", [17, 64, 130, 257])
@pytest.mark.parametrize("mask", ["bool", "additive"])
def test_tensor_core_path_masks(dtype, D, N, mask):
    w = synth.small(dtype, 2, 2, N, D, mask, seed=7 * N + D)
    compare_full(w, expect_path=1)


@pytest.mark.parametrize("dtype,D", [("bf16", 64), ("f16", 128), ("f32", 40)])
@pytest.mark.parametrize("Nq,Nk", [(100, 300), (300, 77), (1, 129), (130, 1)])
@pytest.mark.parametrize("mask", ["none", "causal", "bool", "additive"])
def test_query_and_key_lengths_differ(dtype, D, Nq, Nk, mask):
    # causal keeps key j for query i when j <= i (top-left aligned)
    w = synth.small(dtype, 1, 2, Nq, D, mask, seed=Nq + 3 * Nk, Nk=Nk)
    compare_full(w, expect_path=2 if dtype == "f32" else 1)


@pytest.mark.parametrize("D", [1, 16, 33, 64, 100, 128])
@pytest.mark.parametrize("mask", ["none", "bool", "additive", "causal"])
def test_cuda_core_path_f32(D, mask):
    w = synth.small("f32", 2, 2, 45, D, mask, seed=D)
    compare_full(w, expect_path=2)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("D", [8, 16, 24, 32, 48, 80, 96, 112, 20, 100])
def test_half_precision_other_head_dims(dtype, D):
    # Multiples of 8 up to 128 take the tensor-core kernels (the D = 64 or 128
    # kernel, columns past D zero-filled); other head dimensions the
    # CUDA-core kernel.
    w = synth.small(dtype, 1, 2, 70, D, "causal", seed=D)
    compare_full(w, expect_path=1 if D % 8 == 0 else 2)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("D", [8, 40, 72, 96, 120])
@pytest.mark.parametrize("N", [129, 300])
@pytest.mark.parametrize("mask", ["none", "causal", "bool", "additive"])
def test_tensor_core_path_head_dims_between_powers_of_two(dtype, D, N, mask):
    w = synth.small(dtype, 2, 3, N, D, mask, seed=N + D + len(mask))
    compare_full(w, expect_path=1)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("D", [16, 32])
@pytest.mark.parametrize("N", [1, 17, 64, 129, 333])
@pytest.mark.parametrize("mask", ["none", "causal", "bool", "additive"])
def test_tensor_core_path_small_head_dims(dtype, D, N, mask):
    w = synth.small(dtype, 2, 3, N, D, mask, seed=N + D + len(mask))
    compare_full(w, expect_path=1)


@pytest.mark.parametrize("D", [16, 32])
@pytest.mark.parametrize("Nq,Nk", [(100, 300), (300, 77)])
def test_tensor_core_path_small_head_dims_cross_lengths_and_outputs(D, Nq, Nk):
    # unequal lengths, and outputs written through a wider buffer: columns
    # beyond D must stay untouched (the kernel computes 64 columns and its
    # stores drop the rest)
    w = synth.small("bf16", 2, 2, Nq, D, "causal", seed=Nq + Nk + D, Nk=Nk)
    compare_full(w, expect_path=1)
    inp = synth.make_inputs(w)
    g = [x.cuda() for x in (inp.q, inp.k, inp.v, inp.dq, inp.dk, inp.dv)]
    ref_o, ref_t = A.fwd_dual(*g, is_causal=True)
    wide = [torch.full((2, 2, Nq, 64), 7.0, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    A.fwd_dual(*g, is_causal=True, out=(wide[0][..., :D], wide[1][..., :D]))
    torch.cuda.synchronize()
    assert A.last_path() in A.TENSOR_CORE_PATHS
    assert torch.equal(wide[0][..., :D], ref_o) and torch.equal(wide[1][..., :D], ref_t)
    assert torch.all(wide[0][..., D:] == 7.0) and torch.all(wide[1][..., D:] == 7.0)


def test_nondefault_scale():
    compare_full(synth.small("bf16", 1, 2, 150, 64, "none", seed=3), scale=0.05, expect_path=1)
    compare_full(synth.small("f32", 1, 2, 40, 16, "none", seed=3), scale=0.9, expect_path=2)


@pytest.mark.parametrize("dtype,D", [("bf16", 64), ("f16", 128), ("bf16", 32)])
@pytest.mark.parametrize("mask", ["none", "causal", "bool", "additive"])
def test_negative_scale_on_the_tensor_core_path(dtype, D, mask):
    # The score products are formed negated (the MMA's negate-A bit) with
    # |scale| applied after them; the result is the oracle's at scale < 0.
    w = synth.small(dtype, 2, 2, 257, D, mask, seed=D + 41)
    compare_full(w, scale=-0.11, expect_path=1)


def test_negative_scale_split_kv_and_zero_scale():
    # A key split merges partial states formed with the negated scores; a zero
    # scale (uniform weights) runs the CUDA-core kernel.
    w = synth.small("bf16", 1, 1, 64, 64, "none", seed=5, Nk=8192)
    inp = synth.make_inputs(w)
    g = [x.cuda() for x in (inp.q, inp.k, inp.v, inp.dq, inp.dk, inp.dv)]
    o, t_o = A.fwd_dual(*g, scale=-0.09)
    assert A.last_path() == 3
    ro, rt, _, _ = oracle.fwd_dual(*(np64(x) for x in (inp.q, inp.k, inp.v, inp.dq, inp.dk,
                                                        inp.dv)), "none", None, scale=-0.09)
    assert np.abs(np64(o) - ro).max() <= TOL["bf16"] and np.abs(np64(t_o) - rt).max() <= TOL["bf16"]
    compare_full(synth.small("bf16", 1, 2, 100, 64, "causal", seed=6), scale=0.0, expect_path=2)


def test_fully_masked_rows_follow_the_convention():
    w = synth.small("bf16", 1, 2, 96, 64, "bool", seed=11)
    inp = synth.make_inputs(w)
    inp.mask[:, :, 5, :] = False
    inp.mask[:, :, 70, :] = False
    o, t_o, lse, mu, _ = run_gpu(w, inp)
    assert torch.all(o[:, :, 5] == 0) and torch.all(t_o[:, :, 70] == 0)
    assert torch.all(lse[:, :, 5] == -math.inf) and torch.all(mu[:, :, 70] == 0)


# ------------------------------------------------------------------ exactness
def test_boolean_masking_is_exact_in_which_keys_contribute():
    w = synth.small("bf16", 1, 2, 200, 128, "bool", seed=21)
    inp = synth.make_inputs(w)
    inp.mask[..., 37] = False
    inp.mask[..., 150] = False
    base = run_gpu(w, inp)
    for t in (inp.k, inp.v, inp.dk, inp.dv):
        t[:, :, 37] += 3.0
        t[:, :, 150] -= 5.0
    pert = run_gpu(w, inp)
    for a, b in zip(base[:4], pert[:4]):
        assert torch.equal(a, b)


def test_causal_masking_is_exact_in_which_keys_contribute():
    w = synth.small("f16", 1, 2, 256, 64, "causal", seed=22)
    inp = synth.make_inputs(w)
    base = run_gpu(w, inp)
    for t in (inp.k, inp.v, inp.dk, inp.dv):
        t[:, :, 200:] += 2.0
    pert = run_gpu(w, inp)
    for a, b in zip(base[:2], pert[:2]):
        assert torch.equal(a[:, :, :200], b[:, :, :200])
    assert torch.equal(base[2][:, :, :200], pert[2][:, :, :200])


def test_keys_beyond_the_sequence_are_never_read():
    # K/V views over a longer buffer: data past Nk must not influence anything.
    w = synth.small("bf16", 1, 2, 100, 64, "none", seed=23)
    inp = synth.make_inputs(w)
    dev = "cuda"
    big = [torch.randn(1, 2, 192, 64, dtype=torch.bfloat16, device=dev) for _ in range(4)]
    for bt, t in zip(big, (inp.k, inp.v, inp.dk, inp.dv)):
        bt[:, :, :100] = t.to(dev)
    q, dq = inp.q.to(dev), inp.dq.to(dev)
    views = [bt[:, :, :100] for bt in big]
    r1 = A.fwd_dual(q, views[0], views[1], dq, views[2], views[3], return_stats=True)
    for bt in big:
        bt[:, :, 100:] = 1e4
    r2 = A.fwd_dual(q, views[0], views[1], dq, views[2], views[3], return_stats=True)
    torch.cuda.synchronize()
    for a, b in zip(r1, r2):
        assert torch.equal(a, b)


def test_zero_tangents_give_exactly_zero_and_dv_only_matches_forward_of_dv():
    w = synth.small("bf16", 2, 2, 300, 128, "none", seed=24)
    inp = synth.make_inputs(w)
    dev = "cuda"
    q, k, v, dv = (x.to(dev) for x in (inp.q, inp.k, inp.v, inp.dv))
    z = torch.zeros_like(q)
    o, t_o, lse, mu = A.fwd_dual(q, k, v, z, z, torch.zeros_like(v), return_stats=True)
    assert torch.all(t_o == 0) and torch.all(mu == 0)
    o2, t_o2 = A.fwd_dual(q, k, v, z, z, dv)
    o_dv = A.attention(q, k, dv)
    torch.cuda.synchronize()
    assert torch.equal(o, o2)
    assert (t_o2.float() - o_dv.float()).abs().max().item() <= 1e-2


def test_forward_only_entry_point_matches_oracle():
    for dt, D, mask in (("bf16", 128, "causal"), ("f16", 64, "additive"), ("f32", 16, "bool")):
        w = synth.small(dt, 2, 2, 130, D, mask, seed=25)
        inp = synth.make_inputs(w)
        dev = "cuda"
        m = inp.mask.to(dev) if inp.mask is not None else None
        o, lse = A.attention(inp.q.to(dev), inp.k.to(dev), inp.v.to(dev), attn_mask=m,
                             is_causal=(mask == "causal"), return_lse=True)
        torch.cuda.synchronize()
        kind, mm = mask_for_oracle(w, inp)
        ro, _, rl, _ = oracle.fwd_dual(np64(inp.q), np64(inp.k), np64(inp.v), mask_kind=kind,
                                       mask=mm)
        assert np.abs(np64(o) - ro).max() <= TOL[dt]
        assert np.abs(np64(lse) - rl).max() <= LSE_TOL[dt]


def test_strided_inputs_from_a_bnhd_layout():
    # q/k/v as [B, N, H, D] buffers viewed as [B, H, N, D] (non-contiguous heads).
    w = synth.small("bf16", 2, 4, 140, 64, "none", seed=26)
    inp = synth.make_inputs(w)
    dev = "cuda"
    g = [x.to(dev).transpose(1, 2).contiguous().transpose(1, 2)
         for x in (inp.q, inp.k, inp.v, inp.dq, inp.dk, inp.dv)]
    o, t_o = A.fwd_dual(*g)
    torch.cuda.synchronize()
    assert A.last_path() in A.TENSOR_CORE_PATHS
    ro, rt, _, _ = oracle.fwd_dual(*(np64(x) for x in (inp.q, inp.k, inp.v, inp.dq, inp.dk,
                                                        inp.dv)))
    assert np.abs(np64(o) - ro).max() <= 2e-2 and np.abs(np64(t_o) - rt).max() <= 2e-2


@pytest.mark.parametrize("variant,D", [("tc", 64), ("tc", 128), ("split", 64), ("split", 128),
                                       ("simt", 40), ("simt", 128)])
@pytest.mark.parametrize("causal", [False, True])
def test_strided_and_offset_outputs(variant, D, causal):
    # O and tO written through views: a [B, N, H, D] buffer seen as [B, H, N, D],
    # and the first D columns of a [B, H, N, 2D] buffer (rows 2D apart).  The
    # results must be bit-identical to contiguous outputs, and the memory
    # around the views untouched.  140 query rows: the last query tile is
    # ragged.  Every writer of O and tO is covered: the tensor-core epilogue
    # (TMA stores), the split-KV merge kernel and the CUDA-core kernel.
    if variant == "tc":
        w, split, path = synth.small("bf16", 2, 4, 140, D, "none", seed=27 + D), False, 1
    elif variant == "split":  # 2100 keys over few query tiles: the key range is split
        w, split, path = synth.small("bf16", 1, 2, 140, D, "none", seed=28 + D, Nk=2100), True, 3
    else:  # float32 takes the CUDA-core kernel at any D
        w, split, path = synth.small("f32", 2, 4, 140, D, "none", seed=29 + D), False, 2
    inp = synth.make_inputs(w)
    dev = "cuda"
    g = [x.to(dev) for x in (inp.q, inp.k, inp.v, inp.dq, inp.dk, inp.dv)]
    ref_o, ref_t = A.fwd_dual(*g, is_causal=causal, split_kv=split)
    assert A.last_path() == path
    B, H, N, dt = w.B, w.H, w.N, w.torch_dtype
    bnhd = [torch.full((B, N, H, D), 7.0, dtype=dt, device=dev) for _ in range(2)]
    wide = [torch.full((B, H, N, 2 * D), 7.0, dtype=dt, device=dev) for _ in range(2)]
    for bufs, view in ((bnhd, lambda t: t.transpose(1, 2)), (wide, lambda t: t[..., :D])):
        o, t_o = view(bufs[0]), view(bufs[1])
        A.fwd_dual(*g, is_causal=causal, out=(o, t_o), split_kv=split)
        torch.cuda.synchronize()
        assert A.last_path() == path
        assert torch.equal(o, ref_o) and torch.equal(t_o, ref_t)
        if bufs is wide:
            for t in bufs:
                assert torch.all(t[..., D:] == 7.0)
    kind = "causal" if causal else "none"
    ro, rt, _, _ = oracle.fwd_dual(*(np64(x) for x in (inp.q, inp.k, inp.v, inp.dq, inp.dk,
                                                        inp.dv)), kind, None)
    tol = TOL[w.dtype]
    assert np.abs(np64(ref_o) - ro).max() <= tol and np.abs(np64(ref_t) - rt).max() <= tol


# ------------------------------------------------------------------ specified workloads
def test_workload_f32_b1h2n32d16_full():
    compare_full(synth.WORKLOADS["f32_b1h2n32d16"], expect_path=2)


def sampled_rows(w, inp, o, t_o, lse, n_rows, seed=0):
    rng = np.random.default_rng(seed)
    total = w.B * w.H * w.N
    rows = np.unique(np.concatenate([rng.integers(0, total, n_rows),
                                     [0, w.N - 1, total - 1, total - w.N]]))
    kind, m = mask_for_oracle(w, inp)
    ro, rt, rl, _ = oracle.fwd_dual_rows(np64(inp.q), np64(inp.k), np64(inp.v), np64(inp.dq),
                                         np64(inp.dk), np64(inp.dv), rows, kind, m)
    D = w.D
    go = np64(o).reshape(-1, D)[rows]
    gt = np64(t_o).reshape(-1, D)[rows]
    gl = np64(lse).reshape(-1)[rows]
    return np.abs(go - ro).max(), np.abs(gt - rt).max(), np.abs(gl - rl).max()


@pytest.mark.parametrize("name", ["f16_b2h8n512d64", "f16_b2h8n512d64_causal",
                                  "bf16_b2h8n1024d64_bool", "bf16_b2h8n1024d64_additive",
                                  "bf16_b4h16n2048d128", "bf16_b4h16n2048d128_causal",
                                  "f16_b2h8n2048d64_causal"])
def test_specified_workloads_every_element(name):
    # The full-size launch (the configuration the benchmark times) against the
    # oracle on every element of O, tO, lse and mu.
    w = synth.WORKLOADS[name]
    # (a NaN anywhere on the GPU side makes the max-abs difference NaN, which fails)
    compare_full(w, expect_path=1)


def test_device_timeout_is_reported_and_the_context_survives():
    st = A._abi.load().jvp_attn_selftest_wait_timeout(200000, None)
    assert st == 0
    assert A.device_status(torch.cuda.default_stream()) == A._abi.JVP_ERR_DEVICE_TIMEOUT
    assert A.device_status(torch.cuda.default_stream()) == 0
    compare_full(synth.small("bf16", 1, 1, 64, 64, "none", seed=1), expect_path=1)


def test_host_pipeline_matches_device_call():
    # fwd_dual_host splits batch*heads into chunks and overlaps copies with compute;
    # every (b, h) problem is computed by the same kernel, so results are bit-identical.
    w = synth.small("bf16", 3, 5, 200, 128, "causal", seed=27)
    inp = synth.make_inputs(w)
    host = [x.pin_memory() for x in (inp.q, inp.k, inp.v, inp.dq, inp.dk, inp.dv)]
    o_h, t_h = A.fwd_dual_host(*host, is_causal=True, chunks=4)
    torch.cuda.synchronize()
    o_d, t_d = A.fwd_dual(*[x.cuda() for x in host], is_causal=True, split_kv=False)
    torch.cuda.synchronize()
    assert torch.equal(o_h, o_d.cpu()) and torch.equal(t_h, t_d.cpu())


# ------------------------------------------------------------------ split-KV
@pytest.mark.parametrize("dtype,D", [("bf16", 64), ("f16", 128)])
@pytest.mark.parametrize("mask", ["none", "causal", "bool", "additive"])
@pytest.mark.parametrize("B,H,Nq,Nk", [(1, 2, 300, 4096), (1, 1, 100, 3000), (2, 1, 257, 2500),
                                        (1, 1, 64, 20000)])
def test_split_kv_matches_oracle_and_the_single_pass(dtype, D, mask, B, H, Nq, Nk):
    # Few query tiles, many keys: the key range is split over several CTAs and
    # the partial states are merged by a second kernel.
    w = synth.small(dtype, B, H, Nq, D, mask, seed=Nq + Nk + D, Nk=Nk)
    assert A.fwd_dual_workspace_size(B, H, Nq, Nk, D, w.torch_dtype) > 0
    inp = synth.make_inputs(w)
    o, t_o, lse, mu, path = run_gpu(w, inp)
    assert path == 3
    kind, m = mask_for_oracle(w, inp)
    ro, rt, rl, rm = oracle.fwd_dual(np64(inp.q), np64(inp.k), np64(inp.v), np64(inp.dq),
                                     np64(inp.dk), np64(inp.dv), kind, m)
    tol = TOL[w.dtype]
    eo, et = np.abs(np64(o) - ro).max(), np.abs(np64(t_o) - rt).max()
    fin = np.isfinite(rl)
    assert np.array_equal(np.isfinite(np64(lse)), fin)
    el = np.abs(np64(lse)[fin] - rl[fin]).max()
    log_error(w.name + "[split-kv]", o=eo, t_o=et, lse=el)
    assert eo <= tol and et <= tol, (w.name, eo, et)
    assert el <= LSE_TOL[w.dtype]
    assert np.abs(np64(mu) - rm).max() <= 20 * tol
    # the single-pass kernel on the same inputs agrees to rounding
    dev = "cuda"
    g = [x.to(dev) for x in (inp.q, inp.k, inp.v, inp.dq, inp.dk, inp.dv)]
    mm = inp.mask.to(dev) if inp.mask is not None else None
    o1, t1 = A.fwd_dual(*g, attn_mask=mm, is_causal=(mask == "causal"), split_kv=False)
    assert A.last_path() in (1, 4)
    torch.cuda.synchronize()
    assert (o1.float() - o.float()).abs().max().item() <= tol
    assert (t1.float() - t_o.float()).abs().max().item() <= tol


def test_split_kv_fully_masked_rows_and_empty_ranges():
    # Rows whose every key is masked, and causal rows whose later key ranges
    # are empty, follow the single-pass convention (O = tO = 0, lse = -inf).
    w = synth.small("bf16", 1, 2, 300, 64, "bool", seed=41, Nk=2100)
    inp = synth.make_inputs(w)
    inp.mask[:, :, 5] = False
    inp.mask[:, :, 290, :] = False
    o, t_o, lse, mu, path = run_gpu(w, inp)
    assert path == 3
    for x in (o, t_o):
        assert torch.all(x[:, :, 5] == 0) and torch.all(x[:, :, 290] == 0)
    assert torch.all(lse[:, :, 5] == -float("inf")) and torch.all(mu[:, :, 5] == 0)
    kind, m = mask_for_oracle(w, inp)
    ro, rt, _, _ = oracle.fwd_dual(np64(inp.q), np64(inp.k), np64(inp.v), np64(inp.dq),
                                   np64(inp.dk), np64(inp.dv), kind, m)
    assert np.abs(np64(o) - ro).max() <= TOL["bf16"]
    assert np.abs(np64(t_o) - rt).max() <= TOL["bf16"]


@pytest.mark.parametrize("dtype,D,mask,chunks", [("bf16", 128, "causal", 3), ("f16", 64, "bool", 5),
                                                 ("bf16", 64, "additive", 1),
                                                 ("f32", 40, "none", 4), ("bf16", 64, "none", 64)])
def test_host_buffer_entry_point_matches_oracle(dtype, D, mask, chunks):
    # jvp_attn_fwd_dual_host: host tensors in and out, copies pipelined over
    # `chunks` groups of (batch, head) pairs (more groups than pairs is allowed).
    w = synth.small(dtype, 3, 5, 150, D, mask, seed=70 + D)
    inp = synth.make_inputs(w)
    if inp.mask is not None:
        inp.mask = inp.mask[:1]  # one mask shared by every (batch, head)
    host = [x.pin_memory() for x in (inp.q, inp.k, inp.v, inp.dq, inp.dk, inp.dv)]
    o, t_o, lse, mu = A.fwd_dual_host(*host, attn_mask=inp.mask, is_causal=(mask == "causal"),
                                      chunks=chunks, return_stats=True)
    torch.cuda.synchronize()
    assert o.device.type == "cpu" and lse.device.type == "cpu"
    assert A.last_path() in ((2,) if dtype == "f32" else (1, 4))
    m = None
    if mask == "bool":
        m = np.broadcast_to(inp.mask.numpy(), (3, 1, 150, 150))
    elif mask == "additive":
        m = np.broadcast_to(inp.mask.double().numpy(), (3, 1, 150, 150))
    ro, rt, rl, rm = oracle.fwd_dual(*(np64(x) for x in host), mask, m)
    tol = TOL[dtype]
    assert np.abs(np64(o) - ro).max() <= tol
    assert np.abs(np64(t_o) - rt).max() <= tol
    assert np.abs(np64(lse) - rl).max() <= LSE_TOL[dtype]
    assert np.abs(np64(mu) - rm).max() <= 20 * tol



@pytest.mark.parametrize("dtype,D", [("bf16", 64), ("f16", 64), ("bf16", 128)])
@pytest.mark.parametrize("mask", ["none", "causal", "bool", "additive"])
def test_repeated_calls_are_bit_identical(dtype, D, mask):
    # Every kernel fixes its arithmetic order, so the same inputs must give the
    # same bits on every call; a data race between warps (e.g. one warpgroup
    # overwriting TMEM columns the other has not read yet) shows up here as a
    # call-to-call difference.
    w = synth.small(dtype, 2, 2, 320, D, mask, seed=90 + D)
    inp = synth.make_inputs(w, with_cotangents=True)
    dev = "cuda"
    g = [x.to(dev) for x in (inp.q, inp.k, inp.v, inp.dq, inp.dk, inp.dv)]
    m = inp.mask.to(dev) if inp.mask is not None else None
    causal = mask == "causal"
    runs = [A.fwd_dual(*g, attn_mask=m, is_causal=causal, return_stats=True) for _ in range(8)]
    o, t_o, lse, mu = runs[0]
    bwd = [A.bwd_dual(*g, o, t_o, lse, mu, inp.g_o.to(dev), inp.g_to.to(dev), attn_mask=m,
                      is_causal=causal) for _ in range(4)]
    torch.cuda.synchronize()
    for r in runs[1:]:
        for a, b in zip(runs[0], r):
            assert torch.equal(a, b)
    for r in bwd[1:]:
        for a, b in zip(bwd[0], r):
            assert torch.equal(a, b)


def test_split_kv_repeated_calls_are_bit_identical():
    w = synth.small("bf16", 1, 2, 200, 64, "additive", seed=93, Nk=4000)
    inp = synth.make_inputs(w)
    g = [x.cuda() for x in (inp.q, inp.k, inp.v, inp.dq, inp.dk, inp.dv)]
    m = inp.mask.cuda()
    runs = [A.fwd_dual(*g, attn_mask=m, return_stats=True) for _ in range(6)]
    assert A.last_path() == 3
    torch.cuda.synchronize()
    for r in runs[1:]:
        for a, b in zip(runs[0], r):
            assert torch.equal(a, b)


@pytest.mark.parametrize("dtype,D,mask,B,H,Nq,Nk", [
    ("bf16", 128, "causal", 1, 2, 16384, 16384),   # long causal rows
    ("f16", 64, "none", 1, 1, 256, 65536),          # long key range: 16-way split-KV
    ("bf16", 64, "bool", 1, 2, 8192, 8192),
    ("bf16", 128, "causal", 1, 1, 131072, 131072),  # one very long causal head
    ("f16", 64, "none", 8, 64, 1024, 1024),         # 4096 CTAs (512 heads x 8 tiles)
])
def test_long_sequences_on_sampled_rows(dtype, D, mask, B, H, Nq, Nk):
    w = synth.small(dtype, B, H, Nq, D, mask, seed=Nq // 64 + D, Nk=Nk)
    inp = synth.make_inputs(w)
    o, t_o, lse, mu, path = run_gpu(w, inp)
    assert path in A.TENSOR_CORE_PATHS
    eo, et, el = sampled_rows(w, inp, o, t_o, lse, 64)
    log_error(w.name + "[long]", o=eo, t_o=et, lse=el)
    assert eo <= TOL[dtype] and et <= TOL[dtype], (w.name, eo, et)
    assert el <= LSE_TOL[dtype]
    assert torch.isfinite(o).all() and torch.isfinite(t_o).all()


# ------------------------------------------------------------------ cluster key split
@pytest.mark.parametrize("dtype,D", [("bf16", 64), ("f16", 64), ("bf16", 32), ("f16", 16)])
@pytest.mark.parametrize("mask", ["none", "causal", "bool", "additive"])
@pytest.mark.parametrize("B,H,Nq,Nk", [(2, 8, 512, 1024), (1, 3, 300, 1100), (1, 2, 129, 1000),
                                       (2, 1, 700, 1030), (1, 2, 50, 1000), (1, 4, 1024, 1024)])
def test_cluster_split_matches_oracle_and_the_single_pass(dtype, D, mask, B, H, Nq, Nk):
    # Small problems at D <= 64 split each query tile's key range between the
    # two CTAs of a cluster; rank 1's partial state reaches rank 0 through
    # distributed shared memory.  Against the oracle, and against the single
    # pass on the same inputs (equal up to the rounding order of the merge).
    w = synth.small(dtype, B, H, Nq, D, mask, seed=Nq + Nk + D + len(mask), Nk=Nk)
    compare_full(w, expect_path=4)
    inp = synth.make_inputs(w)
    g = [x.cuda() for x in (inp.q, inp.k, inp.v, inp.dq, inp.dk, inp.dv)]
    m = inp.mask.cuda() if inp.mask is not None else None
    causal = mask == "causal"
    o4, t4, l4, mu4 = A.fwd_dual(*g, attn_mask=m, is_causal=causal, return_stats=True)
    assert A.last_path() == 4
    A.set_cluster_split(False)
    try:
        o1, t1, l1, mu1 = A.fwd_dual(*g, attn_mask=m, is_causal=causal, return_stats=True)
        assert A.last_path() == 1
    finally:
        A.set_cluster_split(True)
    torch.cuda.synchronize()
    tol = TOL[w.dtype]
    assert (o4.float() - o1.float()).abs().max().item() <= tol
    assert (t4.float() - t1.float()).abs().max().item() <= tol
    fin = torch.isfinite(l1)
    assert torch.equal(fin, torch.isfinite(l4))
    assert (l4[fin] - l1[fin]).abs().max().item() <= 1e-4


def test_cluster_split_repeated_calls_and_exactness():
    # bit-identical repeats (every CTA's arithmetic order is fixed); keys that
    # no row keeps never reach the outputs, whichever CTA of the pair owns them.
    w = synth.small("bf16", 1, 2, 300, 64, "bool", seed=61, Nk=1200)
    inp = synth.make_inputs(w)
    inp.mask[..., 37] = False   # in rank 0's key range
    inp.mask[..., 900] = False  # in rank 1's
    base = run_gpu(w, inp)
    assert base[4] == 4
    for _ in range(4):
        again = run_gpu(w, inp)
        for a, b in zip(base[:4], again[:4]):
            assert torch.equal(a, b)
    for t in (inp.k, inp.v, inp.dk, inp.dv):
        t[:, :, 37] += 3.0
        t[:, :, 900] -= 5.0
    pert = run_gpu(w, inp)
    for a, b in zip(base[:4], pert[:4]):
        assert torch.equal(a, b)
    # causal rows see keys j <= i < 400 only: each query tile's short key
    # range is split at its own midpoint (the (1, 2, 50, 1000) causal case of
    # the test above leaves rank 1 an empty range)
    w = synth.small("f16", 1, 2, 400, 64, "causal", seed=62, Nk=1100)
    compare_full(w, expect_path=4)
