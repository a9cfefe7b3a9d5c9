"""The debug build of the library: its tensor-core kernels bounds-check every
hand-computed TMEM column range, shared-memory offset and global row / column
index (a failure skips the access and is reported as JVP_ERR_BOUNDS by
jvp_attn_get_device_status).  Small parity cases over every kernel family run
on it here: the results must match the oracle as with the ordinary build, and
the device status must stay clean.
"""

import numpy as np
import pytest
import torch

import oracle
from forward_mode_flash_gb300 import _abi, api as A, build, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def debug_lib():
    path = build.build(debug=True)
    _abi.use_debug_build(path)
    lib = _abi.load()
    assert lib._name == path
    A.device_status()  # start from a clean status word
    yield lib
    _abi.use_debug_build(None)


def np64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def oracle_mask(w, inp):
    if w.mask == "bool":
        return inp.mask.numpy()
    if w.mask == "additive":
        return inp.mask.double().numpy()
    return None


FWD_CASES = [("bf16", 2, 2, 200, 128, "causal", None, 1), ("f16", 1, 3, 333, 64, "bool", None, 1),
             ("bf16", 2, 2, 130, 64, "additive", None, 1), ("bf16", 1, 2, 100, 32, "none", 300, 1),
             ("f16", 1, 2, 129, 16, "causal", None, 1), ("bf16", 1, 2, 300, 64, "none", 4096, 3),
             ("f16", 1, 2, 300, 128, "additive", 3000, 3), ("bf16", 1, 2, 129, 64, "causal", 1000, 4),
             ("f16", 1, 3, 300, 64, "bool", 1100, 4), ("f32", 1, 2, 45, 40, "bool", None, 2)]


@pytest.mark.parametrize("dtype,B,H,N,D,mask,Nk,path", FWD_CASES)
def test_forward_kernels_pass_their_bounds_checks(debug_lib, dtype, B, H, N, D, mask, Nk, path):
    w = synth.small(dtype, B, H, N, D, mask, seed=N + D, Nk=Nk)
    inp = synth.make_inputs(w)
    g = [x.cuda() for x in (inp.q, inp.k, inp.v, inp.dq, inp.dk, inp.dv)]
    m = inp.mask.cuda() if inp.mask is not None else None
    o, t_o, lse, mu = A.fwd_dual(*g, attn_mask=m, is_causal=(mask == "causal"), return_stats=True)
    assert A.last_path() == path
    assert A.device_status() == 0
    ro, rt, _, _ = oracle.fwd_dual(*(np64(x) for x in (inp.q, inp.k, inp.v, inp.dq, inp.dk,
                                                        inp.dv)), mask, oracle_mask(w, inp))
    tol = 1e-4 if dtype == "f32" else 2e-2
    assert np.abs(np64(o) - ro).max() <= tol and np.abs(np64(t_o) - rt).max() <= tol


@pytest.mark.parametrize("dtype,D,mask,N,Nk", [("bf16", 64, "causal", 130, None),
                                             ("f16", 128, "bool", 257, None),
                                             ("bf16", 128, "additive", 100, 300),
                                             ("f16", 32, "none", 70, None)])
def test_backward_kernels_pass_their_bounds_checks(debug_lib, dtype, D, mask, N, Nk):
    w = synth.small(dtype, 2, 2, N, D, mask, seed=N + D, Nk=Nk)
    inp = synth.make_inputs(w, with_cotangents=True)
    g = [x.cuda() for x in (inp.q, inp.k, inp.v, inp.dq, inp.dk, inp.dv)]
    m = inp.mask.cuda() if inp.mask is not None else None
    causal = mask == "causal"
    o, t_o, lse, mu = A.fwd_dual(*g, attn_mask=m, is_causal=causal, return_stats=True)
    grads = A.bwd_dual(*g, o, t_o, lse, mu, inp.g_o.cuda(), inp.g_to.cuda(), attn_mask=m,
                       is_causal=causal)
    assert A.last_path() == 1
    assert A.device_status() == 0
    ref = oracle.bwd_dual(*(np64(x) for x in (inp.q, inp.k, inp.v, inp.dq, inp.dk, inp.dv,
                                              inp.g_o, inp.g_to)), mask, oracle_mask(w, inp))
    for gg, r in zip(grads, ref):
        assert np.abs(np64(gg) - r).max() <= 2e-2 * max(1.0, np.abs(r).max())


def test_the_debug_library_reports_bounds_failures_as_their_own_status(debug_lib):
    # The status code and its message exist (no kernel is made to fail here).
    assert debug_lib.jvp_attn_status_string(_abi.JVP_ERR_BOUNDS).startswith(b"device-side bounds")
