"""jvp_attn_bwd_dual_noalloc: the backward for callers that cannot allocate
device memory (it keeps its scratch in a fixed device array of the library).

The GPU test calls the entry point through the C ABI several times in a row on
different problems (one of them needs exactly the whole fixed scratch), and
checks that each result is bit-identical to the ordinary jvp_attn_bwd_dual
with a caller workspace: both run the same kernels.  This file is collected
last on purpose.
"""

import ctypes

import pytest
import torch

from forward_mode_flash_gb300 import _abi, api, build, synth


def call_noalloc(q, k, v, dq, dk, dv, o, t_o, lse, mu, g_o, g_to, causal):
    """Marshal the arguments and call the C entry point directly."""
    lib = _abi.load()
    B, H, Nq, D = q.shape
    Nk = k.shape[2]
    outs = [torch.empty_like(x) for x in (q, k, v, dq, dk, dv)]
    mask, _ = api._mask_desc(None, causal, B, H, Nq, Nk, q.device)
    ins = (_abi.Strides * 10)(*[api._strides(t) for t in (q, k, v, dq, dk, dv, o, t_o, g_o, g_to)])
    ost = (_abi.Strides * 6)(*[api._strides(t) for t in outs])
    shape = _abi.Shape(B, H, Nq, Nk, D)
    stream = torch.cuda.current_stream().cuda_stream
    p = api._ptr
    st = lib.jvp_attn_bwd_dual_noalloc(ctypes.byref(shape), api._DT[q.dtype], p(q), p(k), p(v),
                                       p(dq), p(dk), p(dv), p(o), p(t_o), p(lse), p(mu), p(g_o),
                                       p(g_to), ins, ctypes.byref(mask), 1.0 / D ** 0.5,
                                       *[p(x) for x in outs], ost, ctypes.c_void_p(stream))
    _abi.check(st)
    return outs


def test_rejects_problems_beyond_the_fixed_scratch():
    build.build()
    lib = _abi.load()
    shape = _abi.Shape(8, 32, 4096, 4096, 64)  # 8 * B * H * Nq = 8 MiB > 4 MiB
    st = lib.jvp_attn_bwd_dual_noalloc(ctypes.byref(shape), _abi.JVP_BF16, *([None] * 12), None,
                                       None, 0.125, *([None] * 6), None, None)
    assert st == _abi.JVP_ERR_WORKSPACE
    assert b"4 MiB" in lib.jvp_attn_last_error()


def _case(w):
    inp = synth.make_inputs(w, with_cotangents=True)
    g = [x.cuda() for x in (inp.q, inp.k, inp.v, inp.dq, inp.dk, inp.dv)]
    causal = w.mask == "causal"
    o, t_o, lse, mu = api.fwd_dual(*g, is_causal=causal, return_stats=True)
    return g, o, t_o, lse, mu, inp.g_o.cuda(), inp.g_to.cuda(), causal


@pytest.mark.gpu
def test_noalloc_matches_the_workspace_entry_point_on_two_calls():
    build.build()
    # Both entry points run the same kernels in the same order, so the results
    # must be bit-identical; the workspace of the reference call is filled with
    # NaN first, so neither side can lean on scratch contents left behind.  It
    # has the base size (8 * B * H * Nq bytes), so the reference does not split
    # the key side (the fixed scratch holds no partial sums) either.
    B, H, Nq = 8, 16, 4096  # 8 * B * H * Nq == 4 MiB: exactly the fixed scratch
    assert 8 * B * H * Nq == _abi.JVP_BWD_NOALLOC_SCRATCH_BYTES
    cases = [(synth.small("bf16", 2, 4, 300, 64, "causal", seed=31), 1),
             (synth.small("f32", 1, 3, 77, 40, "none", seed=32), 2),
             (synth.small("f16", B, H, Nq, 64, "none", seed=33, Nk=128), 1),
             (synth.small("bf16", 1, 2, 130, 128, "causal", seed=34), 1)]
    for w, path in cases:  # calls in a row; each reuses the scratch the previous one left
        g, o, t_o, lse, mu, go, gto, causal = _case(w)
        ws = torch.full((2 * w.B * w.H * w.N,), float("nan"), dtype=torch.float32, device="cuda")
        ref = api.bwd_dual(*g, o, t_o, lse, mu, go, gto, is_causal=causal, workspace=ws)
        got = call_noalloc(*g, o, t_o, lse, mu, go, gto, causal)
        assert api.last_path() == path, (w.name, api.last_path())
        torch.cuda.synchronize()
        for r, x in zip(ref, got):
            assert torch.equal(r, x), w.name
    assert api.device_status() == 0
