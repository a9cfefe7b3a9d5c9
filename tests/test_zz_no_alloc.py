"""jvp_attn_bwd_dual_noalloc: the backward for callers that cannot allocate
device memory (it keeps its scratch in a fixed device array of the library).

The GPU test calls the entry point through the C ABI, twice in a row on two
different problems, and checks each result against the ordinary
jvp_attn_bwd_dual (with a caller workspace) within the backward tests'
tolerance.  This file is collected last on purpose.
"""

import ctypes

import pytest
import torch

from forward_mode_flash_gb300 import _abi, api, build, synth

TOL = {"f32": 1e-4, "f16": 2e-2, "bf16": 2e-2}


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


@pytest.mark.gpu
def test_noalloc_matches_the_workspace_entry_point_on_two_calls():
    build.build()
    cases = [synth.small("bf16", 2, 4, 300, 64, "causal", seed=31),
             synth.small("f32", 1, 3, 77, 40, "none", seed=32)]
    for w in cases:  # two calls in a row; the second reuses the scratch the first left
        inp = synth.make_inputs(w, with_cotangents=True)
        g = [x.cuda() for x in (inp.q, inp.k, inp.v, inp.dq, inp.dk, inp.dv)]
        causal = w.mask == "causal"
        o, t_o, lse, mu = api.fwd_dual(*g, is_causal=causal, return_stats=True)
        go, gto = inp.g_o.cuda(), inp.g_to.cuda()
        ref = api.bwd_dual(*g, o, t_o, lse, mu, go, gto, is_causal=causal)
        got = call_noalloc(*g, o, t_o, lse, mu, go, gto, causal)
        torch.cuda.synchronize()
        for r, x in zip(ref, got):
            scale = max(1.0, r.float().abs().max().item())
            assert (r.float() - x.float()).abs().max().item() <= TOL[w.dtype] * scale
    assert api.device_status() == 0
