"""The backward's second stream: the key-major kernels run on a stream the
library owns, forked from the caller's stream after the row pass and joined
back before the call returns.  Work the caller enqueues on its own stream
right after the call must see every gradient; a CUDA-graph capture of the
call records the fork and the join.  (The no-allocation entry point, which
uses one stream, is compared bit for bit with the forked path in
test_zz_no_alloc.py.)
"""

import pytest
import torch

from forward_mode_flash_gb300 import api as A
from forward_mode_flash_gb300 import build, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def inputs(dtype, D, mask, N=1024, B=2, H=4):
    w = synth.small(dtype, B, H, N, D, mask, seed=D + N)
    inp = synth.make_inputs(w, with_cotangents=True, device="cuda")
    g = [inp.q, inp.k, inp.v, inp.dq, inp.dk, inp.dv]
    causal = mask == "causal"
    o, t_o, lse, mu = A.fwd_dual(*g, attn_mask=inp.mask, is_causal=causal, return_stats=True)
    return inp, g, (o, t_o, lse, mu), causal


@pytest.mark.parametrize("dtype,D,mask", [("bf16", 64, "causal"), ("f16", 128, "none"),
                                          ("bf16", 128, "bool")])
def test_outputs_are_ready_on_the_callers_stream(dtype, D, mask):
    inp, g, (o, t_o, lse, mu), causal = inputs(dtype, D, mask)
    torch.cuda.synchronize()
    ref = A.bwd_dual(*g, o, t_o, lse, mu, inp.g_o, inp.g_to, attn_mask=inp.mask, is_causal=causal)
    ref_p = A.bwd(*g[:3], o, lse, inp.g_o, attn_mask=inp.mask, is_causal=causal)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(3):  # back to back on one non-default stream
            grads = A.bwd_dual(*g, o, t_o, lse, mu, inp.g_o, inp.g_to, attn_mask=inp.mask,
                               is_causal=causal)
            snap = [x.clone() for x in grads]  # enqueued on s right after the call
            grads_p = A.bwd(*g[:3], o, lse, inp.g_o, attn_mask=inp.mask, is_causal=causal)
            snap_p = [x.clone() for x in grads_p]
    torch.cuda.synchronize()
    assert A.device_status() == 0
    for a, b in zip(snap + snap_p, list(ref) + list(ref_p)):
        assert torch.equal(a, b)


@pytest.mark.parametrize("dtype,D", [("bf16", 64), ("f16", 128)])
def test_backward_in_a_cuda_graph_matches_eager(dtype, D):
    inp, g, (o, t_o, lse, mu), causal = inputs(dtype, D, "none", N=512)
    ws = torch.empty(A.bwd_dual_workspace_size(2, 4, 512, 512, D), dtype=torch.uint8,
                     device="cuda")
    args = (*g, o, t_o, lse, mu, inp.g_o, inp.g_to)
    eager = A.bwd_dual(*args, workspace=ws)  # also sets the kernels' attributes before capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        captured = A.bwd_dual(*args, workspace=ws)
    for x in captured:
        x.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert A.device_status() == 0
    for a, b in zip(captured, eager):
        assert torch.equal(a, b)
