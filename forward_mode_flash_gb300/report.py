"""Sequence-length sweep and memory-scaling report of the fused dual attention.

Both follow the benchmark summary of the "JVP Flash Attention" project page
(the tables of Time / Mem / TFLOP/s against sequence length, causal flag and
mask kind, at B*H*D = 1024): here B=2, H=8, D=64, N from 32 to 2048, every mask
kind, fp16 and bf16.

* ``sweep`` times one ``fwd_dual`` call per configuration with CUDA events on
  the launching stream: hot L2 (inputs already cached), cold L2 (a 256 MiB
  buffer written between calls, outside the events) and, for N <= 512, a CUDA
  graph of 100 calls replayed as one (launch overhead stripped; labelled).
  Throughput is reported against both roofs: TFLOP/s (12 B H N^2 D, halved
  for causal) and GB/s of the algorithmic bytes (each input read once, each
  output written once, the mask once).
* ``memory_scaling`` measures, with the caching allocator's peak counter, the
  device bytes that one call adds on top of its inputs: for ``fwd_dual`` (the
  outputs O, tO, lse, mu; the kernels allocate nothing), for ``bwd_dual`` (six
  gradients and its workspace: 8 B H N bytes, plus the key-major split's
  partial sums, O(Nk), when few CTAs would run the key side) and for one reverse-over-forward
  step through ``JVPAttn.fwd_dual`` (the second-order use the page measures:
  saved tensors, gradients, workspace).  Every term is O(N); nothing N x N is
  ever stored.
"""

from __future__ import annotations

import statistics
from typing import Iterator

import torch

from . import api, metrics, synth
from .autograd import JVPAttn

SWEEP_N = (32, 64, 128, 256, 512, 1024, 2048)
SWEEP_MASKS = ("none", "causal", "bool", "additive")
L2_FLUSH_BYTES = 256 << 20


def _inputs(dtype: str, B: int, H: int, N: int, D: int, mask: str, seed: int = 0,
            cotangents: bool = False):
    w = synth.small(dtype, B, H, N, D, mask, seed=seed)
    return w, synth.make_inputs(w, with_cotangents=cotangents, device="cuda")


def _events_ms(fn, reps: int, flush=None) -> float:
    """Median per-call time; the calls are queued back to back (one sync at the end)."""
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(reps)]
    for r, (a, b) in enumerate(ev):
        if flush is not None:
            flush.fill_(float(r))
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in ev)


def _graph_ms(fn, batch: int = 100, reps: int = 5) -> float:
    """Per-call time of a CUDA graph holding ``batch`` calls."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(3):
            fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(batch):
            fn()
    g.replay()
    torch.cuda.synchronize()
    return _events_ms(g.replay, reps) / batch


def sweep(dtypes=("bf16", "f16"), Ns=SWEEP_N, masks=SWEEP_MASKS, B: int = 2, H: int = 8,
          D: int = 64, peak_tflops: float = 1900.0, peak_gbs: float = 6800.0,
          graph_max_n: int = 512) -> Iterator[dict]:
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    for dtype in dtypes:
        for N in Ns:
            for mask in masks:
                _, inp = _inputs(dtype, B, H, N, D, mask)
                causal = mask == "causal"
                args = (inp.q, inp.k, inp.v, inp.dq, inp.dk, inp.dv)
                o = torch.empty_like(inp.q)
                t_o = torch.empty_like(inp.q)
                lse = torch.empty(B, H, N, dtype=torch.float32, device="cuda")
                mu = torch.empty_like(lse)

                def call():
                    api.fwd_dual(*args, attn_mask=inp.mask, is_causal=causal,
                                 out=(o, t_o, lse, mu))

                for _ in range(5):
                    call()
                torch.cuda.synchronize()
                reps = 200 if N <= 256 else 50
                hot = _events_ms(call, reps)
                cold = _events_ms(call, max(20, reps // 4), flush)
                graph = _graph_ms(call) if N <= graph_max_n else None
                fl = metrics.flops_fwd_dual(B, H, N, N, D, causal)
                by = metrics.bytes_fwd_dual(B, H, N, N, D, inp.q.element_size(), mask,
                                            mask_batch=B)
                best = min(t for t in (hot, graph) if t is not None)
                yield {"dtype": dtype, "N": N, "mask": mask, "B": B, "H": H, "D": D,
                       "path": {1: "tensor-core", 3: "tensor-core split-KV",
                                4: "tensor-core cluster split"}.get(api.last_path(), "cuda-core"),
                       "ms_hot": hot, "ms_cold_l2": cold, "ms_graph_batch100": graph,
                       "tflops_hot": fl / hot / 1e9, "tflops_cold_l2": fl / cold / 1e9,
                       "tflops_graph": None if graph is None else fl / graph / 1e9,
                       "gbs_best": by / best / 1e6, "frac_tensor_best": fl / best / 1e9 / peak_tflops,
                       "frac_hbm_best": by / best / 1e6 / peak_gbs,
                       "flops": fl, "alg_bytes": by}
                del inp
    del flush


def _peak_added(fn) -> int:
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    base = torch.cuda.memory_allocated()
    out = fn()
    torch.cuda.synchronize()
    peak = torch.cuda.max_memory_allocated() - base
    del out
    return peak


def memory_scaling(Ns=SWEEP_N + (4096, 8192, 16384), dtype: str = "bf16", B: int = 2,
                   H: int = 8, D: int = 64, mask: str = "none") -> Iterator[dict]:
    for N in Ns:
        _, inp = _inputs(dtype, B, H, N, D, mask, cotangents=True)
        causal = mask == "causal"
        prim = (inp.q, inp.k, inp.v, inp.dq, inp.dk, inp.dv)
        in_bytes = sum(t.numel() * t.element_size() for t in prim)
        if inp.mask is not None:
            in_bytes += inp.mask.numel() * inp.mask.element_size()
        fwd = _peak_added(lambda: api.fwd_dual(*prim, attn_mask=inp.mask, is_causal=causal,
                                               return_stats=True))
        o, t_o, lse, mu = api.fwd_dual(*prim, attn_mask=inp.mask, is_causal=causal,
                                       return_stats=True)
        bwd = _peak_added(lambda: api.bwd_dual(*prim, o, t_o, lse, mu, inp.g_o, inp.g_to,
                                               attn_mask=inp.mask, is_causal=causal))
        leaves = [t.detach().clone().requires_grad_(True) for t in prim]

        def second_order():
            oo, tt = JVPAttn.fwd_dual(*leaves, attn_mask=inp.mask, is_causal=causal)
            return torch.autograd.grad((oo, tt), leaves, grad_outputs=(inp.g_o, inp.g_to))

        so = _peak_added(second_order)
        yield {"dtype": dtype, "N": N, "B": B, "H": H, "D": D, "mask": mask,
               "inputs_mb": in_bytes / 2**20, "fwd_dual_added_mb": fwd / 2**20,
               "bwd_dual_added_mb": bwd / 2**20, "reverse_over_forward_added_mb": so / 2**20,
               "fwd_dual_added_bytes_per_token": fwd / (B * N),
               "reverse_over_forward_added_bytes_per_token": so / (B * N),
               "one_n_by_n_fp32_matrix_mb": B * H * N * N * 4 / 2**20}
        del inp, o, t_o, lse, mu, leaves
        torch.cuda.empty_cache()
