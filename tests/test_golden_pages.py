"""The FLOP convention used for throughput, pinned to the pages' benchmark rows.

The pages print time and TFLOP/s for the same runs (fixture cited in
tests/golden/pages_benchmark_rows.json).  Their product is the work counted
per call.  With the pages' unstated B*H*D fitted once (from one row), the
convention 12*B*H*N^2*D (halved for causal, masks not counted) must
reproduce every other row's work within the rounding of the printed figures.
"""

import json
import os

from forward_mode_flash_gb300 import metrics

HERE = os.path.dirname(os.path.abspath(__file__))


def load_rows():
    with open(os.path.join(HERE, "golden", "pages_benchmark_rows.json")) as f:
        return json.load(f)["rows"]


def test_flop_convention_reproduces_the_pages_work_per_call():
    rows = load_rows()
    ref = next(r for r in rows if r["dtype"] == "float16" and r["N"] == 2048 and
               not r["causal"] and r["mask"] == "none")
    # Fit B*H*D from one row: work = TFLOP/s * ms * 1e9.
    bhd = ref["tflops"] * ref["ms"] * 1e9 / metrics.flops_fwd_dual(1, 1, 2048, 2048, 1)
    assert abs(bhd - 1024) / 1024 < 0.03  # the inferred size is B*H*D = 1024 (+2%)
    for r in rows:
        work = r["tflops"] * r["ms"] * 1e9
        model = metrics.flops_fwd_dual(1, 1, r["N"], r["N"], bhd, r["causal"])
        # TFLOP/s is printed with 3 significant digits and time with 4.
        assert abs(work - model) / model < 0.03, r


def test_causal_halves_and_masks_do_not_change_the_count():
    assert metrics.flops_fwd_dual(2, 8, 512, 512, 64, True) * 2 == \
        metrics.flops_fwd_dual(2, 8, 512, 512, 64, False)
    assert metrics.flops_fwd_dual(4, 16, 2048, 2048, 128) == 12 * 4 * 16 * 2048 ** 2 * 128


def test_algorithmic_bytes():
    # six bf16 inputs read, two outputs written, lse and mu in fp32
    b = metrics.bytes_fwd_dual(4, 16, 2048, 2048, 128, 2)
    assert b == 8 * 4 * 16 * 2048 * 128 * 2 + 8 * 4 * 16 * 2048
    assert metrics.bytes_fwd_dual(2, 8, 1024, 1024, 64, 2, "bool", 2) - \
        metrics.bytes_fwd_dual(2, 8, 1024, 1024, 64, 2) == 2 * 1024 * 1024


def test_algorithmic_bytes_equal_the_buffers_a_call_reads_and_writes():
    # Independent of the formula: build each workload's actual buffers (the
    # six inputs and the mask from the seeded generator, outputs O and tO of
    # q's shape and dtype, lse and mu as float32 [B, H, Nq]) and add up their
    # sizes; every byte is read or written exactly once by one call.
    import torch

    from forward_mode_flash_gb300 import synth

    for name in ("f16_b2h8n512d64", "bf16_b2h8n1024d64_bool", "bf16_b2h8n1024d64_additive",
                 "bf16_b4h16n2048d128"):
        w = synth.WORKLOADS[name]
        inp = synth.make_inputs(w)
        ins = (inp.q, inp.k, inp.v, inp.dq, inp.dk, inp.dv)
        total = sum(t.numel() * t.element_size() for t in ins)
        total += 2 * inp.q.numel() * inp.q.element_size()           # O, tO
        total += 2 * inp.q.shape[0] * inp.q.shape[1] * inp.q.shape[2] * 4  # lse, mu
        if inp.mask is not None:
            m = inp.mask
            total += m.numel() * (1 if m.dtype == torch.bool else m.element_size())
        mb = 1 if inp.mask is None else inp.mask.shape[0]
        assert metrics.bytes_fwd_dual(w.B, w.H, w.N, w.n_keys, w.D, inp.q.element_size(),
                                      w.mask, mask_batch=mb) == total, name
