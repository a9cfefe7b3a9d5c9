"""GPU checks of the memory-scaling report and a tiny sequence-length sweep.

The kernels allocate no device memory, so the bytes one call adds on top of
its inputs are exactly its outputs (fwd_dual: O, tO and the float32 lse, mu;
bwd_dual: six gradients plus its workspace: 8 B*H*Nq bytes, and for problems
with few key-major CTAs the key-major split's partial sums), linear in N.  The
sizes below are multiples of the caching allocator's 512-byte rounding, so the
counts are exact.
"""

import pytest
import torch

from forward_mode_flash_gb300 import api, build, report

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


@pytest.mark.parametrize("mask", ["none", "causal"])
def test_calls_add_exactly_their_outputs(mask):
    B, H, D = 2, 8, 64
    rows = list(report.memory_scaling(Ns=(256, 512, 1024), B=B, H=H, D=D, mask=mask))
    for r in rows:
        N = r["N"]
        elem = 2  # bf16
        # outputs, plus the split-KV scratch where the key range is split
        fwd = 2 * B * H * N * D * elem + 2 * B * H * N * 4 + \
            api.fwd_dual_workspace_size(B, H, N, N, D, torch.bfloat16)
        bwd = 6 * B * H * N * D * elem + api.bwd_dual_workspace_size(B, H, N, N, D,
                                                                       torch.bfloat16)
        assert api.bwd_dual_workspace_size(B, H, N, N, D, torch.bfloat16) >= 8 * B * H * N
        assert r["fwd_dual_added_mb"] * 2**20 == fwd, r
        assert r["bwd_dual_added_mb"] * 2**20 == bwd, r
    # reverse-over-forward through JVPAttn.fwd_dual: linear in N (no N x N term);
    # the key-major split's partial sums (small problems only: their count of
    # splits falls as N grows) are taken out first
    per_token = []
    for r in rows:
        N = r["N"]
        split = api.bwd_dual_workspace_size(B, H, N, N, D, torch.bfloat16) - 8 * B * H * N
        per_token.append((r["reverse_over_forward_added_mb"] * 2**20 - split) / (B * N))
    assert max(per_token) <= 1.5 * min(per_token), per_token


def test_sweep_rows_are_well_formed():
    rows = list(report.sweep(dtypes=("bf16",), Ns=(64, 512), masks=("none", "bool"),
                             graph_max_n=64))
    assert [(r["N"], r["mask"]) for r in rows] == [(64, "none"), (64, "bool"), (512, "none"),
                                                   (512, "bool")]
    for r in rows:
        assert r["path"].startswith("tensor-core")
        assert r["ms_hot"] > 0 and r["ms_cold_l2"] > 0
        assert (r["ms_graph_batch100"] is not None) == (r["N"] <= 64)
    assert torch.cuda.memory_allocated() < 2**30
