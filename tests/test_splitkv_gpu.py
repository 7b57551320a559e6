"""Split-key forward (fa_fwd_splitkv): each query tile's keys are split over
several CTAs and the partial results merged by their log-sum-exp.  Against
the fp64 oracle on shapes that do split (few query tiles: one head of a few
thousand tokens), ragged N, both head sizes, causal and not; and against
fa_fwd on the same inputs."""

import numpy as np
import pytest
import torch

import exact_tiled_attention_18_gb300 as fa
import oracle
from exact_tiled_attention_18_gb300 import workloads
from tests.helpers import assert_forward_close, scale_for, to64

pytestmark = pytest.mark.gpu

BAND = 4096
SENTINEL = 0xA5


@pytest.mark.parametrize("B,H,N,d,causal", [
    (1, 1, 4096, 64, False),
    (1, 1, 4096, 64, True),
    (1, 1, 1500, 128, True),
    (1, 2, 1000, 64, False),
    (2, 1, 2047, 128, True),
    (1, 1, 513, 128, False),
    (1, 1, 300, 64, True),     # too few key tiles to split: runs fa_fwd
])
def test_splitkv_matches_oracle(B, H, N, d, causal):
    inp = workloads.make_inputs(B, H, N, d, seed=600 + N + d + causal)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    scale = scale_for(d)
    o, lse = fa.forward_splitkv(q, k, v, causal=causal, scale=scale)
    o2, lse2 = fa.forward(q, k, v, causal=causal, scale=scale)
    fa.sync_status()
    o_ref, lse_ref = oracle.forward(to64(inp["q"]), to64(inp["k"]), to64(inp["v"]), scale, causal)
    mx, mean, le = assert_forward_close(o.cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, f"{(B, H, N, d, causal)}")
    # the unsplit forward rounds its weights against other reference maxima:
    # the two agree to the rounding of P
    assert (o - o2).abs().max().item() <= 1e-2
    assert (lse - lse2).abs().max().item() <= 1e-4
    print(f"{(B, H, N, d, causal)}: O max {mx:.2e} mean {mean:.2e}, LSE rel {le:.2e}")


@pytest.mark.parametrize("name", ["memory_exercise_n4096_d64", "memory_exercise_n4096_d64_causal"])
def test_splitkv_memory_exercise_workload(name):
    w = workloads.WORKLOADS[name]
    inp = workloads.workload_inputs(w, 0)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    ws = torch.empty(fa.fa_fwd_splitkv_workspace_bytes(w.B, w.H, w.N, w.d) // 4, dtype=torch.float32, device="cuda")
    o, lse = fa.forward_splitkv(q, k, v, causal=w.causal, scale=w.scale, workspace=ws)
    fa.sync_status()
    o_ref, lse_ref = oracle.forward(to64(inp["q"]), to64(inp["k"]), to64(inp["v"]), w.scale, w.causal)
    assert_forward_close(o.cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, name)


def test_splitkv_guard_bands():
    """Outputs and the workspace inside sentinel bands: nothing is written
    outside them."""
    B, H, N, d = 1, 1, 1500, 128
    inp = workloads.make_inputs(B, H, N, d, seed=611)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))

    def banded(nbytes):
        buf = torch.full((BAND + nbytes + BAND,), SENTINEL, dtype=torch.uint8, device="cuda")
        return buf, buf[BAND:BAND + nbytes]

    nb_o, nb_l = B * H * N * d * 4, B * H * N * 4
    nb_w = fa.fa_fwd_splitkv_workspace_bytes(B, H, N, d)
    (bo, o), (bl, lse), (bw, ws) = banded(nb_o), banded(nb_l), banded(nb_w)
    fa.forward_splitkv(q, k, v, causal=True, workspace=ws.view(torch.float32),
                       out=(o.view(torch.float32).view(B, H, N, d), lse.view(torch.float32).view(B, H, N)))
    fa.sync_status()
    for buf, n in ((bo, nb_o), (bl, nb_l), (bw, nb_w)):
        b = buf.cpu()
        assert torch.all(b[:BAND] == SENTINEL) and torch.all(b[BAND + n:] == SENTINEL)
