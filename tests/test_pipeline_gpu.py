"""HostStepPipeline: a training step on pinned host tensors, cut into chunks of
(batch, head) pairs so that copies overlap kernels, gives exactly the results
of direct calls."""

import pytest
import torch

import exact_tiled_attention_18_gb300 as fa
from exact_tiled_attention_18_gb300 import workloads
from tests.helpers import scale_for

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("chunks", [1, 2, 4, 8])
def test_pipeline_matches_direct_calls(chunks):
    B, H, N, d = 4, 2, 500, 128
    inp = workloads.make_inputs(B, H, N, d, seed=12, with_grad=True)
    scale = scale_for(d)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, causal=True, scale=scale)
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, causal=True, scale=scale)
    fa.sync_status()
    host_in = {n: inp[n].pin_memory() for n in ("q", "k", "v", "do")}
    host_out = {n: torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
                for n, t in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))}
    pipe = fa.HostStepPipeline(B, H, N, d, True, scale, chunks=chunks)
    for _ in range(2):  # the second step reuses every device buffer
        pipe.step(host_in, host_out)
    pipe.synchronize()
    fa.sync_status()
    for name, ref in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv)):
        assert torch.equal(host_out[name], ref.cpu()), name


def test_pipeline_rejects_uneven_chunks():
    with pytest.raises(ValueError):
        fa.HostStepPipeline(3, 1, 128, 64, False, 0.125, chunks=2)
    with pytest.raises(ValueError):
        fa.HostStepPipeline(2, 3, 128, 64, False, 0.125, chunks=4)
