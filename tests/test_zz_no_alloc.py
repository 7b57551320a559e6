"""fa_bwd_noalloc, the backward entry point that allocates nothing.

Some callers cannot let a library allocate device memory while they run: a
framework or inference runtime that hands out every byte of device memory
from its own pool, or a latency-critical loop that reserved its memory up
front.  fa_bwd_noalloc serves them by keeping its scratch (the backward row
term) in a fixed array inside the library.  These tests call it through the
C ABI and check that it returns what the allocating entry point fa_bwd
returns: the same kernels on the same inputs, with only the row term held in
a different buffer, so the gradients must agree bit for bit (a stale or
partly written scratch row would show there first).  One case is also
checked against the fp64 oracle.  The file is named so that pytest collects
it last.
"""

import numpy as np
import pytest
import torch

import exact_tiled_attention_18_gb300 as fa
import oracle
from exact_tiled_attention_18_gb300 import workloads
from tests.helpers import GRAD_MAX_ABS, scale_for, to64

pytestmark = pytest.mark.gpu


def _run(B, H, N, d, causal, seed, against_oracle=False):
    inp = workloads.make_inputs(B, H, N, d, seed=seed, with_grad=True)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    scale = scale_for(d)
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale)
    # the allocating entry point, with a caller-owned workspace
    ref = fa.backward(q, k, v, o, lse, do, causal=causal, scale=scale,
                      workspace=torch.empty(B * H * N, dtype=torch.float32, device="cuda"))
    out = [torch.full((B, H, N, d), float("nan"), dtype=torch.float32, device="cuda") for _ in range(3)]
    stream = torch.cuda.current_stream().cuda_stream
    st = fa.fa_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), do.data_ptr(),
                           out[0].data_ptr(), out[1].data_ptr(), out[2].data_ptr(), B, H, N, d, scale,
                           int(causal), stream)
    assert st == 0, fa.fa_status_string(st)
    assert fa.fa_sync_status(stream) == 0
    for name, a, b in zip(("dQ", "dK", "dV"), out, ref):
        assert torch.equal(a, b), (name, (a - b).abs().max().item())
    if against_oracle:
        x = {n: to64(inp[n]) for n in inp}
        for name, a, r in zip(("dQ", "dK", "dV"), out,
                              oracle.backward(x["q"], x["k"], x["v"], x["do"], scale, causal)[:3]):
            err = float(np.abs(a.cpu().double().numpy() - r).max())
            assert err <= GRAD_MAX_ABS, (name, err)


def test_noalloc_matches_fa_bwd_two_calls_in_a_row():
    # the second call is smaller than the first, so it runs over scratch rows
    # the first call left behind
    _run(2, 3, 700, 128, True, seed=21, against_oracle=True)
    _run(1, 2, 333, 64, False, seed=22)


def test_noalloc_rejects_sizes_above_its_scratch():
    fake = 0x10000
    rows = fa.FA_NOALLOC_MAX_ROWS
    st = fa.fa_bwd_noalloc(fake, fake, fake, fake, fake, fake, fake, fake, fake, 1, 1, rows + 1, 64, 0.125, 0, 0)
    assert st == 1, fa.fa_status_string(st)
