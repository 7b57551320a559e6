"""Decode-shaped forward (fa_fwd_decode): a few query rows against a long
K/V, split over many CTAs and merged by log-sum-exp, against the fp64
oracle."""

import numpy as np
import pytest
import torch

import exact_tiled_attention_18_gb300 as fa
import oracle
from exact_tiled_attention_18_gb300 import workloads
from tests.helpers import LSE_REL, O_MAX_ABS, O_MEAN_ABS, scale_for, to64

pytestmark = pytest.mark.gpu


def _check(o, lse, o_ref, lse_ref, what):
    o, lse = o.cpu().double().numpy(), lse.cpu().double().numpy()
    assert np.all(np.isfinite(o)), what
    err = np.abs(o - o_ref)
    assert err.max() <= O_MAX_ABS and err.mean() <= O_MEAN_ABS, (what, err.max(), err.mean())
    assert np.array_equal(np.isinf(lse), np.isinf(lse_ref)), what
    fin = np.isfinite(lse_ref)
    if fin.any():
        rel = np.abs(lse[fin] - lse_ref[fin]) / np.maximum(np.abs(lse_ref[fin]), 1.0)
        assert rel.max() <= LSE_REL, (what, rel.max())


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal", [
    (1, 1, 1, 1, 128, True),
    (1, 2, 1, 63, 64, True),
    (1, 1, 1, 64, 128, False),
    (2, 1, 1, 65, 128, True),
    (1, 3, 2, 300, 64, True),
    (1, 1, 3, 1000, 128, True),     # rows see 998, 999, 1000 keys
    (1, 2, 5, 777, 128, False),
    (2, 2, 8, 2049, 128, True),
    (1, 1, 8, 4096, 64, True),
    (1, 1, 4, 20000, 128, True),    # many splits
    (1, 1, 8, 3, 128, True),        # more queries than keys: the first 5 see none
])
def test_decode_matches_oracle(B, H, Nq, Nk, d, causal):
    inp = workloads.make_decode_inputs(B, H, Nq, Nk, d, seed=Nq * 7 + Nk + d)
    scale = scale_for(d)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o, lse = fa.forward_decode(q, k, v, causal=causal, scale=scale)
    fa.sync_status()
    o_ref, lse_ref = oracle.forward(to64(inp["q"]), to64(inp["k"]), to64(inp["v"]), scale, causal)
    _check(o, lse, o_ref, lse_ref, (B, H, Nq, Nk, d, causal))


@pytest.mark.parametrize("d", [64, 128])
def test_decode_padded_batch(d):
    """A batch of caches of different lengths (one empty, one sequence with no
    query), with a caller-owned workspace."""
    B, H, Nq, Nk = 6, 2, 4, 3000
    sq, sk = [4, 1, 3, 0, 4, 2], [3000, 1, 2500, 100, 0, 640]
    inp = workloads.make_decode_inputs(B, H, Nq, Nk, d, seed=17 + d)
    scale = scale_for(d)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    lq = torch.tensor(sq, dtype=torch.int32, device="cuda")
    lk = torch.tensor(sk, dtype=torch.int32, device="cuda")
    ws = torch.empty(fa.fa_fwd_decode_workspace_bytes(B, H, Nq, Nk, d) // 4, dtype=torch.float32, device="cuda")
    o, lse = fa.forward_decode(q, k, v, lq, lk, causal=True, scale=scale, workspace=ws)
    fa.sync_status()
    o_ref, lse_ref = oracle.forward_varlen(to64(inp["q"]), to64(inp["k"]), to64(inp["v"]), scale, True, sq, sk)
    _check(o, lse, o_ref, lse_ref, ("padded", d))
    oc, lc = o.cpu(), lse.cpu()
    for b in range(B):
        assert torch.all(oc[b, :, sq[b]:] == 0) and torch.all(torch.isneginf(lc[b, :, sq[b]:]))


def test_decode_agrees_with_prefill_kernel():
    """fa_fwd_decode and fa_fwd_varlen compute the same thing."""
    inp = workloads.make_decode_inputs(2, 4, 2, 5000, 128, seed=3)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    a = fa.forward_decode(q, k, v, causal=True)
    b = fa.forward_varlen(q, k, v, causal=True)
    fa.sync_status()
    assert (a[0] - b[0]).abs().max() <= 2e-3
    assert (a[1] - b[1]).abs().max() <= 1e-4


def test_decode_full_size_sampled_heads():
    """The decode workload in the launch configuration the bench times, 24
    seeded (b, h) heads checked against the oracle row by row."""
    w = workloads.DECODE_WORKLOADS["decode_b8_h32_nq1_nk32768_d128"]
    inp = workloads.make_decode_inputs(w.B, w.H, w.Nq, w.Nk, w.d, seed=0)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o, lse = fa.forward_decode(q, k, v, causal=w.causal, scale=w.scale)
    fa.sync_status()
    o, lse = o.cpu(), lse.cpu()
    g = torch.Generator().manual_seed(11)
    heads = {(0, 0), (w.B - 1, w.H - 1)}
    while len(heads) < 24:
        heads.add((int(torch.randint(0, w.B, (1,), generator=g)), int(torch.randint(0, w.H, (1,), generator=g))))
    rows = [(b, h, i) for (b, h) in sorted(heads) for i in range(w.Nq)]
    o_ref, lse_ref = oracle.forward_rows(to64(inp["q"]), to64(inp["k"]), to64(inp["v"]), w.scale, w.causal, rows)
    got_o = np.stack([o[b, h, i].double().numpy() for (b, h, i) in rows])
    got_l = np.array([float(lse[b, h, i]) for (b, h, i) in rows])
    _check(torch.from_numpy(got_o), torch.from_numpy(got_l), o_ref, lse_ref, "decode full size")


def test_decode_allocates_nothing_with_workspace():
    w = workloads.DECODE_WORKLOADS["decode_b8_h32_nq1_nk32768_d128"]
    B, H = 2, 4
    inp = workloads.make_decode_inputs(B, H, w.Nq, w.Nk, w.d, seed=1)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o = torch.empty((B, H, w.Nq, w.d), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, H, w.Nq), dtype=torch.float32, device="cuda")
    ws = torch.empty(fa.fa_fwd_decode_workspace_bytes(B, H, w.Nq, w.Nk, w.d) // 4, dtype=torch.float32,
                     device="cuda")
    torch.cuda.synchronize()
    before = torch.cuda.memory_allocated()
    torch.cuda.reset_peak_memory_stats()
    fa.forward_decode(q, k, v, causal=True, workspace=ws, out=(o, lse))
    fa.sync_status()
    assert torch.cuda.max_memory_allocated() == before
