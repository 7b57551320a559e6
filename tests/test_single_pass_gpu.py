"""Single-pass backward (fa_bwd_single_pass, stages 2 and 3 of fa_bwd_stage)
against the fp64 oracle.

The row-term pass forms D_i = sum_j P_ij dP_ij from the recomputed
probabilities; the dK/dV sweep then also forms every tile's dQ share and adds
it into dQ ("FlashAttention Interview Questions", section "Why can
recomputation help training?").  Gradients are held to the stated max-abs
tolerance and D to the fp32 bound of tests/helpers.py, on small ragged
shapes, padded and masked batches, and whole heads of the full-size
training and long-context workloads (the latter with its 10x query rows).
"""

import numpy as np
import pytest
import torch

import exact_tiled_attention_18_gb300 as fa
import oracle
from exact_tiled_attention_18_gb300 import workloads
from tests.helpers import GRAD_MAX_ABS, assert_row_term_close, scale_for, to64

pytestmark = pytest.mark.gpu


def _run(q, k, v, do, causal, scale, bias=None, lq=None, lk=None):
    o, lse = (fa.forward_bias(q, k, v, bias, lq, lk, causal=causal, scale=scale) if bias is not None else
              fa.forward_varlen(q, k, v, lq, lk, causal=causal, scale=scale))
    ws = torch.empty(q.shape[0] * q.shape[1] * q.shape[2], dtype=torch.float32, device="cuda")
    g = fa.backward_single_pass(q, k, v, lse, do, bias, lq, lk, causal=causal, scale=scale, workspace=ws)
    fa.sync_status()
    return tuple(t.cpu() for t in g) + (ws.cpu(),)


def _check(got, ref, ref_abs_d, what):
    errs = []
    for name, g, r in zip(("dQ", "dK", "dV"), got[:3], ref[:3]):
        g = g.double().numpy()
        assert np.all(np.isfinite(g)), (what, name)
        err = float(np.abs(g - r).max())
        errs.append(err)
        assert err <= GRAD_MAX_ABS, (what, name, err)
    rel = assert_row_term_close(got[3].numpy(), ref[3], ref_abs_d, f"{what} D")
    print(f"{what}: dQ {errs[0]:.2e} dK {errs[1]:.2e} dV {errs[2]:.2e}; D largest error / D_abs {rel:.2e}")


SMALL = [
    (1, 1, 256, 64, False),
    (1, 1, 256, 64, True),
    (1, 1, 1, 64, True),
    (1, 1, 1, 128, False),
    (1, 1, 127, 128, True),
    (2, 1, 129, 128, False),
    (1, 2, 200, 64, True),
    (1, 1, 257, 128, True),
    (2, 2, 384, 128, True),
    (1, 3, 517, 128, True),
    (1, 2, 1000, 64, True),
    (1, 1, 1024, 128, False),
]


@pytest.mark.parametrize("B,H,N,d,causal", SMALL)
def test_single_pass_small_matches_oracle(B, H, N, d, causal):
    inp = workloads.make_inputs(B, H, N, d, seed=500 + N + d + causal, with_grad=True)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    scale = scale_for(d)
    got = _run(q, k, v, do, causal, scale)
    x = {n: to64(inp[n]) for n in inp}
    ref = oracle.backward(x["q"], x["k"], x["v"], x["do"], scale, causal)
    ref_abs = oracle.backward(x["q"], x["k"], np.abs(x["v"]), np.abs(x["do"]), scale, causal)[3]
    _check(got, ref, ref_abs, (B, H, N, d, causal))


@pytest.mark.parametrize("name,heads", [
    ("training_b4_h16_n8192_d128_causal", [(0, 0), (3, 15)]),
    ("long_context_b1_h32_n16384_d128_causal", [(0, 17), (0, 3)]),
])
def test_single_pass_full_size_whole_heads(name, heads):
    w = workloads.WORKLOADS[name]
    inp = workloads.workload_inputs(w, 0)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    got = _run(q, k, v, do, w.causal, w.scale)
    ws = got[3].reshape(w.B, w.H, w.N)
    for (b, h) in heads:
        x = {n: to64(inp[n][b:b + 1, h:h + 1]) for n in inp}
        ref = oracle.backward(x["q"], x["k"], x["v"], x["do"], w.scale, w.causal)
        ref_abs = oracle.backward(x["q"], x["k"], np.abs(x["v"]), np.abs(x["do"]), w.scale, w.causal)[3]
        sel = tuple(t[b:b + 1, h:h + 1] for t in got[:3]) + (ws[b:b + 1, h:h + 1],)
        _check(sel, ref, ref_abs, f"{name} head {(b, h)}")


@pytest.mark.parametrize("d,causal", [(64, True), (64, False), (128, False), (128, True)])
def test_single_pass_padded_unequal(d, causal):
    """Padded batch with unequal lengths, an empty sequence and one without
    keys.  Without the causal rule the padding keys inside a key tile are not
    masked; their dS must still add nothing to dQ."""
    B, H, Nq, Nk = 4, 2, 700, 900
    sq, sk = [700, 0, 333, 129], [900, 77, 0, 500]
    g = workloads.make_decode_inputs(B, H, Nq, Nk, d, seed=520 + d)
    do = workloads.randn_bf16((B, H, Nq, d), 523 + d)
    q, k, v, doc = g["q"].cuda(), g["k"].cuda(), g["v"].cuda(), do.cuda()
    lq = torch.tensor(sq, dtype=torch.int32, device="cuda")
    lk = torch.tensor(sk, dtype=torch.int32, device="cuda")
    scale = scale_for(d)
    got = _run(q, k, v, doc, causal, scale, lq=lq, lk=lk)
    x = {n: to64(g[n]) for n in g}
    ref = oracle.backward_varlen(x["q"], x["k"], x["v"], to64(do), scale, causal, sq, sk)
    ref_abs = oracle.backward_varlen(x["q"], x["k"], np.abs(x["v"]), np.abs(to64(do)), scale, causal, sq, sk)[3]
    _check(got, ref, ref_abs, ("padded", d, causal))
    for b in range(B):
        assert torch.all(got[0][b, :, sq[b]:] == 0)
        assert torch.all(got[1][b, :, sk[b]:] == 0) and torch.all(got[2][b, :, sk[b]:] == 0)


@pytest.mark.parametrize("d", [64, 128])
def test_single_pass_with_mask(d):
    """A random additive mask with hidden keys, a fully hidden row and rows
    whose first key tiles are hidden."""
    B, H, N = 1, 2, 700
    g = workloads.make_decode_inputs(B, H, N, N, d, seed=531 + d)
    do = workloads.randn_bf16((B, H, N, d), 537 + d)
    gen = torch.Generator().manual_seed(541)
    b = torch.randn(B, H, N, N, generator=gen) * 2.0
    b[torch.rand(B, H, N, N, generator=gen) < 0.3] = -float("inf")
    b[0, 0, 5, :] = -float("inf")
    b[0, 1, 10:20, :300] = -float("inf")
    bias = b.to(torch.bfloat16).cuda()
    scale = scale_for(d)
    bb = bias.float().cpu().double().numpy()
    x = {n: to64(g[n]) for n in g}
    for causal in (False, True):
        got = _run(g["q"].cuda(), g["k"].cuda(), g["v"].cuda(), do.cuda(), causal, scale, bias=bias)
        ref = oracle.backward(x["q"], x["k"], x["v"], to64(do), scale, causal, bb)
        ref_abs = oracle.backward(x["q"], x["k"], np.abs(x["v"]), np.abs(to64(do)), scale, causal, bb)[3]
        _check(got, ref, ref_abs, ("mask", d, causal))
        assert torch.all(got[0][0, 0, 5] == 0)


def test_single_pass_repeatability_and_stages():
    """dK and dV are the same bit for bit from run to run (each CTA sums its
    key tile's products in a fixed order); dQ, summed over key tiles by
    concurrent CTAs, agrees to fp32 rounding.  Stages 2 and 3 of
    fa_bwd_stage are the same computation."""
    B, H, N, d = 2, 3, 1100, 128
    inp = workloads.make_inputs(B, H, N, d, seed=551, with_grad=True)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    scale = scale_for(d)
    a = _run(q, k, v, do, True, scale)
    b = _run(q, k, v, do, True, scale)
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2]) and torch.equal(a[3], b[3])
    assert (a[0] - b[0]).abs().max().item() <= 1e-5
    o, lse = fa.forward(q, k, v, causal=True, scale=scale)
    out = [torch.full((B, H, N, d), float("nan"), dtype=torch.float32, device="cuda") for _ in range(3)]
    ws = torch.empty(B * H * N, dtype=torch.float32, device="cuda")
    for stage in (2, 3):
        fa.backward_stage(stage, q, k, v, None, lse, do, *out, ws, causal=True, scale=scale)
    fa.sync_status()
    assert torch.equal(out[1].cpu(), a[1]) and torch.equal(out[2].cpu(), a[2])
    assert (out[0].cpu() - a[0]).abs().max().item() <= 1e-5


def test_single_pass_agrees_with_two_pass():
    """Both algorithms compute the same gradients: dV bit for bit (same P,
    same products), dK and dQ to fp32 rounding (their row terms agree to
    about 1e-7 relative and dQ is summed in a different order)."""
    B, H, N, d = 1, 4, 1500, 64
    inp = workloads.make_inputs(B, H, N, d, seed=561, with_grad=True)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    scale = scale_for(d)
    o, lse = fa.forward(q, k, v, causal=True, scale=scale)
    two = fa.backward(q, k, v, o, lse, do, causal=True, scale=scale)
    one = fa.backward_single_pass(q, k, v, lse, do, causal=True, scale=scale)
    fa.sync_status()
    assert torch.equal(one[2], two[2])
    assert (one[1] - two[1]).abs().max().item() <= 1e-4
    assert (one[0] - two[0]).abs().max().item() <= 1e-2
