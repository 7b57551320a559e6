"""General additive mask (fa_fwd_bias): softmax(scale * q k^T + bias) v
against the fp64 oracle."""

import numpy as np
import pytest
import torch

import exact_tiled_attention_18_gb300 as fa
import oracle
from exact_tiled_attention_18_gb300 import workloads
from tests.helpers import GRAD_MAX_ABS, LSE_REL, O_MAX_ABS, O_MEAN_ABS, assert_row_term_close, scale_for, to64

pytestmark = pytest.mark.gpu


def _check(o, lse, o_ref, lse_ref, what, o_tol=O_MAX_ABS):
    o, lse = o.cpu().double().numpy(), lse.cpu().double().numpy()
    assert np.all(np.isfinite(o)), what
    err = np.abs(o - o_ref)
    assert err.max() <= o_tol and err.mean() <= O_MEAN_ABS, (what, err.max(), err.mean())
    assert np.array_equal(np.isinf(lse), np.isinf(lse_ref)), what
    fin = np.isfinite(lse_ref)
    if fin.any():
        rel = np.abs(lse[fin] - lse_ref[fin]) / np.maximum(np.abs(lse_ref[fin]), 1.0)
        assert rel.max() <= LSE_REL, (what, rel.max())


def _bias(shape, seed, gain=2.0, hide=0.0, row_stride=None):
    """bf16 bias of the given [b, h, nq, nk] shape (N(0,1) * gain, a fraction
    `hide` of entries -inf); with row_stride the rows live in a wider buffer
    (padded to a multiple of 8 elements) and a view is returned."""
    g = torch.Generator().manual_seed(seed)
    b = torch.randn(*shape, generator=g) * gain
    if hide:
        b[torch.rand(*shape, generator=g) < hide] = -float("inf")
    if row_stride is not None:
        wide = torch.zeros(*shape[:-1], row_stride)
        wide[..., :shape[-1]] = b
        return wide.to(torch.bfloat16).cuda()[..., :shape[-1]]
    return b.to(torch.bfloat16).cuda()


def _ref(q, k, v, bias, scale, causal, sq=None, sk=None):
    B, H, Nq, Nk = q.shape[0], q.shape[1], q.shape[2], k.shape[2]
    bb = bias.expand(B, H, Nq, Nk).float().cpu().double().numpy()
    if sq is None:
        return oracle.forward(to64(q), to64(k), to64(v), scale, causal, bb)
    return oracle.forward_varlen(to64(q), to64(k), to64(v), scale, causal, sq, sk, bb)


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal", [
    (1, 2, 300, 300, 64, False),
    (2, 1, 517, 517, 128, True),
    (1, 2, 256, 640, 128, True),
    (1, 1, 1000, 1000, 64, True),
    (2, 2, 129, 384, 128, False),
])
def test_random_bias(B, H, Nq, Nk, d, causal):
    g = workloads.make_decode_inputs(B, H, Nq, Nk, d, seed=Nq + Nk + d)
    q, k, v = (g[n].cuda() for n in ("q", "k", "v"))
    bias = _bias((B, H, Nq, Nk), seed=Nk)
    scale = scale_for(d)
    o, lse = fa.forward_bias(q, k, v, bias, causal=causal, scale=scale)
    fa.sync_status()
    _check(o, lse, *_ref(g["q"], g["k"], g["v"], bias, scale, causal), (B, H, Nq, Nk, d, causal))


@pytest.mark.parametrize("d", [64, 128])
def test_hidden_keys_and_rows(d):
    """A sparse -inf mask, a fully hidden row, and rows whose whole first key
    tile is hidden while later keys are visible."""
    B, H, N = 1, 2, 700
    g = workloads.make_decode_inputs(B, H, N, N, d, seed=5 + d)
    q, k, v = (g[n].cuda() for n in ("q", "k", "v"))
    b = _bias((B, H, N, N), seed=9, hide=0.3).cpu()
    b[0, 0, 5, :] = -float("inf")          # no key at all
    b[0, 1, 10:20, :300] = -float("inf")   # first key tiles hidden, keys from 300 on
    b[0, 1, 30, :690] = -float("inf")      # only the last keys
    bias = b.cuda()
    scale = scale_for(d)
    for causal in (False, True):
        o, lse = fa.forward_bias(q, k, v, bias, causal=causal, scale=scale)
        fa.sync_status()
        o_ref, lse_ref = _ref(g["q"], g["k"], g["v"], bias, scale, causal)
        _check(o, lse, o_ref, lse_ref, ("hidden", d, causal))
        oc = o.cpu()
        assert torch.all(oc[0, 0, 5] == 0) and torch.isneginf(lse.cpu()[0, 0, 5])


@pytest.mark.parametrize("shape", ["shared", "per_head", "key_row"])
def test_broadcast_bias(shape):
    B, H, Nq, Nk, d = 2, 3, 400, 400, 128
    g = workloads.make_decode_inputs(B, H, Nq, Nk, d, seed=11)
    q, k, v = (g[n].cuda() for n in ("q", "k", "v"))
    dims = {"shared": (1, 1, Nq, Nk), "per_head": (1, H, Nq, Nk), "key_row": (B, 1, 1, Nk)}[shape]
    bias = _bias(dims, seed=13, hide=0.1 if shape == "key_row" else 0.0)
    scale = scale_for(d)
    o, lse = fa.forward_bias(q, k, v, bias, causal=True, scale=scale)
    fa.sync_status()
    _check(o, lse, *_ref(g["q"], g["k"], g["v"], bias, scale, True), shape)


def test_padded_batch_with_bias_and_ragged_keys():
    """Unequal and padded lengths, Nk not a multiple of 8 (rows padded to a
    stride of 304), bf16 output."""
    B, H, Nq, Nk, d = 3, 2, 260, 300, 128
    sq, sk = [260, 100, 7], [300, 299, 150]
    g = workloads.make_decode_inputs(B, H, Nq, Nk, d, seed=17)
    q, k, v = (g[n].cuda() for n in ("q", "k", "v"))
    bias = _bias((B, H, Nq, Nk), seed=19, hide=0.05, row_stride=304)
    assert bias.stride(2) == 304
    lq = torch.tensor(sq, dtype=torch.int32, device="cuda")
    lk = torch.tensor(sk, dtype=torch.int32, device="cuda")
    scale = scale_for(d)
    o, lse = fa.forward_bias(q, k, v, bias, lq, lk, causal=True, scale=scale, o_dtype=torch.bfloat16)
    fa.sync_status()
    o_ref, lse_ref = _ref(g["q"], g["k"], g["v"], bias, scale, True, sq, sk)
    _check(o.float(), lse, o_ref, lse_ref, "padded bias", o_tol=O_MAX_ABS + 2 ** -8 * np.abs(o_ref).max())


def test_zero_bias_matches_unmasked_forward():
    g = workloads.make_decode_inputs(1, 2, 500, 500, 128, seed=23)
    q, k, v = (g[n].cuda() for n in ("q", "k", "v"))
    zero = torch.zeros((1, 1, 500, 504), dtype=torch.bfloat16, device="cuda")[..., :500]
    a = fa.forward_bias(q, k, v, zero, causal=True)
    b = fa.forward(q, k, v, causal=True)
    fa.sync_status()
    assert (a[0] - b[0]).abs().max() <= 2e-3 and (a[1] - b[1]).abs().max() <= 1e-5


# ---------------------------------------------------------------- gradients

def _check_grads(got, ref, what):
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        g = g.cpu().double().numpy()
        assert np.all(np.isfinite(g)), (what, name)
        err = np.abs(g - r).max()
        assert err <= GRAD_MAX_ABS, (what, name, err)


def _grads(q, k, v, do, bias, scale, causal, lq=None, lk=None, o_dtype=None, with_row_term=False):
    qc, kc, vc, doc = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = fa.forward_bias(qc, kc, vc, bias, lq, lk, causal=causal, scale=scale, o_dtype=o_dtype)
    ws = torch.empty(q.shape[0] * q.shape[1] * q.shape[2], dtype=torch.float32, device="cuda")
    g = fa.backward_bias(qc, kc, vc, o, lse, doc, bias, lq, lk, causal=causal, scale=scale, workspace=ws)
    fa.sync_status()
    out = tuple(t.cpu() for t in g)
    return out + (ws.cpu(),) if with_row_term else out


def _ref_grads(q, k, v, do, bias, scale, causal, sq=None, sk=None, with_row_term=False):
    B, H, Nq, Nk = q.shape[0], q.shape[1], q.shape[2], k.shape[2]
    bb = bias.expand(B, H, Nq, Nk).float().cpu().double().numpy()
    if sq is None:
        r = oracle.backward(to64(q), to64(k), to64(v), to64(do), scale, causal, bb)
    else:
        r = oracle.backward_varlen(to64(q), to64(k), to64(v), to64(do), scale, causal, sq, sk, bb)
    return r if with_row_term else r[:3]


def _check_row_term(ws, q, k, v, do, bias, scale, causal, rd, what, sq=None, sk=None):
    """D in the workspace against the oracle, at the fp32 bound of
    tests/helpers.py (D_abs from the oracle on |V| and |dO|)."""
    rd_abs = _ref_grads(q, k, v.abs(), do.abs(), bias, scale, causal, sq, sk, with_row_term=True)[3]
    rel = assert_row_term_close(ws.numpy(), rd, rd_abs, what)
    print(f"{what}: D largest error / D_abs {rel:.2e}")


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal", [
    (1, 2, 300, 300, 64, False),
    (2, 1, 517, 517, 128, True),
    (1, 2, 256, 640, 128, True),
    (2, 2, 384, 384, 64, False),
    (1, 1, 200, 129, 128, False),
    (1, 2, 640, 256, 64, True),
])
def test_backward_random_bias(B, H, Nq, Nk, d, causal):
    seed = 3 * Nq + Nk + d
    g = workloads.make_decode_inputs(B, H, Nq, Nk, d, seed=seed)
    do = workloads.randn_bf16((B, H, Nq, d), seed + 3)
    bias = _bias((B, H, Nq, Nk), seed=seed + 4, hide=0.05)
    scale = scale_for(d)
    *got, ws = _grads(g["q"], g["k"], g["v"], do, bias, scale, causal, with_row_term=True)
    ref = _ref_grads(g["q"], g["k"], g["v"], do, bias, scale, causal, with_row_term=True)
    _check_grads(got, ref[:3], (B, H, Nq, Nk, d, causal))
    _check_row_term(ws, g["q"], g["k"], g["v"], do, bias, scale, causal, ref[3], (B, H, Nq, Nk, d, causal))


@pytest.mark.parametrize("d", [64, 128])
def test_backward_hidden_keys_and_rows(d):
    B, H, N = 1, 2, 700
    g = workloads.make_decode_inputs(B, H, N, N, d, seed=31 + d)
    do = workloads.randn_bf16((B, H, N, d), 37 + d)
    b = _bias((B, H, N, N), seed=41, hide=0.3).cpu()
    b[0, 0, 5, :] = -float("inf")
    b[0, 1, 10:20, :300] = -float("inf")
    b[0, 1, 30, :690] = -float("inf")
    b[0, 0, :, 650:] = -float("inf")   # keys no query sees: dK = dV = 0 there
    bias = b.cuda()
    scale = scale_for(d)
    for causal in (False, True):
        *got, ws = _grads(g["q"], g["k"], g["v"], do, bias, scale, causal, with_row_term=True)
        ref = _ref_grads(g["q"], g["k"], g["v"], do, bias, scale, causal, with_row_term=True)
        _check_grads(got, ref[:3], ("hidden", d, causal))
        _check_row_term(ws, g["q"], g["k"], g["v"], do, bias, scale, causal, ref[3], ("hidden", d, causal))
        assert torch.all(ws.reshape(B, H, N)[0, 0, 5] == 0)
        assert torch.all(got[0][0, 0, 5] == 0)
        assert torch.all(got[1][0, 0, 650:] == 0) and torch.all(got[2][0, 0, 650:] == 0)


@pytest.mark.parametrize("shape", ["shared", "per_head", "key_row"])
def test_backward_broadcast_bias(shape):
    B, H, Nq, Nk, d = 2, 3, 400, 400, 128
    g = workloads.make_decode_inputs(B, H, Nq, Nk, d, seed=43)
    do = workloads.randn_bf16((B, H, Nq, d), 47)
    dims = {"shared": (1, 1, Nq, Nk), "per_head": (1, H, Nq, Nk), "key_row": (B, 1, 1, Nk)}[shape]
    # key_row: a key-padding style mask (0 or -inf, with a little noise)
    bias = _bias(dims, seed=53, gain=0.5 if shape == "key_row" else 2.0, hide=0.1 if shape == "key_row" else 0.0)
    scale = scale_for(d)
    got = _grads(g["q"], g["k"], g["v"], do, bias, scale, True)
    _check_grads(got, _ref_grads(g["q"], g["k"], g["v"], do, bias, scale, True), shape)


def test_backward_dominant_keys_within_rounding_bound():
    """A per-key bias of N(0, 4) makes a few keys dominate every query, so
    dV_j = sum_i P_ij dO_i sums hundreds of large terms (|dV| about 4x the
    unmasked case).  The tensor-core product takes P in bf16 (unit roundoff
    2^-8), which bounds the error of dV_jc by 2^-8 sum_i P_ij |dO_ic|; the
    oracle gives that sum exactly as its dV for |dO|.  dQ and dK keep the
    plain tolerance.  ("FlashAttention Interview Questions", section "Why can
    recomputation help training?": a tolerance fitted to each configuration.)"""
    B, H, Nq, Nk, d = 2, 3, 400, 400, 128
    g = workloads.make_decode_inputs(B, H, Nq, Nk, d, seed=43)
    do = workloads.randn_bf16((B, H, Nq, d), 47)
    bias = _bias((B, 1, 1, Nk), seed=53, gain=2.0, hide=0.1)
    scale = scale_for(d)
    got = _grads(g["q"], g["k"], g["v"], do, bias, scale, True)
    ref = _ref_grads(g["q"], g["k"], g["v"], do, bias, scale, True)
    _check_grads(got[:2], ref[:2], "dominant keys")
    mass = _ref_grads(g["q"], g["k"], g["v"], do.abs(), bias, scale, True)[2]
    err = np.abs(got[2].double().numpy() - ref[2])
    # reported against the plain tolerance as well: the kernel feeds P to the
    # dV product as one bf16 value (a hi + lo pair, one more GEMM per tile,
    # would bring this under 2e-2)
    print(f"dominant keys: dV max abs error {err.max():.4f} (plain tolerance {GRAD_MAX_ABS}, "
          f"{'within' if err.max() <= GRAD_MAX_ABS else 'above'} it), |dV| up to {np.abs(ref[2]).max():.1f}")
    assert np.all(err <= GRAD_MAX_ABS + 2.0 ** -8 * mass), err.max()


def test_backward_padded_batch_with_bias():
    """Unequal and padded lengths, rows padded to a stride of 304 elements,
    bf16 O from the forward; padding rows of the gradients are 0."""
    B, H, Nq, Nk, d = 3, 2, 260, 300, 128
    sq, sk = [260, 100, 7], [300, 299, 150]
    g = workloads.make_decode_inputs(B, H, Nq, Nk, d, seed=59)
    do = workloads.randn_bf16((B, H, Nq, d), 61)
    bias = _bias((B, H, Nq, Nk), seed=67, hide=0.05, row_stride=304)
    lq = torch.tensor(sq, dtype=torch.int32, device="cuda")
    lk = torch.tensor(sk, dtype=torch.int32, device="cuda")
    scale = scale_for(d)
    *got, ws = _grads(g["q"], g["k"], g["v"], do, bias, scale, True, lq, lk, o_dtype=torch.bfloat16,
                      with_row_term=True)
    ref = _ref_grads(g["q"], g["k"], g["v"], do, bias, scale, True, sq, sk, with_row_term=True)
    _check_grads(got, ref[:3], "padded bias")
    _check_row_term(ws, g["q"], g["k"], g["v"], do, bias, scale, True, ref[3], "padded bias (bf16 O)", sq, sk)
    dq, dk, dv = got
    for b in range(B):
        assert torch.all(dq[b, :, sq[b]:] == 0)
        assert torch.all(dk[b, :, sk[b]:] == 0) and torch.all(dv[b, :, sk[b]:] == 0)


def test_backward_zero_bias_matches_unmasked():
    g = workloads.make_decode_inputs(1, 2, 500, 500, 128, seed=71)
    q, k, v = (g[n].cuda() for n in ("q", "k", "v"))
    do = workloads.randn_bf16((1, 2, 500, 128), 73).cuda()
    zero = torch.zeros((1, 1, 1, 500), dtype=torch.bfloat16, device="cuda")
    o, lse = fa.forward(q, k, v, causal=True)
    a = fa.backward_bias(q, k, v, o, lse, do, zero, causal=True)
    b = fa.backward(q, k, v, o, lse, do, causal=True)
    fa.sync_status()
    for x, y in zip(a, b):
        assert (x - y).abs().max() <= 1e-4
