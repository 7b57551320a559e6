"""Unequal query/key lengths and padded batches (fa_fwd_varlen and
fa_bwd_varlen) against the fp64 oracle, with the bottom-right causal
alignment."""

import numpy as np
import pytest
import torch

import exact_tiled_attention_18_gb300 as fa
import oracle
from exact_tiled_attention_18_gb300 import workloads
from tests.helpers import GRAD_MAX_ABS, O_MAX_ABS, O_MEAN_ABS, LSE_REL, assert_row_term_close, scale_for, to64

pytestmark = pytest.mark.gpu


def _inputs(B, H, Nq, Nk, d, seed):
    q = workloads.randn_bf16((B, H, Nq, d), seed)
    k = workloads.randn_bf16((B, H, Nk, d), seed + 1)
    v = workloads.randn_bf16((B, H, Nk, d), seed + 2)
    return q, k, v


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


UNEQUAL = [
    (1, 2, 1, 300, 64, True),      # one decoding query sees every key
    (1, 2, 1, 300, 128, False),
    (1, 1, 100, 300, 128, True),
    (1, 1, 300, 100, 128, True),   # the first 200 queries see no key
    (2, 1, 129, 257, 64, False),
    (1, 2, 640, 384, 128, True),
    (1, 1, 384, 640, 64, True),
    (1, 1, 1, 1, 64, True),
]

# valid lengths of a padded batch of B = 5 sequences (Nq = 300, Nk = 400):
# full, short, no keys, more keys than queries, no queries
PAD_SQ = [300, 17, 129, 256, 0]
PAD_SK = [400, 250, 0, 131, 77]


def _pad_garbage(t, lens, gain, seed):
    """Copy of t whose rows past each sequence's valid length hold gain * N(0, 1)
    values (finite), so that a result can be shown not to depend on them."""
    t = t.clone()
    g = workloads.randn_bf16(tuple(t.shape), seed).float() * gain
    for b, n in enumerate(lens):
        t[b, :, n:] = g[b, :, n:].to(t.dtype)
    return t


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal", UNEQUAL)
def test_unequal_lengths(B, H, Nq, Nk, d, causal):
    q, k, v = _inputs(B, H, Nq, Nk, d, seed=Nq + 3 * Nk + d)
    scale = scale_for(d)
    o, lse = fa.forward_varlen(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale)
    fa.sync_status()
    o_ref, lse_ref = oracle.forward(to64(q), to64(k), to64(v), scale, causal)
    _check(o, lse, o_ref, lse_ref, (B, H, Nq, Nk, d, causal))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_padded_batch(causal, d):
    B, H, Nq, Nk = 5, 2, 300, 400
    sq, sk = PAD_SQ, PAD_SK
    q, k, v = _inputs(B, H, Nq, Nk, d, seed=40 + d)
    scale = scale_for(d)
    lq = torch.tensor(sq, dtype=torch.int32, device="cuda")
    lk = torch.tensor(sk, dtype=torch.int32, device="cuda")
    o, lse = fa.forward_varlen(q.cuda(), k.cuda(), v.cuda(), lq, lk, causal=causal, scale=scale)
    fa.sync_status()
    o_ref, lse_ref = oracle.forward_varlen(to64(q), to64(k), to64(v), scale, causal, sq, sk)
    _check(o, lse, o_ref, lse_ref, ("padded", causal, d))
    oc, lc = o.cpu(), lse.cpu()
    for b in range(B):
        assert torch.all(oc[b, :, sq[b]:] == 0) and torch.all(torch.isneginf(lc[b, :, sq[b]:]))
    # padding rows with large values (scores far past any LSE) change nothing
    q2, k2, v2 = _pad_garbage(q, sq, 30.0, 91), _pad_garbage(k, sk, 30.0, 92), _pad_garbage(v, sk, 30.0, 93)
    o2, lse2 = fa.forward_varlen(q2.cuda(), k2.cuda(), v2.cuda(), lq, lk, causal=causal, scale=scale)
    fa.sync_status()
    assert torch.allclose(o2.cpu(), oc, rtol=0, atol=1e-6)
    assert torch.equal(torch.isinf(lse2.cpu()), torch.isinf(lc))
    fin = torch.isfinite(lc)
    assert torch.allclose(lse2.cpu()[fin], lc[fin], rtol=0, atol=1e-5)


def _check_grads(got, ref, what):
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        g = g.cpu().double().numpy()
        assert np.all(np.isfinite(g)), (what, name)
        err = np.abs(g - r).max()
        assert err <= GRAD_MAX_ABS, (what, name, err)


def _check_delta(ws, rd, rd_abs, what):
    """The workspace ends holding D.  Rows with keys: within the fp32 bound
    of tests/helpers.py against the oracle's sum_j P_ij dP_ij (rd_abs: the
    oracle's row term for |dO| and |V|); padding and key-less rows: exactly 0."""
    got = ws.cpu().double().numpy().reshape(rd.shape)
    assert_row_term_close(got, rd, rd_abs, what)
    assert np.all(got[rd_abs == 0] == 0), what


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal", UNEQUAL)
def test_unequal_lengths_backward(B, H, Nq, Nk, d, causal):
    seed = 5 * Nq + Nk + d
    q, k, v = _inputs(B, H, Nq, Nk, d, seed=seed)
    do = workloads.randn_bf16((B, H, Nq, d), seed + 3)
    scale = scale_for(d)
    qc, kc, vc, doc = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = fa.forward_varlen(qc, kc, vc, causal=causal, scale=scale)
    ws = torch.empty(B * H * Nq, dtype=torch.float32, device="cuda")
    got = fa.backward_varlen(qc, kc, vc, o, lse, doc, causal=causal, scale=scale, workspace=ws)
    fa.sync_status()
    rq, rk, rv, rd = oracle.backward(to64(q), to64(k), to64(v), to64(do), scale, causal)
    rd_abs = oracle.backward(to64(q), to64(k), np.abs(to64(v)), np.abs(to64(do)), scale, causal)[3]
    _check_grads(got, (rq, rk, rv), (B, H, Nq, Nk, d, causal))
    _check_delta(ws, rd, rd_abs, (B, H, Nq, Nk, d, causal))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_padded_batch_backward(causal, d):
    B, H, Nq, Nk = 5, 2, 300, 400
    sq, sk = PAD_SQ, PAD_SK
    q, k, v = _inputs(B, H, Nq, Nk, d, seed=60 + d)
    do = workloads.randn_bf16((B, H, Nq, d), 64 + d)
    scale = scale_for(d)
    lq = torch.tensor(sq, dtype=torch.int32, device="cuda")
    lk = torch.tensor(sk, dtype=torch.int32, device="cuda")

    def run(q, k, v, do):
        qc, kc, vc, doc = q.cuda(), k.cuda(), v.cuda(), do.cuda()
        o, lse = fa.forward_varlen(qc, kc, vc, lq, lk, causal=causal, scale=scale)
        ws = torch.empty(B * H * Nq, dtype=torch.float32, device="cuda")
        g = fa.backward_varlen(qc, kc, vc, o, lse, doc, lq, lk, causal=causal, scale=scale, workspace=ws)
        fa.sync_status()
        return tuple(t.cpu() for t in g), ws

    got, ws = run(q, k, v, do)
    rq, rk, rv, rd = oracle.backward_varlen(to64(q), to64(k), to64(v), to64(do), scale, causal, sq, sk)
    rd_abs = oracle.backward_varlen(to64(q), to64(k), np.abs(to64(v)), np.abs(to64(do)), scale, causal, sq, sk)[3]
    _check_grads(got, (rq, rk, rv), ("padded", causal, d))
    _check_delta(ws, rd, rd_abs, ("padded", causal, d))
    dq, dk, dv = got
    for b in range(B):
        assert torch.all(dq[b, :, sq[b]:] == 0)
        assert torch.all(dk[b, :, sk[b]:] == 0) and torch.all(dv[b, :, sk[b]:] == 0)
    # large finite values in every padding row change nothing
    got2, _ = run(_pad_garbage(q, sq, 30.0, 95), _pad_garbage(k, sk, 30.0, 96), _pad_garbage(v, sk, 30.0, 97),
                  _pad_garbage(do, sq, 30.0, 98))
    for a, b in zip(got2, got):
        assert torch.allclose(a, b, rtol=0, atol=1e-5)


def test_square_call_equals_fa_fwd():
    q, k, v = _inputs(2, 2, 333, 333, 128, seed=77)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    for causal in (False, True):
        a = fa.forward(q, k, v, causal=causal)
        b = fa.forward_varlen(q, k, v, causal=causal)
        fa.sync_status()
        assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_square_call_equals_fa_bwd():
    q, k, v = _inputs(2, 2, 333, 333, 128, seed=78)
    do = workloads.randn_bf16((2, 2, 333, 128), 79)
    q, k, v, do = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    for causal in (False, True):
        o, lse = fa.forward(q, k, v, causal=causal)
        a = fa.backward(q, k, v, o, lse, do, causal=causal)
        b = fa.backward_varlen(q, k, v, o, lse, do, causal=causal)
        fa.sync_status()
        for x, y in zip(a, b):
            assert torch.equal(x, y)


@pytest.mark.parametrize("d,causal", [(128, True), (64, False)])
def test_padded_batch_longer_sequences(d, causal):
    """A padded batch of multi-tile sequences (lengths not multiples of 128,
    more keys than queries and the reverse), forward and backward, every
    head against the oracle."""
    B, H, Nq, Nk = 3, 2, 1500, 2100
    sq, sk = [1500, 901, 1279], [2100, 1800, 640]
    g = workloads.make_decode_inputs(B, H, Nq, Nk, d, seed=90 + d)
    do = workloads.randn_bf16((B, H, Nq, d), 93 + d)
    scale = scale_for(d)
    q, k, v, doc = g["q"].cuda(), g["k"].cuda(), g["v"].cuda(), do.cuda()
    lq = torch.tensor(sq, dtype=torch.int32, device="cuda")
    lk = torch.tensor(sk, dtype=torch.int32, device="cuda")
    o, lse = fa.forward_varlen(q, k, v, lq, lk, causal=causal, scale=scale)
    ws = torch.empty(B * H * Nq, dtype=torch.float32, device="cuda")
    got = fa.backward_varlen(q, k, v, o, lse, doc, lq, lk, causal=causal, scale=scale, workspace=ws)
    fa.sync_status()
    x = {n: to64(g[n]) for n in g}
    o_ref, lse_ref = oracle.forward_varlen(x["q"], x["k"], x["v"], scale, causal, sq, sk)
    _check(o, lse, o_ref, lse_ref, ("long padded", d, causal))
    rq, rk, rv, rd = oracle.backward_varlen(x["q"], x["k"], x["v"], to64(do), scale, causal, sq, sk)
    rd_abs = oracle.backward_varlen(x["q"], x["k"], np.abs(x["v"]), np.abs(to64(do)), scale, causal, sq, sk)[3]
    _check_grads(got, (rq, rk, rv), ("long padded", d, causal))
    _check_delta(ws, rd, rd_abs, ("long padded", d, causal))
