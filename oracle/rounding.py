"""Rounding companion of the fp64 oracle -- test infrastructure, not the product.

Like ``attention.py`` this module may be imported only by the test suite, the
smoke check and the CPU-baseline leg of ``bench.py``; it shares no code with
the CUDA path.

Parity is graded against the plain definition in ``attention.py``.  This
module answers a different question: how large an error does the rounding
that the method itself prescribes leave?  The FlashAttention pages feed the
tensor-core products bf16 operands ("FlashAttention Interview Questions",
section "What is FlashAttention exact about?": exact means the same
mathematical function, not bitwise equality), so the probabilities P enter
O = P V and dV = P^T dO rounded to bf16, and dS enters dQ = dS K rounded to
bf16.  Here the definition is evaluated in fp64 with exactly those operands
rounded (to fp32, then to bf16 with round-to-nearest-even) and nothing else:
the softmax normaliser l, the row term D and dK (whose dS the kernels carry
as a hi + lo pair, about 16 significant bits) stay in fp64.  The dQ operand
is the one the recomputation backward rounds: dS formed with the row term
of the rounded forward output, whose difference from the exact row term is
then taken out again in fp64.

The FP8 forward takes its inputs as E4M3 values and rounds P to E4M3 before
O = P V; ``forward(..., p_round=round_e4m3)`` is its companion, the plain
definition applied to those input values its parity reference.

A kernel result much closer to this prediction than to the definition shows
that its error is the prescribed rounding rather than a defect.  The kernels
round P relative to a running reference maximum that may lag the row maximum
(by less than 2^8 in the weights), so their rounding points differ from these
in detail, not in size.
"""

from __future__ import annotations

import numpy as np

from . import attention

__all__ = ["round_bf16", "round_e4m3", "forward_head", "forward", "backward_head", "backward"]


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round to the nearest bf16 value (ties to even), returned as float64.

    bf16 is the top half of an IEEE binary32 word: the value is first
    rounded to float32, then the low 16 bits are rounded away, the carry
    going into the kept bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).astype(np.float64).reshape(np.shape(x))


def round_e4m3(x: np.ndarray) -> np.ndarray:
    """Round to the nearest FP8 E4M3 value (ties to even), saturating at
    +-448, returned as float64.

    E4M3: 1 sign, 4 exponent bits (bias 7), 3 mantissa bits, no infinities.
    Normal values 1.mmm * 2^e for e >= -6 (largest 1.75 * 2^8 = 448);
    below 2^-6 the subnormals 0.mmm * 2^-6, spacing 2^-9.  So a value in the
    binade [2^e, 2^(e+1)) rounds on a grid of spacing 2^(e-3), with e held
    at -6 for the subnormal range."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, e = np.frexp(a)                      # a = f * 2^e, f in [0.5, 1): binade exponent e - 1
    e = np.maximum(e.astype(np.float64) - 1.0, -6.0)
    step = np.exp2(e - 3.0)
    r = np.minimum(np.round(a / step) * step, 448.0)   # np.round: half to even
    return np.copysign(r, x)


def forward_head(q, k, v, scale, causal, bias=None, p_round=None):
    """attention.forward_head with the weights rounded before the product
    with V (the normaliser l is the sum of the unrounded weights): to bf16
    by default, or by ``p_round`` (round_e4m3 for the FP8 forward)."""
    p_round = round_bf16 if p_round is None else p_round
    s, ok = attention._masked_scores(q, k, scale, causal, bias)
    has_key = ok.any(axis=1)
    m = np.where(has_key, s.max(axis=1, initial=-np.inf), 0.0)
    w = np.where(ok, np.exp(s - m[:, None]), 0.0)
    l = w.sum(axis=1)
    safe_l = np.where(has_key, l, 1.0)
    o = (p_round(w) @ v) / safe_l[:, None]
    o[~has_key] = 0.0
    lse = np.where(has_key, m + np.log(safe_l), -np.inf)
    return o, lse


def forward(q, k, v, scale, causal, bias=None, p_round=None):
    """forward_head over [B, H, N, d] arrays; returns (O, LSE)."""
    b, h, nq, _ = q.shape
    o = np.empty((b, h, nq, v.shape[-1]), dtype=np.float64)
    lse = np.empty((b, h, nq), dtype=np.float64)
    for bi in range(b):
        for hi in range(h):
            o[bi, hi], lse[bi, hi] = forward_head(q[bi, hi], k[bi, hi], v[bi, hi], scale, causal,
                                                  None if bias is None else bias[bi, hi], p_round)
    return o, lse


def backward_head(q, k, v, do, scale, causal, bias=None):
    """attention.backward_head with P rounded to bf16 in dV = P^T dO, and dQ
    formed the way the recomputation backward forms it from a rounded
    forward output: the row term first comes in as D'_i = sum_c dO_ic O_ic
    with O from ``forward_head`` above (whose P was rounded), dS'_ij =
    P_ij (dP_ij - D'_i) enters the product rounded to bf16, and the
    difference is taken out again exactly:
    dQ_i = scale (sum_j bf16(dS'_ij) k_j - delta_i sum_j P_ij k_j)
    with delta_i = sum_j dS'_ij.  D and dK from the unrounded values.
    Returns (dQ, dK, dV, D)."""
    s, ok = attention._masked_scores(q, k, scale, causal, bias)
    _, lse = attention.forward_head(q, k, v, scale, causal, bias)
    o_rounded, _ = forward_head(q, k, v, scale, causal, bias)
    has_key = np.isfinite(lse)
    p = np.where(ok & has_key[:, None], np.exp(s - np.where(has_key, lse, 0.0)[:, None]), 0.0)
    dv = round_bf16(p).T @ do
    dp = do @ v.T
    dd = (p * dp).sum(axis=1)
    ds = p * (dp - dd[:, None])
    d_out = np.where(has_key, (do * o_rounded).sum(axis=1), 0.0)
    ds_out = p * (dp - d_out[:, None])
    delta = ds_out.sum(axis=1)
    dq = scale * (round_bf16(ds_out) @ k - delta[:, None] * (p @ k))
    dk = scale * (ds.T @ q)
    return dq, dk, dv, dd


def backward(q, k, v, do, scale, causal, bias=None):
    """backward_head over [B, H, N, d] arrays; returns (dQ, dK, dV, D)."""
    b, h, n, d = q.shape
    dq = np.empty(q.shape, dtype=np.float64)
    dk = np.empty(k.shape, dtype=np.float64)
    dv = np.empty(v.shape, dtype=np.float64)
    dd = np.empty((b, h, n), dtype=np.float64)
    for bi in range(b):
        for hi in range(h):
            dq[bi, hi], dk[bi, hi], dv[bi, hi], dd[bi, hi] = backward_head(
                q[bi, hi], k[bi, hi], v[bi, hi], do[bi, hi], scale, causal, None if bias is None else bias[bi, hi])
    return dq, dk, dv, dd
