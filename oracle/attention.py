"""fp64 CPU oracle for exact scaled-dot-product attention and its gradient.

TEST INFRASTRUCTURE ONLY.  This module is the checker, not the product: only the
test suite, the smoke check in ``__graft_entry__`` and the CPU-baseline leg of
``bench.py`` may import it.  It shares no code with the CUDA path and never
touches a GPU.

What it computes is the plain definition of attention, written out with numpy
fp64 matrix products as the only library step; there is no tiling, no running
maximum and no reordering.  Sources (the three FlashAttention pages):

* "FlashAttention Interview Questions: IO Complexity, Tiling, and Numerical
  Stability", section "What is FlashAttention exact about?": per head,
  scores = Q K^T / sqrt(d), weights = row_softmax(scores + mask),
  output = weights V.  The method is exact, so the oracle is this definition.
* "FlashAttention 1, 2 & 3: Memory Tiling ...", section 1 "The Standard
  Attention Memory Bottleneck": Attention(Q,K,V) = softmax(QK^T/sqrt(d)) V.
* Same FlashAttention Interview Questions page, section "Does subtracting the
  maximum solve every numerical issue?": a row whose keys are all masked has
  no softmax distribution; the behaviour must be defined.  Defined here as
  O_i = 0 and LSE_i = -inf (no NaN).
* Same page, section "Why can recomputation help training?": the backward pass
  works from the saved normalisation (the log-sum-exp) and the gradients must
  be validated.  The gradient below is the textbook chain rule of the
  definition above; nothing of the tiled backward is used.

Readings where the pages are silent (each is also a test pin or an argument):

* tensors are [B, H, N, d], one (b, h) pair is one head, queries and keys have
  the same length N;
* the mask is either none or causal; with Nq queries and Nk keys, causal key
  j is eligible for query i iff j <= i + (Nk - Nq): the last query sits at the
  last key ("Do not infer the correct causal mask solely from a square
  training example" -- same page, section "Does subtracting the maximum solve
  every numerical issue?").  For Nq == Nk this is j <= i; one query (decoding)
  sees every key; if Nq > Nk the first Nq - Nk queries see none;
* padded batches carry a valid length per sequence; rows past it are padding
  and are defined as O = 0, LSE = -inf (gradients 0);
* the "+ mask" of the definition, in general form, is an additive bias
  B_ij on the scaled scores (s_ij = scale * q_i.k_j + B_ij), -inf entries
  hiding a key; it combines with the causal rule, and a row whose keys are
  all hidden is a fully masked row (O = 0, LSE = -inf);
* the log-sum-exp is in natural-log units of the scaled scores:
  LSE_i = ln sum_j exp(s_ij) over eligible j;
* ``scale`` is an argument (the pages' 1/sqrt(d) is the caller's default);
* D_i, the row term of the backward pass, is computed as sum_j P_ij dP_ij
  (its definition through the chain rule), not as rowsum(dO * O).

Every function takes float64 numpy arrays; callers widen their bf16 inputs to
float64 before calling, so the oracle sees exactly the values the kernels see.
"""

from __future__ import annotations

import math

import numpy as np

__all__ = [
    "scores",
    "eligible",
    "forward_head",
    "forward",
    "forward_rows",
    "forward_varlen",
    "backward_head",
    "backward",
    "backward_varlen",
    "score_matrix_payload_bytes",
    "tensor_payload_bytes",
]


def scores(q: np.ndarray, k: np.ndarray, scale: float) -> np.ndarray:
    """s_ij = scale * <q_i, k_j> for one head (q: [Nq, d], k: [Nk, d])."""
    return scale * (q @ k.T)


def eligible(nq: int, nk: int, causal: bool) -> np.ndarray:
    """Boolean [Nq, Nk] matrix: True where key j may be seen by query i.

    Non-causal: every key.  Causal: j <= i + (nk - nq), the last query aligned
    with the last key (for square sequences query i and key i are the same
    position).
    """
    if not causal:
        return np.ones((nq, nk), dtype=bool)
    i = np.arange(nq)[:, None]
    j = np.arange(nk)[None, :]
    return j <= i + (nk - nq)


def _masked_scores(q, k, scale, causal, bias=None):
    s = scores(q, k, scale)
    ok = eligible(q.shape[0], k.shape[0], causal)
    if bias is not None:
        s = s + bias
        ok = ok & (bias > -np.inf)
    return np.where(ok, s, -np.inf), ok


def forward_head(q, k, v, scale, causal, bias=None):
    """One head of softmax(scale * q k^T + mask) v; ``bias`` ([Nq, Nk] or
    None) is the additive mask, on top of the causal rule.

    Returns (O [N, d], LSE [N]) in float64.  The row maximum is subtracted
    before exponentiating only so that exp() cannot overflow; the result is
    the same number the definition gives (softmax is shift invariant).
    """
    s, ok = _masked_scores(q, k, scale, causal, bias)
    has_key = ok.any(axis=1)
    m = np.where(has_key, s.max(axis=1, initial=-np.inf), 0.0)
    w = np.where(ok, np.exp(s - m[:, None]), 0.0)  # unnormalised weights
    l = w.sum(axis=1)
    safe_l = np.where(has_key, l, 1.0)
    o = (w @ v) / safe_l[:, None]
    o[~has_key] = 0.0
    lse = np.where(has_key, m + np.log(safe_l), -np.inf)
    return o, lse


def forward(q, k, v, scale, causal, bias=None):
    """Attention over [B, H, N, d] arrays; returns (O [B,H,N,d], LSE [B,H,N]).
    ``bias``: None or [B, H, Nq, Nk] additive mask."""
    b, h, n, d = q.shape
    o = np.empty((b, h, n, v.shape[-1]), dtype=np.float64)
    lse = np.empty((b, h, n), dtype=np.float64)
    for bi in range(b):
        for hi in range(h):
            o[bi, hi], lse[bi, hi] = forward_head(q[bi, hi], k[bi, hi], v[bi, hi], scale, causal,
                                                  None if bias is None else bias[bi, hi])
    return o, lse


def forward_rows(q, k, v, scale, causal, rows, bias=None):
    """O and LSE for selected query rows only.

    ``rows`` is a sequence of (b, h, i) triples.  Each row is the definition
    evaluated for that one query against every eligible key of its head, so a
    long sequence can be checked on a sample without the N x N matrix.
    ``bias``: None or [B, H, Nq, Nk] additive mask.  Returns (O [R, d], LSE [R]).
    """
    out_o = np.empty((len(rows), v.shape[-1]), dtype=np.float64)
    out_l = np.empty(len(rows), dtype=np.float64)
    nq, nk_all = q.shape[2], k.shape[2]
    for r, (bi, hi, i) in enumerate(rows):
        count = min(i + (nk_all - nq) + 1, nk_all) if causal else nk_all
        if count <= 0:
            out_o[r] = 0.0
            out_l[r] = -np.inf
            continue
        kk = k[bi, hi, :count]
        vv = v[bi, hi, :count]
        s = scale * (kk @ q[bi, hi, i])
        if bias is not None:
            s = s + bias[bi, hi, i, :count]
        if not np.any(s > -np.inf):
            out_o[r] = 0.0
            out_l[r] = -np.inf
            continue
        m = s.max()
        w = np.exp(s - m)  # hidden keys (s = -inf) give 0
        l = w.sum()
        out_o[r] = (w @ vv) / l
        out_l[r] = m + math.log(l)
    return out_o, out_l


def forward_varlen(q, k, v, scale, causal, seqlens_q, seqlens_k, bias=None):
    """Padded batch: sequence b uses its first seqlens_q[b] query rows and
    seqlens_k[b] key rows of q [B,H,Nq,d] and k, v [B,H,Nk,d] (and the
    matching corner of bias [B,H,Nq,Nk]).  Padding rows are O = 0,
    LSE = -inf.  Returns (O [B,H,Nq,d], LSE [B,H,Nq])."""
    b, h, nq, _ = q.shape
    o = np.zeros((b, h, nq, v.shape[-1]), dtype=np.float64)
    lse = np.full((b, h, nq), -np.inf, dtype=np.float64)
    for bi in range(b):
        lq, lk = int(seqlens_q[bi]), int(seqlens_k[bi])
        for hi in range(h):
            o[bi, hi, :lq], lse[bi, hi, :lq] = forward_head(q[bi, hi, :lq], k[bi, hi, :lk], v[bi, hi, :lk],
                                                            scale, causal,
                                                            None if bias is None else bias[bi, hi, :lq, :lk])
    return o, lse


def backward_head(q, k, v, do, scale, causal, lse=None, bias=None):
    """Gradient of sum(O * dO) with respect to q, k, v for one head.

    Chain rule of the definition, with P_ij = exp(s_ij - LSE_i) and s_ij the
    masked score (scale * q_i.k_j plus the additive ``bias`` [Nq, Nk] when
    given; the bias is a constant of the differentiation):
      dV_j  = sum_i P_ij dO_i
      dP_ij = <dO_i, v_j>
      D_i   = sum_j P_ij dP_ij
      dS_ij = P_ij (dP_ij - D_i)
      dQ_i  = scale * sum_j dS_ij k_j
      dK_j  = scale * sum_i dS_ij q_i
    Returns (dQ, dK, dV, D).
    """
    s, ok = _masked_scores(q, k, scale, causal, bias)
    if lse is None:
        _, lse = forward_head(q, k, v, scale, causal, bias)
    has_key = np.isfinite(lse)
    p = np.where(ok & has_key[:, None], np.exp(s - np.where(has_key, lse, 0.0)[:, None]), 0.0)
    dv = p.T @ do
    dp = do @ v.T
    dd = (p * dp).sum(axis=1)
    ds = p * (dp - dd[:, None])
    dq = scale * (ds @ k)
    dk = scale * (ds.T @ q)
    return dq, dk, dv, dd


def backward(q, k, v, do, scale, causal, bias=None):
    """Gradients over [B, H, N, d] arrays (``bias``: None or [B, H, Nq, Nk]
    additive mask); returns (dQ, dK, dV, D)."""
    b, h, n, d = q.shape
    dq = np.empty_like(q, dtype=np.float64)
    dk = np.empty_like(k, dtype=np.float64)
    dv = np.empty_like(v, dtype=np.float64)
    dd = np.empty((b, h, n), dtype=np.float64)
    for bi in range(b):
        for hi in range(h):
            dq[bi, hi], dk[bi, hi], dv[bi, hi], dd[bi, hi] = backward_head(
                q[bi, hi], k[bi, hi], v[bi, hi], do[bi, hi], scale, causal,
                bias=None if bias is None else bias[bi, hi])
    return dq, dk, dv, dd


def backward_varlen(q, k, v, do, scale, causal, seqlens_q, seqlens_k, bias=None):
    """Gradients of a padded batch (see forward_varlen; ``bias`` as there);
    padding rows of dQ, dK, dV and D are 0.  Returns (dQ, dK, dV, D)."""
    b, h, nq, _ = q.shape
    dq = np.zeros(q.shape, dtype=np.float64)
    dk = np.zeros(k.shape, dtype=np.float64)
    dv = np.zeros(v.shape, dtype=np.float64)
    dd = np.zeros((b, h, nq), dtype=np.float64)
    for bi in range(b):
        lq, lk = int(seqlens_q[bi]), int(seqlens_k[bi])
        for hi in range(h):
            gq, gk, gv, gd = backward_head(q[bi, hi, :lq], k[bi, hi, :lk], v[bi, hi, :lk], do[bi, hi, :lq],
                                           scale, causal,
                                           bias=None if bias is None else bias[bi, hi, :lq, :lk])
            dq[bi, hi, :lq], dk[bi, hi, :lk], dv[bi, hi, :lk], dd[bi, hi, :lq] = gq, gk, gv, gd
    return dq, dk, dv, dd


def score_matrix_payload_bytes(n: int, bytes_per_element: int) -> int:
    """Payload of one N x N score matrix (FlashAttention Interview Questions
    page, section "Which complexity becomes smaller, and which does not?",
    memory-budget table)."""
    return n * n * bytes_per_element


def tensor_payload_bytes(n: int, d: int, bytes_per_element: int) -> int:
    """Payload of one N x d tensor such as Q (same table)."""
    return n * d * bytes_per_element
