"""Checks that pin the fp64 oracle to facts fixed outside itself.

Each ``check_*`` takes an oracle module and raises AssertionError when the
module disagrees with a fact the FlashAttention pages print, a closed form, an
invariant of the mathematics, or a brute-force high-precision evaluation.
``test_oracle.py`` runs them on the real oracle; ``test_oracle_mutants.py``
runs them on copies of the oracle with a planted mistake and expects a
failure, which shows that the pins would catch that kind of mistake.
"""

from __future__ import annotations

import functools
import json
import math
import os
from fractions import Fraction

import mpmath
import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _bf16_values(shape, seed):
    """Random values exactly representable in bf16 (and so in fp64/mpmath)."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(shape).astype(np.float32)
    bits = x.view(np.uint32)
    # round to nearest even on the top 16 bits
    rounded = ((bits.astype(np.uint64) + 0x7FFF + ((bits >> 16) & 1)) >> 16) << 16
    return rounded.astype(np.uint32).view(np.float32).astype(np.float64)


def _head(x):
    return x[None, None]


# ---------------------------------------------------------------- worked example

def check_two_tile_example(ora):
    """Scores (0, ln 3) with values (2, 6) give 5; the same under causal
    masking for the second query, and 2 for the first one."""
    g = _golden("two_tile_example.json")
    want = float(Fraction(g["output"]))
    q = _head(np.array([[1.0], [1.0]]))
    k = _head(np.array([[0.0], [math.log(3.0)]]))
    v = _head(np.array([[float(g["tile1"]["value"])], [float(g["tile2"]["value"])]]))
    o, lse = ora.forward(q, k, v, 1.0, False)
    assert abs(o[0, 0, 0, 0] - want) < 1e-13, o
    assert abs(o[0, 0, 1, 0] - want) < 1e-13, o
    assert abs(lse[0, 0, 0] - math.log(4.0)) < 1e-13, lse
    oc, lc = ora.forward(q, k, v, 1.0, True)
    assert abs(oc[0, 0, 0, 0] - 2.0) < 1e-13, oc
    assert abs(oc[0, 0, 1, 0] - want) < 1e-13, oc
    assert abs(lc[0, 0, 0] - 0.0) < 1e-13, lc
    # the full-softmax weights 1/4 and 3/4, recovered from the LSE
    w = [math.exp(s - lse[0, 0, 0]) for s in (0.0, math.log(3.0))]
    assert abs(w[0] - float(Fraction(g["full_softmax_weights"][0]))) < 1e-13
    assert abs(w[1] - float(Fraction(g["full_softmax_weights"][1]))) < 1e-13


def check_common_shift(ora):
    """Adding 1000 to both scores leaves the output at 5."""
    g = _golden("two_tile_example.json")
    shift = float(g["common_shift"])
    q = _head(np.array([[1.0], [1.0]]))
    k = _head(np.array([[shift], [shift + math.log(3.0)]]))
    v = _head(np.array([[2.0], [6.0]]))
    o, lse = ora.forward(q, k, v, 1.0, False)
    assert abs(o[0, 0, 0, 0] - float(Fraction(g["output_after_shift"]))) < 1e-12, o
    assert abs(lse[0, 0, 0] - (shift + math.log(4.0))) < 1e-12, lse


# ---------------------------------------------------------------- invariants

def _random_case(b, h, n, d, seed):
    shape = (b, h, n, d)
    return (_bf16_values(shape, seed), _bf16_values(shape, seed + 1),
            _bf16_values(shape, seed + 2), _bf16_values(shape, seed + 3))


def check_rows_sum_to_one(ora):
    """sum_j exp(s_ij - LSE_i) = 1 over eligible keys, with the scores formed
    here by an explicit loop over the feature index."""
    q, k, v, _ = _random_case(2, 2, 37, 8, 11)
    scale = 0.3
    for causal in (False, True):
        _, lse = ora.forward(q, k, v, scale, causal)
        s = np.zeros((2, 2, 37, 37))
        for c in range(8):
            s += q[..., :, None, c] * k[..., None, :, c]
        s *= scale
        if causal:
            s = np.where(np.tril(np.ones((37, 37), dtype=bool)), s, -np.inf)
        tot = np.exp(s - lse[..., None]).sum(-1)
        assert np.max(np.abs(tot - 1.0)) < 1e-12, (causal, np.max(np.abs(tot - 1.0)))


def check_equal_scores(ora):
    """Q = 0 makes every score equal: O is the mean of the eligible V rows
    (the prefix mean under causal masking) and LSE = ln(#eligible)."""
    n, d = 29, 6
    _, k, v, _ = _random_case(1, 2, n, d, 21)
    q = np.zeros_like(k)
    o, lse = ora.forward(q, k, v, 0.125, False)
    assert np.max(np.abs(o - v.mean(axis=2, keepdims=True))) < 1e-13
    assert np.max(np.abs(lse - math.log(n))) < 1e-13
    oc, lc = ora.forward(q, k, v, 0.125, True)
    counts = np.arange(1, n + 1, dtype=np.float64)
    prefix_mean = np.cumsum(v, axis=2) / counts[None, None, :, None]
    assert np.max(np.abs(oc - prefix_mean)) < 1e-13
    assert np.max(np.abs(lc - np.log(counts)[None, None, :])) < 1e-13


def check_causal_row0(ora):
    """Under the causal mask query 0 sees only key 0: O_0 = V_0 and
    LSE_0 = scale * <q_0, k_0>."""
    q, k, v, _ = _random_case(1, 3, 17, 8, 31)
    scale = 0.35355339059327373
    o, lse = ora.forward(q, k, v, scale, True)
    assert np.max(np.abs(o[:, :, 0] - v[:, :, 0])) < 1e-15
    s00 = scale * np.array([[sum(q[0, h, 0, c] * k[0, h, 0, c] for c in range(8)) for h in range(3)]])
    assert np.max(np.abs(lse[:, :, 0] - s00)) < 1e-14


def check_causal_is_prefix(ora):
    """Causal row i equals the non-causal answer on the first i+1 positions."""
    q, k, v, _ = _random_case(1, 1, 12, 4, 41)
    o, lse = ora.forward(q, k, v, 0.5, True)
    for i in (0, 1, 5, 11):
        oi, li = ora.forward(q[:, :, :i + 1], k[:, :, :i + 1], v[:, :, :i + 1], 0.5, False)
        assert np.max(np.abs(o[:, :, i] - oi[:, :, i])) < 1e-13
        assert abs(lse[0, 0, i] - li[0, 0, i]) < 1e-13


def check_backward_row_identity(ora):
    """sum_j P_ij dP_ij equals rowsum(dO * O) (the identity the backward's
    row term starts from), to fp64 rounding."""
    q, k, v, do = _random_case(1, 2, 23, 8, 51)
    for causal in (False, True):
        o, _ = ora.forward(q, k, v, 0.4, causal)
        _, _, _, dd = ora.backward(q, k, v, do, 0.4, causal)
        assert np.max(np.abs(dd - (do * o).sum(-1))) < 1e-12


def check_forward_rows_agree(ora):
    """The sampled-row evaluation equals the full evaluation on those rows."""
    q, k, v, _ = _random_case(2, 2, 19, 8, 61)
    rows = [(0, 0, 0), (0, 1, 18), (1, 0, 7), (1, 1, 11)]
    for causal in (False, True):
        o, lse = ora.forward(q, k, v, 0.3, causal)
        ro, rl = ora.forward_rows(q, k, v, 0.3, causal, rows)
        for r, (b, h, i) in enumerate(rows):
            assert np.max(np.abs(ro[r] - o[b, h, i])) < 1e-13
            assert abs(rl[r] - lse[b, h, i]) < 1e-13


# ---------------------------------------------------------------- brute force

def _mp_forward(q, k, v, scale, causal, bias=None):
    """Definition evaluated entry by entry in 50-digit arithmetic (one head).
    Causal keys of query i: 0 .. i + (nk - nq), the last query aligned with
    the last key; a query with no key gets O = 0 and LSE = -inf.  ``bias``
    (finite, [nq][nk]) is added to each scaled score."""
    nq, nk, d, dv = len(q), len(k), len(q[0]), len(v[0])
    o = [[mpmath.mpf(0)] * dv for _ in range(nq)]
    lse = [mpmath.mpf("-inf")] * nq
    for i in range(nq):
        keys = range(max(0, min(i + nk - nq + 1, nk))) if causal else range(nk)
        if len(keys) == 0:
            continue
        w = {}
        for j in keys:
            s = mpmath.mpf(0)
            for c in range(d):
                s += q[i][c] * k[j][c]
            w[j] = mpmath.exp(scale * s + (bias[i][j] if bias is not None else 0))
        tot = mpmath.fsum(w.values())
        lse[i] = mpmath.log(tot)
        for c in range(dv):
            o[i][c] = mpmath.fsum(w[j] * v[j][c] for j in keys) / tot
    return o, lse


def _to_mp(a):
    return [[mpmath.mpf(float(x)) for x in row] for row in a]


@functools.lru_cache(maxsize=None)
def _brute(nq, nk, d, causal, seed, with_bias=False):
    """50-digit forward values and central-difference gradients of
    sum(O * dO) for one random head with nq queries and nk keys (with a
    random finite additive mask when ``with_bias``)."""
    mpmath.mp.dps = 50
    q, do = (_bf16_values((nq, d), seed + t) for t in (0, 3))
    k, v = (_bf16_values((nk, d), seed + t) for t in (1, 2))
    bias = np.random.default_rng(seed + 9).standard_normal((nq, nk)) * 1.5 if with_bias else None
    B = _to_mp(bias) if with_bias else None
    scale = mpmath.mpf(1) / mpmath.sqrt(d)
    Q, K, V, DO = _to_mp(q), _to_mp(k), _to_mp(v), _to_mp(do)
    o, lse = _mp_forward(Q, K, V, scale, causal, B)

    def f(Q_, K_, V_):
        oo, _ = _mp_forward(Q_, K_, V_, scale, causal, B)
        return mpmath.fsum(oo[i][c] * DO[i][c] for i in range(nq) for c in range(d))

    h = mpmath.mpf("1e-18")
    grads = []
    for which, rows in ((0, nq), (1, nk), (2, nk)):
        g = np.zeros((rows, d))
        for i in range(rows):
            for c in range(d):
                mats = [[row[:] for row in M] for M in (Q, K, V)]
                x0 = mats[which][i][c]
                mats[which][i][c] = x0 + h
                fp = f(*mats)
                mats[which][i][c] = x0 - h
                fm = f(*mats)
                g[i, c] = float((fp - fm) / (2 * h))
        grads.append(g)
    o_np = np.array([[float(x) for x in row] for row in o])
    lse_np = np.array([float(x) for x in lse])
    return (q, k, v, do, float(scale), o_np, lse_np, bias) + tuple(grads)


def _check_brute(ora, nq, nk, d, causal, seed, with_bias=False):
    q, k, v, do, scale, o_ref, lse_ref, bias, dq_ref, dk_ref, dv_ref = _brute(nq, nk, d, causal, seed, with_bias)
    b4 = None if bias is None else bias[None, None]
    o, lse = ora.forward(_head(q), _head(k), _head(v), scale, causal, b4)
    assert np.max(np.abs(o[0, 0] - o_ref)) < 1e-13, np.max(np.abs(o[0, 0] - o_ref))
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lse[0, 0]), fin)
    assert np.max(np.abs(lse[0, 0][fin] - lse_ref[fin]), initial=0.0) < 1e-13
    dq, dk, dv, _ = ora.backward(_head(q), _head(k), _head(v), _head(do), scale, causal, b4)
    for got, ref in ((dq, dq_ref), (dk, dk_ref), (dv, dv_ref)):
        assert np.max(np.abs(got[0, 0] - ref)) < 1e-12, np.max(np.abs(got[0, 0] - ref))


def check_brute_force_4x4(ora):
    _check_brute(ora, 4, 4, 4, False, 101)
    _check_brute(ora, 4, 4, 4, True, 201)


def check_brute_force_8x8(ora):
    _check_brute(ora, 8, 8, 8, False, 301)
    _check_brute(ora, 8, 8, 8, True, 401)


def check_brute_force_unequal(ora):
    """Unequal query/key counts, both ways, with the bottom-right causal
    alignment (and one query row with no key when nq > nk)."""
    _check_brute(ora, 3, 5, 4, True, 501)
    _check_brute(ora, 5, 3, 4, True, 601)
    _check_brute(ora, 3, 5, 4, False, 701)


# ---------------------------------------------------------------- alignment

def check_decode_row(ora):
    """A single query against N keys (decoding) sees every key under the
    causal mask: it equals the unmasked answer, and the last row of a square
    causal problem."""
    q, k, v, _ = _random_case(1, 2, 40, 8, 801)
    last = q[:, :, -1:, :]
    oc, lc = ora.forward(last, k, v, 0.3, True)
    on, ln = ora.forward(last, k, v, 0.3, False)
    assert np.max(np.abs(oc - on)) < 1e-15 and np.max(np.abs(lc - ln)) < 1e-15
    osq, lsq = ora.forward(q, k, v, 0.3, True)
    assert np.max(np.abs(oc[:, :, 0] - osq[:, :, -1])) < 1e-13


def check_leading_rows_masked(ora):
    """With two more queries than keys the first two queries see no key
    (O = 0, LSE = -inf, no NaN), the third sees key 0 only (O = v_0,
    LSE = s_00) and the last sees every key."""
    _, k, v, _ = _random_case(1, 1, 6, 8, 901)
    q = _random_case(1, 1, 8, 8, 911)[0]
    o, lse = ora.forward(q, k, v, 0.5, True)
    assert np.all(o[0, 0, :2] == 0.0) and np.all(lse[0, 0, :2] == -np.inf)
    assert np.max(np.abs(o[0, 0, 2] - v[0, 0, 0])) < 1e-15
    s00 = 0.5 * sum(q[0, 0, 2, c] * k[0, 0, 0, c] for c in range(8))
    assert abs(lse[0, 0, 2] - s00) < 1e-14
    on, ln = ora.forward(q[:, :, -1:], k, v, 0.5, False)
    assert np.max(np.abs(o[0, 0, -1] - on[0, 0, 0])) < 1e-13
    dq, dk, dv, _ = ora.backward(q, k, v, _random_case(1, 1, 8, 8, 921)[0], 0.5, True)
    assert np.all(dq[0, 0, :2] == 0.0) and np.all(np.isfinite(dk)) and np.all(np.isfinite(dv))


def check_varlen_slices(ora):
    """A padded batch equals each sequence computed on its own valid rows;
    padding rows are O = 0, LSE = -inf and zero gradients."""
    q = _random_case(3, 2, 9, 4, 1001)[0]
    k, v = _random_case(3, 2, 7, 4, 1011)[1:3]
    do = _random_case(3, 2, 9, 4, 1021)[0]
    sq, sk = [9, 4, 6], [7, 7, 2]
    for causal in (False, True):
        o, lse = ora.forward_varlen(q, k, v, 0.4, causal, sq, sk)
        dq, dk, dv, _ = ora.backward_varlen(q, k, v, do, 0.4, causal, sq, sk)
        for b in range(3):
            ob, lb = ora.forward(q[b:b + 1, :, :sq[b]], k[b:b + 1, :, :sk[b]], v[b:b + 1, :, :sk[b]], 0.4, causal)
            assert np.max(np.abs(o[b, :, :sq[b]] - ob[0]), initial=0.0) < 1e-15
            assert np.array_equal(lse[b, :, :sq[b]], lb[0])
            assert np.all(o[b, :, sq[b]:] == 0.0) and np.all(lse[b, :, sq[b]:] == -np.inf)
            assert np.all(dq[b, :, sq[b]:] == 0.0) and np.all(dk[b, :, sk[b]:] == 0.0)
            assert np.all(dv[b, :, sk[b]:] == 0.0)


# ---------------------------------------------------------------- memory exercise

def check_memory_exercise(ora):
    g = _golden("memory_exercise.json")
    n, d, b = g["N"], g["d"], g["bytes_per_element"]
    mib = 1024 * 1024
    assert ora.score_matrix_payload_bytes(n, b) == g["score_matrix_MiB"] * mib
    assert ora.tensor_payload_bytes(n, d, b) == g["one_N_by_d_tensor_MiB"] * mib
    assert 4 * ora.tensor_payload_bytes(n, d, b) == g["q_k_v_and_output_MiB"] * mib
    assert ora.score_matrix_payload_bytes(n, b) // b == g["score_matrix_elements"]
    assert ora.tensor_payload_bytes(n, d, b) // b == g["q_sized_tensor_elements"]
    assert ora.score_matrix_payload_bytes(2 * n, b) == g["doubled_N_score_matrix_MiB"] * mib
    assert ora.tensor_payload_bytes(2 * n, d, b) == g["doubled_N_q_sized_tensor_MiB"] * mib
    assert ora.score_matrix_payload_bytes(8000, 1) == g["score_elements_8000_tokens"]
    assert ora.score_matrix_payload_bytes(64000, 1) == g["score_elements_64000_tokens"]


# ---------------------------------------------------------------- additive mask

def _bias_case(nq, nk, seed):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((1, 2, nq, nk)) * 2.0


def check_bias_zero_is_no_bias(ora):
    """A zero additive mask changes nothing, bit for bit."""
    q, k, v, _ = _random_case(1, 2, 11, 8, 61)
    for causal in (False, True):
        a = ora.forward(q, k, v, 0.3, causal)
        b = ora.forward(q, k, v, 0.3, causal, np.zeros((1, 2, 11, 11)))
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def check_bias_row_constant(ora):
    """A bias constant along each row cancels in the softmax: O is unchanged
    and LSE_i moves by exactly that constant."""
    q, k, v, _ = _random_case(1, 2, 9, 8, 62)
    c = np.random.default_rng(7).standard_normal((1, 2, 9)) * 3.0
    bias = np.broadcast_to(c[..., None], (1, 2, 9, 9)).copy()
    for causal in (False, True):
        o0, l0 = ora.forward(q, k, v, 0.4, causal)
        o1, l1 = ora.forward(q, k, v, 0.4, causal, bias)
        assert np.max(np.abs(o1 - o0)) < 1e-13
        assert np.max(np.abs(l1 - (l0 + c))) < 1e-12


def check_bias_masks_like_causal(ora):
    """A bias of 0 on eligible keys and -inf elsewhere, without the causal
    rule, is the causal rule (unequal lengths, bottom-right alignment)."""
    rng = np.random.default_rng(63)
    q = rng.standard_normal((1, 1, 6, 4))
    k, v = rng.standard_normal((2, 1, 1, 9, 4))
    i = np.arange(6)[:, None]
    j = np.arange(9)[None, :]
    bias = np.where(j <= i + 3, 0.0, -np.inf)[None, None]
    a = ora.forward(q, k, v, 0.5, True)
    b = ora.forward(q, k, v, 0.5, False, bias)
    assert np.max(np.abs(a[0] - b[0])) < 1e-14 and np.max(np.abs(a[1] - b[1])) < 1e-14


def check_bias_fully_hidden_row(ora):
    """A row whose keys the mask hides entirely: O = 0, LSE = -inf, no NaN;
    other rows as without that row's mask."""
    q, k, v, _ = _random_case(1, 1, 5, 4, 64)
    bias = np.zeros((1, 1, 5, 5))
    bias[0, 0, 2, :] = -np.inf
    o, lse = ora.forward(q, k, v, 0.5, False, bias)
    assert np.all(o[0, 0, 2] == 0) and lse[0, 0, 2] == -np.inf and np.all(np.isfinite(o))
    o0, l0 = ora.forward(q, k, v, 0.5, False)
    keep = [0, 1, 3, 4]
    assert np.max(np.abs(o[0, 0, keep] - o0[0, 0, keep])) < 1e-15


def check_brute_force_bias(ora):
    """Random bias on a 4-query x 6-key head, causal, against the definition
    in 50-digit arithmetic."""
    mpmath.mp.dps = 50
    q = _bf16_values((4, 4), 71)
    k, v = (_bf16_values((6, 4), 72 + t) for t in range(2))
    bias = np.random.default_rng(73).standard_normal((4, 6)) * 1.5
    scale = 0.5
    o_ref, lse_ref = _mp_forward(_to_mp(q), _to_mp(k), _to_mp(v), mpmath.mpf(scale), True,
                                 [[mpmath.mpf(float(x)) for x in row] for row in bias])
    o, lse = ora.forward(_head(q), _head(k), _head(v), scale, True, bias[None, None])
    o_ref = np.array([[float(x) for x in row] for row in o_ref])
    lse_ref = np.array([float(x) for x in lse_ref])
    assert np.max(np.abs(o[0, 0] - o_ref)) < 1e-13
    assert np.max(np.abs(lse[0, 0] - lse_ref)) < 1e-13


def check_brute_force_bias_gradients(ora):
    """Gradients under a random additive mask against 50-digit central
    differences of the masked definition (causal and not, unequal lengths)."""
    _check_brute(ora, 4, 6, 4, True, 801, with_bias=True)
    _check_brute(ora, 5, 5, 4, False, 901, with_bias=True)


def check_bias_backward_masks_like_causal(ora):
    """Gradients under a 0 / -inf mask shaped like the causal rule equal the
    causal gradients (padded batch, bottom-right alignment)."""
    rng = np.random.default_rng(67)
    q, do = rng.standard_normal((2, 1, 1, 6, 4))
    k, v = rng.standard_normal((2, 1, 1, 9, 4))
    i = np.arange(6)[:, None]
    j = np.arange(9)[None, :]
    bias = np.where(j <= i + 3, 0.0, -np.inf)[None, None]
    a = ora.backward(q, k, v, do, 0.5, True)
    b = ora.backward(q, k, v, do, 0.5, False, bias)
    for x, y in zip(a, b):
        assert np.max(np.abs(x - y)) < 1e-13
    lq, lk = [5], [7]
    bias_v = np.where(j <= i + 2, 0.0, -np.inf)[None, None]
    a = ora.backward_varlen(q, k, v, do, 0.5, True, lq, lk)
    b = ora.backward_varlen(q, k, v, do, 0.5, False, lq, lk, bias_v)
    for x, y in zip(a, b):
        assert np.max(np.abs(x - y)) < 1e-13


def check_bias_backward_hidden_row(ora):
    """A row the mask hides entirely has zero gradient and adds nothing to
    dK and dV."""
    q, k, v, do = _random_case(1, 1, 5, 4, 68)
    bias = np.random.default_rng(69).standard_normal((1, 1, 5, 5))
    bias[0, 0, 3, :] = -np.inf
    dq, dk, dv, dd = ora.backward(q, k, v, do, 0.5, False, bias)
    assert np.all(dq[0, 0, 3] == 0) and dd[0, 0, 3] == 0
    keep = [0, 1, 2, 4]
    dq2, dk2, dv2, _ = ora.backward(q[:, :, keep], k, v, do[:, :, keep], 0.5, False, bias[:, :, keep])
    assert np.max(np.abs(dk - dk2)) < 1e-14 and np.max(np.abs(dv - dv2)) < 1e-14
    assert np.max(np.abs(dq[0, 0, keep] - dq2[0, 0])) < 1e-14


def check_forward_rows_with_bias(ora):
    """The row sampler sees the same bias as the full forward."""
    q, k, v, _ = _random_case(2, 2, 13, 8, 65)
    bias = np.random.default_rng(66).standard_normal((2, 2, 13, 13))
    bias[1, 0, 4, :3] = -np.inf
    rows = [(0, 0, 0), (1, 0, 4), (1, 1, 12), (0, 1, 7)]
    for causal in (False, True):
        o, lse = ora.forward(q, k, v, 0.35, causal, bias)
        ro, rl = ora.forward_rows(q, k, v, 0.35, causal, rows, bias)
        for r, (b_, h_, i_) in enumerate(rows):
            assert np.max(np.abs(ro[r] - o[b_, h_, i_])) < 1e-13
            assert abs(rl[r] - lse[b_, h_, i_]) < 1e-13


ALL_CHECKS = [
    check_two_tile_example,
    check_common_shift,
    check_rows_sum_to_one,
    check_equal_scores,
    check_causal_row0,
    check_causal_is_prefix,
    check_backward_row_identity,
    check_forward_rows_agree,
    check_brute_force_4x4,
    check_brute_force_8x8,
    check_brute_force_unequal,
    check_decode_row,
    check_leading_rows_masked,
    check_varlen_slices,
    check_memory_exercise,
    check_bias_zero_is_no_bias,
    check_bias_row_constant,
    check_bias_masks_like_causal,
    check_bias_fully_hidden_row,
    check_brute_force_bias,
    check_forward_rows_with_bias,
    check_brute_force_bias_gradients,
    check_bias_backward_masks_like_causal,
    check_bias_backward_hidden_row,
]


def failing_checks(ora):
    """Names of the checks the given oracle module fails."""
    bad = []
    for chk in ALL_CHECKS:
        try:
            with np.errstate(all="ignore"):
                chk(ora)
        except Exception:  # AssertionError, or a crash caused by the mutation
            bad.append(chk.__name__)
    return bad
