"""The fp64 oracle against facts fixed outside it (CPU only)."""

import math

import numpy as np
import pytest

import oracle
from tests import oracle_pins


@pytest.mark.parametrize("check", oracle_pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    check(oracle)


def test_online_restatement_matches_page_intermediates():
    """The running-maximum update of the tiled method, restated here for the
    two-tile example, passes through m=0, l=1, a=2 and then l=4/3, a=20/3,
    output 5; normalising each tile alone and averaging gives 4."""
    from fractions import Fraction
    g = oracle_pins._golden("two_tile_example.json")
    tiles = [(0.0, 2.0), (math.log(3.0), 6.0)]
    m, l, a = -math.inf, 0.0, 0.0
    seen = []
    for s, val in tiles:
        m_new = max(m, s)
        c = math.exp(m - m_new)
        l = c * l + math.exp(s - m_new)
        a = c * a + math.exp(s - m_new) * val
        m = m_new
        seen.append((m, l, a))
    assert seen[0] == (0.0, 1.0, 2.0)
    assert abs(seen[1][1] - float(Fraction(g["tile2"]["after"]["l"]))) < 1e-15
    assert abs(seen[1][2] - float(Fraction(g["tile2"]["after"]["a"]))) < 1e-15
    assert abs(a / l - 5.0) < 1e-15
    per_tile_average = sum(val for _, val in tiles) / len(tiles)
    assert per_tile_average == float(Fraction(g["per_tile_normalise_then_average"]))
    # raw exponentials without the max shift overflow at the shifted scores
    with np.errstate(over="ignore", invalid="ignore"):
        raw = np.exp(np.array([1000.0, 1000.0 + math.log(3.0)]))
        assert not np.isfinite((raw * np.array([2.0, 6.0])).sum() / raw.sum())


def test_fully_masked_row_defined():
    """A row with no eligible key gives O = 0 and LSE = -inf, never NaN."""
    from oracle import attention as A
    q = np.ones((3, 2))
    k = np.ones((3, 2))
    v = np.arange(6.0).reshape(3, 2)
    orig = A.eligible
    try:
        A.eligible = lambda nq, nk, causal: np.array([[False] * 3, [True, False, False], [True] * 3])
        o, lse = A.forward_head(q, k, v, 1.0, True)
    finally:
        A.eligible = orig
    assert np.all(o[0] == 0.0) and lse[0] == -np.inf
    assert np.all(np.isfinite(o))
    assert np.allclose(o[1], v[0])


def test_gradient_matches_torch_autograd():
    """The oracle's gradient equals torch's fp64 autograd of its own
    attention routine (an independent implementation)."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    q, k, v, do = (rng.standard_normal((2, 3, 33, 16)) for _ in range(4))
    scale = 0.25
    for causal in (False, True):
        o, lse = oracle.forward(q, k, v, scale, causal)
        dq, dk, dv, _ = oracle.backward(q, k, v, do, scale, causal)
        tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
        to = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=scale)
        to.backward(torch.tensor(do))
        assert np.max(np.abs(o - to.detach().numpy())) < 1e-12
        for ours, theirs in ((dq, tq), (dk, tk), (dv, tv)):
            assert np.max(np.abs(ours - theirs.grad.numpy())) < 1e-11
