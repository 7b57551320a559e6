"""Pins of the rounding companion of the oracle (CPU only)."""

import numpy as np
import torch

import oracle
from oracle import rounding


def _case(b, h, n, d, seed, boost=False):
    rng = np.random.default_rng(seed)
    x = [rng.standard_normal((b, h, n, d)) for _ in range(4)]
    if boost:
        x[0][:, :, ::8] *= 10.0
    return [rounding.round_bf16(t) for t in x]


def test_round_bf16_matches_torch_cast():
    """Against torch's float32 -> bfloat16 cast, including exact ties, both
    parities of the kept bit, carries into the exponent, tiny and huge
    values."""
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000)).astype(np.float32)
    u = x.view(np.uint32).copy()
    u[:5000] = (u[:5000] & 0xFFFF0000) | 0x8000          # exact ties
    u[5000:6000] = (u[5000:6000] | 0x007F0000) | 0x8001  # carries into the exponent
    x = u.view(np.float32)
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(rounding.round_bf16(x.astype(np.float64)), ref.astype(np.float64))


def test_without_rounding_it_is_the_definition(monkeypatch):
    q, k, v, do = _case(1, 2, 37, 8, 2)
    monkeypatch.setattr(rounding, "round_bf16", lambda x: np.asarray(x, dtype=np.float64))
    for causal in (False, True):
        a, b = rounding.forward(q, k, v, 0.3, causal), oracle.forward(q, k, v, 0.3, causal)
        assert np.max(np.abs(a[0] - b[0])) < 1e-13 and np.max(np.abs(a[1] - b[1])) < 1e-13
        ga, gb = rounding.backward(q, k, v, do, 0.3, causal), oracle.backward(q, k, v, do, 0.3, causal)
        for x, y in zip(ga, gb):
            assert np.max(np.abs(x - y)) < 1e-12


def test_forward_rounding_error_within_its_bound():
    """|bf16(w) - w| <= 2^-8 w, so |dO_i| <= 2^-8 sum_j P_ij |v_j|: checked
    elementwise, with P and sum_j P_ij |v_j| from the definition (the oracle
    applied to |v|)."""
    q, k, v, _ = _case(1, 2, 64, 16, 3, boost=True)
    for causal in (False, True):
        o, lse = oracle.forward(q, k, v, 0.5, causal)
        oe, lsee = rounding.forward(q, k, v, 0.5, causal)
        mass, _ = oracle.forward(q, k, np.abs(v), 0.5, causal)
        err = np.abs(oe - o)
        assert np.all(err <= 2.0 ** -8 * mass + 1e-15) and err.max() > 0
        assert np.array_equal(lse, lsee)


def test_backward_rounding_error_within_its_bound():
    """dV: |d(dV_j)| <= 2^-8 sum_i P_ij |dO_i| (the oracle's dV for |dO|);
    dQ: |d(dQ_i)| <= 2^-8 scale sum_j |dS'_ij| |k_j|, dS' formed with the
    row term of the rounded forward output; dK and D unrounded."""
    q, k, v, do = _case(1, 1, 48, 8, 4, boost=True)
    scale = 0.5
    for causal in (False, True):
        dq, dk, dv, dd = oracle.backward(q, k, v, do, scale, causal)
        eq, ek, ev, ed = rounding.backward(q, k, v, do, scale, causal)
        mass_v = oracle.backward(q, k, v, np.abs(do), scale, causal)[2]
        assert np.all(np.abs(ev - dv) <= 2.0 ** -8 * mass_v + 1e-14) and np.abs(ev - dv).max() > 0
        s = scale * (q[0, 0] @ k[0, 0].T)
        ok = oracle.eligible(48, 48, causal)
        _, lse = oracle.forward(q, k, v, scale, causal)
        p = np.where(ok, np.exp(np.where(ok, s, -np.inf) - lse[0, 0][:, None]), 0.0)
        o_r, _ = rounding.forward(q, k, v, scale, causal)
        d_out = (do[0, 0] * o_r[0, 0]).sum(axis=1)
        ds_out = p * ((do[0, 0] @ v[0, 0].T) - d_out[:, None])
        bound_q = 2.0 ** -8 * scale * (np.abs(ds_out) @ np.abs(k[0, 0]))
        assert np.all(np.abs(eq[0, 0] - dq[0, 0]) <= bound_q + 1e-13) and np.abs(eq - dq).max() > 0
        assert np.max(np.abs(ek - dk)) < 1e-13 and np.max(np.abs(ed - dd)) < 1e-13


def test_round_e4m3_matches_torch_cast():
    """Against torch's float32 -> float8_e4m3fn cast over the E4M3 range:
    every representable value, the midpoints between neighbours (ties to
    even), subnormals, and random values."""
    grid = np.unique(torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float32).numpy())
    grid = grid[np.isfinite(grid)]
    mids = (grid[:-1] + grid[1:]) / 2
    rng = np.random.default_rng(5)
    rand = (rng.standard_normal(20000) * 2.0 ** rng.integers(-12, 9, 20000)).astype(np.float32)
    x = np.concatenate([grid, mids, rand]).astype(np.float32)
    x = x[np.abs(x) <= 448]
    ref = torch.from_numpy(x.copy()).to(torch.float8_e4m3fn).to(torch.float32).numpy().astype(np.float64)
    assert np.array_equal(rounding.round_e4m3(x.astype(np.float64)), ref)
    assert rounding.round_e4m3(np.array([500.0, -1e6]))[0] == 448 and rounding.round_e4m3(np.array([-1e6]))[0] == -448


def test_fp8_forward_error_within_its_bound():
    """|e4m3(w) - w| <= 2^-4 w + 2^-10 (relative half-spacing of 3 mantissa
    bits; half the subnormal spacing), so with the weights w_ij = P_ij e^(LSE_i
    - m_i) <= 1, |dO_i| <= 2^-4 sum_j P_ij |v_j| + 2^-10 e^(m_i - LSE_i) sum_j |v_j|."""
    q, k, v, _ = _case(1, 2, 64, 16, 6, boost=True)
    q, k, v = (rounding.round_e4m3(t) for t in (q, k, v))
    for causal in (False, True):
        o, lse = oracle.forward(q, k, v, 0.5, causal)
        oe, lsee = rounding.forward(q, k, v, 0.5, causal, p_round=rounding.round_e4m3)
        mass, _ = oracle.forward(q, k, np.abs(v), 0.5, causal)
        s = 0.5 * np.einsum("bhid,bhjd->bhij", q, k)
        ok = oracle.eligible(64, 64, causal)
        m = np.where(ok, s, -np.inf).max(axis=-1)
        vsum = np.einsum("ij,bhjd->bhid", ok.astype(np.float64), np.abs(v))
        bound = 2.0 ** -4 * mass + 2.0 ** -10 * np.exp(m - lse)[..., None] * vsum
        err = np.abs(oe - o)
        assert np.all(err <= bound + 1e-15) and err.max() > 1e-3
        assert np.array_equal(lse, lsee)
