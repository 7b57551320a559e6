"""FP8 forward (fa_fwd_fp8) against the fp64 oracle on the same E4M3 input
values.  Parity: LSE to the stated 1e-3; O within the bound that rounding P to
E4M3 gives, |dO_i| <= 2^-4 sum_j P_ij |v_j| + 2^-10 e^(m_i - LSE_i) sum_j |v_j|
(relative half-spacing of three mantissa bits; half the subnormal spacing),
element for element, plus 1e-4 for the fp32 arithmetic.  A tolerance of its
own for this dtype, as "FlashAttention Interview Questions", section "Why
can recomputation help training?", asks for each configuration."""

import numpy as np
import pytest
import torch

import exact_tiled_attention_18_gb300 as fa
import oracle
from oracle import rounding
from exact_tiled_attention_18_gb300 import workloads
from tests.helpers import LSE_REL, lse_rel_err, scale_for

pytestmark = pytest.mark.gpu


def _run(x, causal, scale):
    o, lse = fa.forward_fp8(x["q"].cuda(), x["k"].cuda(), x["vt"].cuda(), causal=causal, scale=scale)
    fa.sync_status()
    return o.cpu().double().numpy(), lse.cpu().double().numpy()


def _vals(x):
    return {n: workloads.fp8_values(x[n]).double().numpy() for n in ("q", "k", "v")}


@pytest.mark.parametrize("B,H,N,causal", [
    (1, 2, 256, False),
    (2, 1, 384, True),
    (1, 2, 1024, True),
    (1, 1, 144, False),
    (1, 1, 16, True),
    (1, 3, 2000, True),
])
def test_fp8_forward_matches_oracle_within_rounding_bound(B, H, N, causal):
    x = workloads.make_fp8_inputs(B, H, N, 128, seed=N + causal)
    scale = scale_for(128)
    o, lse = _run(x, causal, scale)
    v = _vals(x)
    o_ref, lse_ref = oracle.forward(v["q"], v["k"], v["v"], scale, causal)
    assert np.all(np.isfinite(o))
    assert lse_rel_err(lse, lse_ref) <= LSE_REL
    mass, _ = oracle.forward(v["q"], v["k"], np.abs(v["v"]), scale, causal)
    s = scale * np.einsum("bhid,bhjd->bhij", v["q"], v["k"])
    ok = oracle.eligible(N, N, causal)
    m = np.where(ok, s, -np.inf).max(axis=-1)
    vsum = np.einsum("ij,bhjd->bhid", ok.astype(np.float64), np.abs(v["v"]))
    bound = 2.0 ** -4 * mass + 2.0 ** -10 * np.exp(m - lse_ref)[..., None] * vsum + 1e-4
    err = np.abs(o - o_ref)
    assert np.all(err <= bound), (err.max(), (err / bound).max())
    # and the same size as the companion's own error (P rounded to E4M3)
    o_c, _ = rounding.forward(v["q"], v["k"], v["v"], scale, causal, p_round=rounding.round_e4m3)
    e_c = np.abs(o_c - o_ref)
    assert err.mean() <= 2.0 * e_c.mean() + 1e-6, (err.mean(), e_c.mean())


def test_fp8_forward_full_size_sampled_rows():
    """B=4, H=16, N=8192 causal (the training workload's shape), in the bench's
    launch configuration; 128 seeded rows checked one by one."""
    B, H, N, d = 4, 16, 8192, 128
    x = workloads.make_fp8_inputs(B, H, N, d, seed=3)
    scale = scale_for(d)
    o, lse = _run(x, True, scale)
    v = _vals(x)
    rows = workloads.sample_rows(B, H, N, 128, seed=7)
    ro, rl = oracle.forward_rows(v["q"], v["k"], v["v"], scale, True, rows)
    mass, _ = oracle.forward_rows(v["q"], v["k"], np.abs(v["v"]), scale, True, rows)
    for n_, (b, h, i) in enumerate(rows):
        s = scale * (v["k"][b, h, :i + 1] @ v["q"][b, h, i])
        vsum = np.abs(v["v"][b, h, :i + 1]).sum(axis=0)
        bound = 2.0 ** -4 * mass[n_] + 2.0 ** -10 * np.exp(s.max() - rl[n_]) * vsum + 1e-4
        assert np.all(np.abs(o[b, h, i] - ro[n_]) <= bound), (b, h, i)
        assert abs(lse[b, h, i] - rl[n_]) / max(abs(rl[n_]), 1.0) <= LSE_REL
