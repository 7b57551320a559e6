"""Backward parity: dQ, dK, dV (and D) from the CUDA path against the fp64 oracle."""

import numpy as np
import pytest
import torch

import exact_tiled_attention_18_gb300 as fa
import oracle
from exact_tiled_attention_18_gb300 import workloads
from tests.helpers import GRAD_MAX_ABS, assert_row_term_close, scale_for, to64

pytestmark = pytest.mark.gpu


def gpu_fwd_bwd(inp, causal, scale, workspace=True):
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    B, H, N, d = q.shape
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale)
    ws = torch.empty(fa.fa_bwd_workspace_bytes(B, H, N) // 4, dtype=torch.float32, device="cuda") if workspace else None
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, causal=causal, scale=scale, workspace=ws)
    fa.sync_status()
    return dq.cpu(), dk.cpu(), dv.cpu(), (ws.cpu() if ws is not None else None)


def check_grads(got, ref, what, heads=None):
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        g = g.numpy().astype(np.float64)
        if heads is not None:
            g = g[heads]
        assert np.all(np.isfinite(g)), f"{what} {name}: non-finite"
        err = np.abs(g - r).max()
        assert err <= GRAD_MAX_ABS, f"{what} {name}: max abs {err:.3e}"


SMALL = [
    (1, 1, 256, 64, False),
    (1, 1, 256, 64, True),
    (1, 1, 1, 64, True),
    (1, 1, 1, 128, False),
    (1, 1, 127, 128, True),
    (2, 1, 129, 128, False),
    (1, 2, 200, 64, True),
    (1, 1, 257, 128, True),
    (1, 2, 300, 64, False),
    (2, 2, 384, 128, True),
    (1, 3, 517, 128, True),
    (1, 2, 1000, 64, True),
    (1, 1, 1024, 128, False),
]


@pytest.mark.parametrize("B,H,N,d,causal", SMALL)
def test_backward_small_matches_oracle(B, H, N, d, causal):
    inp = workloads.make_inputs(B, H, N, d, seed=100 + N + d + causal, with_grad=True)
    scale = scale_for(d)
    dq, dk, dv, ws = gpu_fwd_bwd(inp, causal, scale)
    x = {n: to64(inp[n]) for n in inp}
    rq, rk, rv, rd = oracle.backward(x["q"], x["k"], x["v"], x["do"], scale, causal)
    check_grads((dq, dk, dv), (rq, rk, rv), f"{(B, H, N, d, causal)}")
    # D left in the workspace against the oracle's sum_j P_ij dP_ij, row by
    # row, at the fp32 bound (tests/helpers.py)
    rd_abs = oracle.backward(x["q"], x["k"], np.abs(x["v"]), np.abs(x["do"]), scale, causal)[3]
    rel = assert_row_term_close(ws.numpy(), rd, rd_abs, f"{(B, H, N, d, causal)}")
    print(f"D: largest error / D_abs {rel:.2e}")


def test_backward_without_workspace():
    inp = workloads.make_inputs(1, 2, 333, 128, seed=9, with_grad=True)
    scale = scale_for(128)
    a = gpu_fwd_bwd(inp, True, scale, workspace=True)
    b = gpu_fwd_bwd(inp, True, scale, workspace=False)
    for x, y in zip(a[:3], b[:3]):
        assert torch.equal(x, y)


def test_gradient_sum_properties_full_size():
    """At full size: sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i per head
    (softmax rows sum to one; shifting every key by one vector changes nothing)."""
    w = workloads.WORKLOADS["training_b4_h16_n8192_d128_causal"]
    inp = workloads.workload_inputs(w, 0)
    dq, dk, dv, _ = gpu_fwd_bwd(inp, w.causal, w.scale)
    sum_dk = dk.double().sum(dim=2)
    sum_dv = dv.double().sum(dim=2)
    sum_do = inp["do"].double().sum(dim=2)
    assert sum_dk.abs().max() < 0.5, sum_dk.abs().max()
    assert (sum_dv - sum_do).abs().max() < 0.5, (sum_dv - sum_do).abs().max()


@pytest.mark.parametrize("name,heads", [
    ("training_b4_h16_n8192_d128_causal", [(0, 0), (3, 15)]),
    ("long_context_b1_h32_n16384_d128_causal", [(0, 17)]),
])
def test_backward_full_size_whole_heads(name, heads):
    """Full-size run in the bench's launch configuration; whole heads checked
    against the oracle (heads are independent)."""
    w = workloads.WORKLOADS[name]
    inp = workloads.workload_inputs(w, 0)
    dq, dk, dv, ws = gpu_fwd_bwd(inp, w.causal, w.scale)
    ws = ws.reshape(w.B, w.H, w.N)
    for (b, h) in heads:
        x = {n: to64(inp[n][b:b + 1, h:h + 1]) for n in inp}
        rq, rk, rv, rd = oracle.backward(x["q"], x["k"], x["v"], x["do"], w.scale, w.causal)
        got = tuple(t[b:b + 1, h:h + 1] for t in (dq, dk, dv))
        check_grads(got, (rq, rk, rv), f"{name} head {(b, h)}")
        errs = [float(np.abs(g.numpy().astype(np.float64) - r).max()) for g, r in zip(got, (rq, rk, rv))]
        rd_abs = oracle.backward(x["q"], x["k"], np.abs(x["v"]), np.abs(x["do"]), w.scale, w.causal)[3]
        rel = assert_row_term_close(ws[b:b + 1, h:h + 1].numpy(), rd, rd_abs, f"{name} head {(b, h)} D")
        print(f"{name} head {(b, h)}: dQ {errs[0]:.2e} dK {errs[1]:.2e} dV {errs[2]:.2e}; "
              f"D largest error / D_abs {rel:.2e}")


def test_row_term_follows_its_own_rows_across_units():
    """Each persistent CTA of the dQ kernel handles several 128-row work units
    in turn, its loader warps forming the next unit's row term while the
    current one runs.  Query tiles here carry dO scaled by 0.1, 1 or 10 in
    turn (so neighbouring units' row terms differ by 10-100x) and there are
    about two units per CTA: a row term taken from a stale slot or a wrong
    row fails the row-by-row check at once."""
    B, H, N, d = 1, 4, 10000, 128
    inp = workloads.make_inputs(B, H, N, d, seed=77, with_grad=True)
    tile_scale = torch.tensor([0.1, 1.0, 10.0])[(torch.arange(N) // 128) % 3]
    inp["do"] = (inp["do"].float() * tile_scale[None, None, :, None]).to(torch.bfloat16)
    scale = scale_for(d)
    dq, dk, dv, ws = gpu_fwd_bwd(inp, True, scale)
    x = {n: to64(inp[n]) for n in inp}
    rq, rk, rv, rd = oracle.backward(x["q"], x["k"], x["v"], x["do"], scale, True)
    rd_abs = oracle.backward(x["q"], x["k"], np.abs(x["v"]), np.abs(x["do"]), scale, True)[3]
    rel = assert_row_term_close(ws.numpy(), rd, rd_abs, "alternating dO scales")
    print(f"alternating dO scales: D largest error / D_abs {rel:.2e}")
    # gradients scale with dO (up to 10x): tolerance 2e-2 per unit of dO scale
    for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), (rq, rk, rv)):
        err = np.abs(g.numpy().astype(np.float64) - r).max()
        assert err <= 10 * GRAD_MAX_ABS, (name, err)


def test_backward_masked_positions_do_not_leak():
    """Extreme values at causally masked key/value positions leave the
    gradients of the rows that cannot see them unchanged: with keys from 160
    on set to +1e4 and their values to -1e4, dQ and the row term D of
    queries 0..159 stay bit for bit the same (160 is a warp boundary)."""
    B, H, N, d = 1, 2, 300, 64
    inp = workloads.make_inputs(B, H, N, d, seed=13, with_grad=True)
    scale = scale_for(d)

    def run(x):
        q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
        o, lse = fa.forward(q, k, v, causal=True, scale=scale)
        ws = torch.empty(B * H * N, dtype=torch.float32, device="cuda")
        dq, dk, dv = fa.backward(q, k, v, o, lse, do, causal=True, scale=scale, workspace=ws)
        fa.sync_status()
        return dq.cpu(), ws.cpu().reshape(B, H, N)

    dq1, d1 = run(inp)
    poisoned = {n: t.clone() for n, t in inp.items()}
    poisoned["k"][:, :, 160:, :] = 1e4
    poisoned["v"][:, :, 160:, :] = -1e4
    dq2, d2 = run(poisoned)
    assert torch.isfinite(dq2).all()
    assert torch.equal(dq1[:, :, :160], dq2[:, :, :160])
    assert torch.equal(d1[:, :, :160], d2[:, :, :160])


def test_stages_equal_fa_bwd():
    """fa_bwd_stage 0, 1 in order is exactly fa_bwd."""
    inp = workloads.make_inputs(2, 2, 300, 128, seed=31, with_grad=True)
    scale = scale_for(128)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, causal=True, scale=scale)
    ref = fa.backward(q, k, v, o, lse, do, causal=True, scale=scale)
    ws = torch.empty(2 * 2 * 300, dtype=torch.float32, device="cuda")
    out = [torch.empty_like(x) for x in ref]
    for stage in range(2):
        fa.backward_stage(stage, q, k, v, o, lse, do, *out, ws, causal=True, scale=scale)
    fa.sync_status()
    for a, b in zip(out, ref):
        assert torch.equal(a, b)
