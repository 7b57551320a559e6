"""bf16 O output (fa_fwd_ex / fa_bwd_ex) against the fp32 path and the oracle."""

import numpy as np
import pytest
import torch

import exact_tiled_attention_18_gb300 as fa
import oracle
from exact_tiled_attention_18_gb300 import workloads
from tests.helpers import GRAD_MAX_ABS, O_MAX_ABS, scale_for, to64

pytestmark = pytest.mark.gpu

# bf16 keeps 8 significant bits: rounding to nearest moves x by at most
# 2^-8 |x|, on top of the fp32 result's own tolerance.
BF16_REL = 2.0 ** -8


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal", [
    (1, 2, 300, 300, 64, False),
    (2, 1, 517, 517, 128, True),
    (1, 2, 200, 640, 128, True),
    (1, 1, 1, 999, 64, False),
])
def test_bf16_output_is_rounded_fp32_output(B, H, Nq, Nk, d, causal):
    """Same kernel, same arithmetic: the bf16 O is the fp32 O rounded to
    nearest even, bit for bit, and the LSE is identical."""
    g = workloads.make_decode_inputs(B, H, Nq, Nk, d, seed=Nq + Nk + d)
    q, k, v = (g[n].cuda() for n in ("q", "k", "v"))
    o32, l32 = fa.forward_varlen(q, k, v, causal=causal)
    o16, l16 = fa.forward_varlen(q, k, v, causal=causal, o_dtype=torch.bfloat16)
    fa.sync_status()
    assert o16.dtype == torch.bfloat16
    assert torch.equal(o16, o32.to(torch.bfloat16))
    assert torch.equal(l16, l32)


def test_bf16_output_padded_batch_matches_oracle():
    B, H, Nq, Nk, d = 4, 2, 300, 400, 128
    sq, sk = [300, 17, 0, 256], [400, 250, 99, 0]
    g = workloads.make_decode_inputs(B, H, Nq, Nk, d, seed=8)
    scale = scale_for(d)
    q, k, v = (g[n].cuda() for n in ("q", "k", "v"))
    lq = torch.tensor(sq, dtype=torch.int32, device="cuda")
    lk = torch.tensor(sk, dtype=torch.int32, device="cuda")
    o, lse = fa.forward_varlen(q, k, v, lq, lk, causal=True, scale=scale, o_dtype=torch.bfloat16)
    fa.sync_status()
    o_ref, _ = oracle.forward_varlen(to64(g["q"]), to64(g["k"]), to64(g["v"]), scale, True, sq, sk)
    err = np.abs(o.cpu().double().numpy() - o_ref)
    assert np.all(err <= O_MAX_ABS + BF16_REL * np.abs(o_ref))
    oc = o.cpu()
    for b in range(B):
        assert torch.all(oc[b, :, sq[b]:] == 0)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_from_bf16_output(causal):
    """The row term is corrected to the recomputed probabilities, so the
    gradients from a bf16 O match the oracle and the fp32-O gradients: dK and
    dV to 1e-3; dQ, which takes dS rounded to bf16 (whose rounding differs
    between the two runs, whose D' differ), within the gradient tolerance."""
    B, H, N, d = 1, 2, 640, 128
    inp = workloads.make_inputs(B, H, N, d, seed=44 + causal, with_grad=True, boost_every=64, boost=10.0)
    scale = scale_for(d)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    o32, lse = fa.forward(q, k, v, causal=causal, scale=scale)
    o16, _ = fa.forward_varlen(q, k, v, causal=causal, scale=scale, o_dtype=torch.bfloat16)
    g32 = fa.backward(q, k, v, o32, lse, do, causal=causal, scale=scale)
    g16 = fa.backward_varlen(q, k, v, o16, lse, do, causal=causal, scale=scale)
    fa.sync_status()
    ref = oracle.backward(to64(inp["q"]), to64(inp["k"]), to64(inp["v"]), to64(inp["do"]), scale, causal)
    for name, a, b, r in zip(("dQ", "dK", "dV"), g16, g32, ref[:3]):
        a64 = a.cpu().double().numpy()
        assert np.abs(a64 - r).max() <= GRAD_MAX_ABS, name
        assert (a - b).abs().max() <= (GRAD_MAX_ABS if name == "dQ" else 1e-3), name
