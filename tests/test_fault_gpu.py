"""Failure detection on the GPU without faulting it: a pipeline wait is made
to run out (one tile is left unloaded through the fa_test_set_stall hook),
and the kernel must return, report FA_ERR_TIMEOUT through fa_sync_status(),
and leave the context usable for the next call.  Covers the forward, both
kernels of each backward algorithm (two-pass and single-pass), the decode
kernel, the FP8 forward and the split-key forward."""

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import json, os, sys, time
sys.path.insert(0, {root!r})
import numpy as np, torch
import exact_tiled_attention_18_gb300 as fa
import oracle
from exact_tiled_attention_18_gb300 import workloads
which = {which!r}
stream = torch.cuda.current_stream().cuda_stream
scale = float(torch.tensor(64 ** -0.5))
inp = workloads.make_inputs(1, 2, 600, 64, seed=3, with_grad=True)
q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
x = {{n: inp[n].float().double().numpy() for n in inp}}
if which in ("dq", "dkdv", "rowterm", "fused"):
    o, lse = fa.forward(q, k, v, causal=True, scale=scale)
    fa.sync_status()
    grads = [torch.empty(q.shape, dtype=torch.float32, device="cuda") for _ in range(3)]
    ws = torch.empty(2 * 600, dtype=torch.float32, device="cuda")
if which == "decode":
    g = workloads.make_decode_inputs(1, 2, 1, 6000, 64, seed=4)
    dq_, dk_, dv_ = (g[n].cuda() for n in ("q", "k", "v"))
if which == "splitkv":
    xs = workloads.make_inputs(1, 1, 2000, 64, seed=6)
    qs, ks, vs = (xs[n].cuda() for n in ("q", "k", "v"))
if which == "fp8":
    x8 = workloads.make_fp8_inputs(1, 2, 640, 128, seed=5)
    q8, k8, vt8 = (x8[n].cuda() for n in ("q", "k", "vt"))
    s8 = float(torch.tensor(128 ** -0.5))

def run():
    if which == "fwd":
        return fa.forward(q, k, v, causal=True, scale=scale)
    if which == "dq":
        fa.backward_stage(0, q, k, v, o, lse, do, *grads, ws, causal=True, scale=scale)
        return grads
    if which == "dkdv":
        fa.backward_stage(0, q, k, v, o, lse, do, *grads, ws, causal=True, scale=scale)
        fa.sync_status()
        fa.fa_test_set_stall(pending)
        fa.backward_stage(1, q, k, v, o, lse, do, *grads, ws, causal=True, scale=scale)
        return grads
    if which == "rowterm":
        fa.backward_stage(2, q, k, v, None, lse, do, *grads, ws, causal=True, scale=scale)
        if pending == -1:  # the recovery run completes the single pass
            fa.backward_stage(3, q, k, v, None, lse, do, *grads, ws, causal=True, scale=scale)
        return grads
    if which == "fused":
        fa.backward_stage(2, q, k, v, None, lse, do, *grads, ws, causal=True, scale=scale)
        fa.sync_status()
        fa.fa_test_set_stall(pending)
        fa.backward_stage(3, q, k, v, None, lse, do, *grads, ws, causal=True, scale=scale)
        return grads
    if which == "fp8":
        return fa.forward_fp8(q8, k8, vt8, causal=True, scale=s8)
    if which == "splitkv":
        return fa.forward_splitkv(qs, ks, vs, causal=True, scale=scale)
    return fa.forward_decode(dq_, dk_, dv_, causal=True, scale=scale)

out = {{}}
pending = 0
if which not in ("dkdv", "fused"):
    fa.fa_test_set_stall(pending)
t0 = time.time()
run()
out["stalled_status"] = fa.fa_sync_status(stream)
out["seconds"] = time.time() - t0
out["failure"] = fa.fa_last_failure()
pending = -1
fa.fa_test_set_stall(pending)
res = run()
out["after_status"] = fa.fa_sync_status(stream)
if which == "fwd":
    ref = oracle.forward(x["q"], x["k"], x["v"], scale, True)[0]
    out["after_err"] = float(np.abs(res[0].cpu().double().numpy() - ref).max())
elif which in ("dq", "dkdv", "rowterm", "fused"):
    ref = oracle.backward(x["q"], x["k"], x["v"], x["do"], scale, True)
    idx = 0 if which in ("dq", "rowterm") else 1
    out["after_err"] = float(np.abs(res[idx].cpu().double().numpy() - ref[idx]).max())
elif which == "splitkv":
    xx = {{n: xs[n].float().double().numpy() for n in xs}}
    ref = oracle.forward(xx["q"], xx["k"], xx["v"], scale, True)[0]
    out["after_err"] = float(np.abs(res[0].cpu().double().numpy() - ref).max())
elif which == "fp8":
    # within the bound that rounding P to E4M3 gives (normalised to the 2e-2 check below)
    vx = {{n: workloads.fp8_values(x8[n]).double().numpy() for n in ("q", "k", "v")}}
    ref = oracle.forward(vx["q"], vx["k"], vx["v"], s8, True)[0]
    mass = oracle.forward(vx["q"], vx["k"], np.abs(vx["v"]), s8, True)[0]
    bound = 2.0 ** -4 * mass + 2.0 ** -10 * np.abs(vx["v"]).sum(axis=2, keepdims=True) + 1e-4
    out["after_err"] = float((np.abs(res[0].cpu().double().numpy() - ref) / bound).max()) * 2e-2
else:
    gx = {{n: g[n].float().double().numpy() for n in g}}
    ref = oracle.forward(gx["q"], gx["k"], gx["v"], scale, True)[0]
    out["after_err"] = float(np.abs(res[0].cpu().double().numpy() - ref).max())
print("RESULT " + json.dumps(out))
"""


@pytest.mark.parametrize("which", ["fwd", "dq", "dkdv", "decode", "fp8", "rowterm", "fused", "splitkv"])
def test_stalled_wait_reports_timeout_and_recovers(which):
    env = dict(os.environ, FA_WAIT_LIMIT_MS="300")
    env.pop("FA_TEST_STALL_UNIT", None)
    r = subprocess.run([sys.executable, "-c", SCRIPT.format(root=ROOT, which=which)], env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    res = json.loads(next(l for l in r.stdout.splitlines() if l.startswith("RESULT "))[7:])
    assert res["stalled_status"] == 5, res          # FA_ERR_TIMEOUT
    assert res["failure"][0] == 5 and res["failure"][2] == 0, res   # code, block 0
    assert res["seconds"] < 30, res
    assert res["after_status"] == 0, res
    assert res["after_err"] <= 2e-2, res
