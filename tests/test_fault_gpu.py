"""Failure detection on the GPU without faulting it: a pipeline wait is made
to run out (one K tile is left unloaded through the FA_TEST_STALL_UNIT hook),
and the kernel must return, report FA_ERR_TIMEOUT through fa_sync_status(),
and leave the context usable for the next call."""

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
inp = workloads.make_inputs(1, 2, 600, 64, seed=3)
q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
stream = torch.cuda.current_stream().cuda_stream
out = {{}}
os.environ["FA_TEST_STALL_UNIT"] = "0"
t0 = time.time()
fa.forward(q, k, v, causal=True)
out["stalled_status"] = fa.fa_sync_status(stream)
out["seconds"] = time.time() - t0
out["failure"] = fa.fa_last_failure()
del os.environ["FA_TEST_STALL_UNIT"]
o, lse = fa.forward(q, k, v, causal=True)
out["after_status"] = fa.fa_sync_status(stream)
x = {{n: inp[n].float().double().numpy() for n in ("q", "k", "v")}}
o_ref, lse_ref = oracle.forward(x["q"], x["k"], x["v"], float(torch.tensor(64 ** -0.5)), True)
out["after_err"] = float(np.abs(o.cpu().double().numpy() - o_ref).max())
print("RESULT " + json.dumps(out))
"""


def test_stalled_wait_reports_timeout_and_recovers():
    env = dict(os.environ, FA_WAIT_LIMIT_MS="300")
    env.pop("FA_TEST_STALL_UNIT", None)
    r = subprocess.run([sys.executable, "-c", SCRIPT.format(root=ROOT)], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    res = json.loads(next(l for l in r.stdout.splitlines() if l.startswith("RESULT "))[7:])
    assert res["stalled_status"] == 5, res          # FA_ERR_TIMEOUT
    assert res["failure"][0] == 5 and res["failure"][2] == 0, res   # code, block 0
    assert res["seconds"] < 30, res
    assert res["after_status"] == 0, res
    assert res["after_err"] <= 1e-2, res
