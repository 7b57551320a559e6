"""Shared helpers for the GPU tests: run the CUDA path, compare with the oracle."""

from __future__ import annotations

import numpy as np
import torch

import exact_tiled_attention_18_gb300 as fa
from exact_tiled_attention_18_gb300 import workloads

# Tolerances stated for the method: O max-abs <= 1e-2 and mean-abs <= 1e-3;
# LSE relative <= 1e-3, read as |dLSE| / max(|LSE|, 1); gradients max-abs <= 2e-2.
O_MAX_ABS = 1e-2
O_MEAN_ABS = 1e-3
LSE_REL = 1e-3
GRAD_MAX_ABS = 2e-2


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def scale_for(d: int) -> float:
    return float(torch.tensor(d ** -0.5, dtype=torch.float32))


def gpu_forward(inp: dict, causal: bool, scale: float):
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale)
    fa.sync_status()
    return o.cpu(), lse.cpu()


def lse_rel_err(got: np.ndarray, ref: np.ndarray) -> float:
    return float(np.max(np.abs(got - ref) / np.maximum(np.abs(ref), 1.0)))


def assert_forward_close(o, lse, o_ref, lse_ref, what=""):
    o = np.asarray(o, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    assert np.all(np.isfinite(o)), f"{what}: non-finite O"
    err = np.abs(o - o_ref)
    assert err.max() <= O_MAX_ABS, f"{what}: O max abs {err.max():.3e}"
    assert err.mean() <= O_MEAN_ABS, f"{what}: O mean abs {err.mean():.3e}"
    le = lse_rel_err(lse, lse_ref)
    assert le <= LSE_REL, f"{what}: LSE rel {le:.3e}"
    return err.max(), err.mean(), le


# Row term D_i = sum_j P_ij dP_ij left in the backward workspace.  The kernels
# form it in fp32 from fp32 probabilities and fp32 dot products, so its error
# is a small multiple of fp32 rounding of the terms it sums, not of the bf16
# operands: bounded here by ROW_TERM_REL times D_abs_i = sum_j P_ij sum_c
# |dO_ic| |v_jc| (the oracle's row term for |dO| and |V|, an upper bound on
# sum_j P_ij |dP_ij|), plus ROW_TERM_ABS.  At d = 128 with N(0,1) data D_abs
# is about 80, so the bound is near 1e-3 absolute: far below a row term taken
# from a wrong or stale row (order 1) or left uncorrected as rowsum(dO o O)
# of the bf16-rounded forward output (order 1e-2).
ROW_TERM_REL = 1e-5
ROW_TERM_ABS = 1e-6


def assert_row_term_close(got, ref, ref_abs, what=""):
    """Element-wise check of the workspace D against the oracle; returns the
    largest |error| / D_abs seen."""
    got = np.asarray(got, dtype=np.float64).reshape(np.shape(ref))
    err = np.abs(got - ref)
    assert np.all(np.isfinite(got)), f"{what}: non-finite D"
    bound = ROW_TERM_REL * ref_abs + ROW_TERM_ABS
    bad = err > bound
    assert not bad.any(), (f"{what}: D error {err[bad].max():.3e} above its bound at {int(bad.sum())} rows "
                           f"(largest error / D_abs {float((err / np.maximum(ref_abs, 1e-30)).max()):.2e})")
    return float((err / np.maximum(ref_abs, 1e-30)).max())
