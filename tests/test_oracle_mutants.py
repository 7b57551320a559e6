"""Plant plausible mistakes in copies of the oracle and check that the pins
catch every one of them (CPU only)."""

import importlib.util
import os
import types

import pytest

from tests import oracle_pins

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "attention.py")

MUTATIONS = {
    "scale_dropped": ("return scale * (q @ k.T)", "return (q @ k.T)"),
    "operands_transposed": ("return scale * (q @ k.T)", "return scale * (k @ q.T)"),
    "causal_strict": ("return j <= i + (nk - nq)", "return j < i + (nk - nq)"),
    "causal_flipped": ("return j <= i + (nk - nq)", "return j >= i + (nk - nq)"),
    "no_max_shift": ("np.exp(s - m[:, None])", "np.exp(s)"),
    "no_normalisation": ("o = (w @ v) / safe_l[:, None]", "o = (w @ v)"),
    "values_from_keys": ("o = (w @ v) / safe_l[:, None]", "o = (w @ k) / safe_l[:, None]"),
    "lse_without_max": ("m + np.log(safe_l), -np.inf)", "np.log(safe_l), -np.inf)"),
    "row_term_dropped": ("ds = p * (dp - dd[:, None])", "ds = p * dp"),
    "row_term_wrong_axis": ("dd = (p * dp).sum(axis=1)", "dd = (p * dp).sum(axis=0)"),
    "dk_scale_dropped": ("dk = scale * (ds.T @ q)", "dk = (ds.T @ q)"),
    "dv_transposed": ("dv = p.T @ do", "dv = p @ do"),
    "dq_from_values": ("dq = scale * (ds @ k)", "dq = scale * (ds @ v)"),
    "rows_off_by_one": ("count = min(i + (nk_all - nq) + 1, nk_all)", "count = min(i + (nk_all - nq), nk_all)"),
    "causal_offset_flipped": ("return j <= i + (nk - nq)", "return j <= i - (nk - nq)"),
    "causal_top_left": ("return j <= i + (nk - nq)", "return j <= i"),
    "bias_ignored": ("        s = s + bias\n        ok = ok & (bias > -np.inf)", "        ok = ok & (bias > -np.inf)"),
    "bias_scaled_with_scores": ("        s = s + bias\n        ok", "        s = s + scale * bias\n        ok"),
    "bias_transposed": ("        s = s + bias\n        ok", "        s = s + bias.T\n        ok"),
    "bias_sign_flipped": ("        s = s + bias\n        ok", "        s = s - bias\n        ok"),
    "rows_bias_ignored": ("            s = s + bias[bi, hi, i, :count]", "            s = s + 0.0"),
    "backward_bias_ignored": ("    s, ok = _masked_scores(q, k, scale, causal, bias)\n    if lse is None:",
                              "    s, ok = _masked_scores(q, k, scale, causal)\n    if lse is None:"),
    "backward_lse_without_bias": ("_, lse = forward_head(q, k, v, scale, causal, bias)",
                                  "_, lse = forward_head(q, k, v, scale, causal)"),
    "varlen_backward_bias_dropped": ("bias=None if bias is None else bias[bi, hi, :lq, :lk])", "bias=None)"),
    "varlen_keys_sliced_by_query_length": ("v[bi, hi, :lk],\n                                                            scale", "v[bi, hi, :lq],\n                                                            scale"),
}


def _mutant(name):
    old, new = MUTATIONS[name]
    with open(SRC) as f:
        text = f.read()
    assert text.count(old) == 1, (name, text.count(old))
    mod = types.ModuleType("oracle_mutant_" + name)
    exec(compile(text.replace(old, new), SRC + ":" + name, "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutation(name):
    assert oracle_pins.failing_checks(_mutant(name)), name


def test_unmutated_copy_passes():
    with open(SRC) as f:
        text = f.read()
    mod = types.ModuleType("oracle_copy")
    exec(compile(text, SRC, "exec"), mod.__dict__)
    assert oracle_pins.failing_checks(mod) == []
