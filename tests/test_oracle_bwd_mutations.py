"""Plant plausible mistakes in a copy of the backward oracle's per-head
arithmetic and check that the pins of ``test_oracle_bwd.py`` catch every
one of them.  CPU only.

The copy follows the oracle step by step; each ``mut`` switch changes one
thing (a dropped term, a wrong sign or scale, a transposed operand, a
missing mask or normalisation).  ``_bwd_head`` is monkeypatched, so the
pins exercise the real driver code around it.
"""

import numpy as np
import pytest

import oracle.backward as ob
from test_oracle_bwd import BWD_PINS


def _bwd_copy(q, k, v, do, scale, causal, window=None, mut=None):
    n = q.shape[0]
    if n == 0:
        return np.zeros_like(q), np.zeros_like(k), np.zeros_like(v), np.zeros(0)
    keep = ob._mask(n, np.arange(n), causal and mut != "mask_dropped", window)
    sc = 1.0 if mut == "no_scale_in_p" else scale
    s = np.where(keep, sc * (q @ k.T), -np.inf)
    m = s.max(axis=1, keepdims=True)
    e = np.where(keep, np.exp(s - m), 0.0)
    p = e if mut == "p_unnormalised" else e / e.sum(axis=1, keepdims=True)
    o = p @ v
    dv = (p @ do) if mut == "dv_not_transposed" else p.T @ do
    dp = (v @ do.T) if mut == "dp_transposed" else do @ v.T
    if mut == "delta_from_do":
        delta = do.sum(axis=1)
    else:
        delta = np.sum(do * o, axis=1)
    if mut == "no_delta":
        ds = p * dp
    elif mut == "delta_sign":
        ds = p * (dp + delta[:, None])
    else:
        ds = p * (dp - delta[:, None])
    dq = (ds @ k) if mut == "dq_no_scale" else scale * (ds.T @ k if mut == "dq_transposed" else ds @ k)
    if mut == "dk_no_scale":
        dk = ds.T @ q
    elif mut == "dk_uses_k":
        dk = scale * (ds.T @ k)
    elif mut == "dk_not_transposed":
        dk = scale * (ds @ q)
    else:
        dk = scale * (ds.T @ q)
    return dq, dk, dv, delta


MUTATIONS = ["mask_dropped", "no_scale_in_p", "p_unnormalised", "dv_not_transposed",
             "dp_transposed", "delta_from_do", "no_delta", "delta_sign", "dq_no_scale",
             "dq_transposed", "dk_no_scale", "dk_uses_k", "dk_not_transposed"]


def _run_pins(monkeypatch, mut):
    monkeypatch.setattr(ob, "_bwd_head", lambda *a, **kw: _bwd_copy(*a, **kw, mut=mut))
    failed = []
    for pin in BWD_PINS:
        try:
            pin(lambda q, k, v, do, s, c: ob.attention_bwd_ref(q, k, v, do, s, c)[:3])
        except (AssertionError, FloatingPointError, ValueError):
            failed.append(pin.__name__)
    return failed


def test_unmutated_copy_passes(monkeypatch):
    assert _run_pins(monkeypatch, None) == []


@pytest.mark.parametrize("mut", MUTATIONS)
def test_planted_mistake_is_caught(monkeypatch, mut):
    failed = _run_pins(monkeypatch, mut)
    assert failed, f"no pin caught mutation {mut}"
