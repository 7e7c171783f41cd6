"""Plant plausible mistakes in a copy of the oracle's per-head arithmetic and
check that the pins of ``test_oracle.py`` catch every one of them.  CPU only.

The copy below follows the oracle step by step; each ``mut`` switch changes
one thing (a dropped term, a wrong sign, index or base, a transposed
operand).  ``attention_ref`` is monkeypatched to use the copy, so the pins
exercise the real driver code around it.
"""

import numpy as np
import pytest

import oracle.attention as oa
from test_oracle import ALL_PINS


def _attend_copy(q, k, v, scale, causal, row_pos, mut=None):
    r = q.shape[0]
    n = k.shape[0]
    o = np.zeros((r, v.shape[1]))
    lse = np.full(r, -np.inf)
    if r == 0 or n == 0:
        return o, lse
    if mut == "transpose_qk":
        s = scale * (k @ q.T)[:r, :n] if n == r else scale * (q @ k.T)
    elif mut == "no_scale":
        s = q @ k.T
    elif mut == "scale_squared":
        s = scale * scale * (q @ k.T)
    else:
        s = scale * (q @ k.T)
    if causal:
        key_pos = np.arange(n)
        if mut == "mask_flipped":
            s = np.where(key_pos[None, :] < row_pos[:, None], -np.inf, s)
        elif mut == "mask_diagonal":
            s = np.where(key_pos[None, :] >= row_pos[:, None], -np.inf, s)
        elif mut == "mask_off_by_one":
            s = np.where(key_pos[None, :] > row_pos[:, None] + 1, -np.inf, s)
        elif mut != "mask_dropped":
            s = np.where(key_pos[None, :] > row_pos[:, None], -np.inf, s)
    m = s.max(axis=1)
    live = np.isfinite(m)
    m_shift = np.where(live, m, 0.0)
    if mut == "no_max_shift":
        m_shift = np.zeros_like(m_shift)
    if mut == "exp_sign":
        e = np.exp(m_shift[:, None] - s)
        e[~np.isfinite(s)] = 0.0
    else:
        with np.errstate(over="ignore", invalid="ignore"):
            e = np.exp(s - m_shift[:, None])
    l = e.sum(axis=1)
    with np.errstate(over="ignore", invalid="ignore", divide="ignore"):
        if mut == "no_normalise":
            o[live] = e[live] @ v
        elif mut == "p_transposed" and r == n:
            o[live] = (e.T[live] @ v) / l[live, None]
        else:
            o[live] = (e[live] @ v) / l[live, None]
        if mut == "log2":
            lse[live] = m[live] + np.log2(l[live])
        elif mut == "drop_max_in_L":
            lse[live] = np.log(l[live])
        elif mut == "no_max_shift":
            lse[live] = np.log(l[live])
        else:
            lse[live] = m[live] + np.log(l[live])
    return o, lse


MUTATIONS = ["transpose_qk", "no_scale", "scale_squared", "mask_flipped",
             "mask_diagonal", "mask_off_by_one", "mask_dropped",
             "no_max_shift", "exp_sign", "no_normalise", "p_transposed",
             "log2", "drop_max_in_L"]


def _run_pins(monkeypatch, mut):
    def patched(*a, window=None):
        assert window is None  # the pins use no band
        return _attend_copy(*a, mut=mut)
    monkeypatch.setattr(oa, "_attend", patched)
    failed = []
    for pin in ALL_PINS:
        try:
            pin(oa.attention_ref)
        except (AssertionError, FloatingPointError, ValueError):
            failed.append(pin.__name__)
    return failed


def test_unmutated_copy_passes(monkeypatch):
    assert _run_pins(monkeypatch, None) == []


@pytest.mark.parametrize("mut", MUTATIONS)
def test_planted_mistake_is_caught(monkeypatch, mut):
    failed = _run_pins(monkeypatch, mut)
    assert failed, f"no pin caught mutation {mut}"
