"""Pins of the backward oracle (CPU only).

The gradients of sum(O * dO) are checked against things that do not share
the oracle's formula: central finite differences of the (separately pinned)
forward oracle, torch's own autograd in float64, closed forms and
invariants that follow from the definition of the row softmax.
"""

import math

import numpy as np
import pytest
import torch

from oracle import (attention_bwd_magnitudes, attention_bwd_recompute, attention_bwd_ref,
                    attention_bwd_ref_varlen,
                    attention_ref, forward_for_backward)


def _rng(seed):
    return np.random.default_rng(seed)


def _case(seed, n, d, dv, qk=1.0):
    r = _rng(seed)
    return (r.normal(size=(n, d)) * qk, r.normal(size=(n, d)) * qk, r.normal(size=(n, dv)),
            r.normal(size=(n, dv)))


# ---------------------------------------------------------------------------
# pins: each takes grad(q, k, v, do, scale, causal) -> (dq, dk, dv)
# ---------------------------------------------------------------------------
def pin_finite_differences(grad):
    """Central differences of f = sum(attention(Q, K, V) * dO), f from the
    forward oracle, step 1e-5: truncation ~1e-10, checked to 1e-7."""
    for causal in (False, True):
        q, k, v, do = _case(1, 5, 3, 2)
        dq, dk, dv = grad(q, k, v, do, 0.7, causal)

        def f(qq, kk, vv):
            return float(np.sum(attention_ref(qq, kk, vv, 0.7, causal)[0] * do))
        h = 1e-5
        for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            for idx in np.ndindex(x.shape):
                xp, xm = x.copy(), x.copy()
                xp[idx] += h
                xm[idx] -= h
                args_p = {"q": q, "k": k, "v": v}
                args_m = dict(args_p)
                args_p[name], args_m[name] = xp, xm
                fd = (f(args_p["q"], args_p["k"], args_p["v"]) -
                      f(args_m["q"], args_m["k"], args_m["v"])) / (2 * h)
                assert abs(fd - g[idx]) <= 1e-7, (name, idx, causal, fd, g[idx])


def pin_torch_autograd(grad):
    """torch.nn.functional.scaled_dot_product_attention's autograd in
    float64 (CPU math path)."""
    for causal in (False, True):
        q, k, v, do = _case(2, 37, 8, 5, qk=1.5)
        dq, dk, dv = grad(q, k, v, do, 0.4, causal)
        tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
        out = torch.nn.functional.scaled_dot_product_attention(
            tq[None, None], tk[None, None], tv[None, None], is_causal=causal, scale=0.4)[0, 0]
        out.backward(torch.tensor(do, dtype=torch.float64))
        for mine, ref in ((dq, tq.grad), (dk, tk.grad), (dv, tv.grad)):
            assert np.max(np.abs(mine - ref.numpy())) <= 1e-12


def pin_dv_sums_to_do(grad):
    """Rows of P sum to one, so the rows of dV = P^T dO sum to those of dO."""
    for causal in (False, True):
        q, k, v, do = _case(3, 23, 4, 6)
        _, _, dv = grad(q, k, v, do, 0.9, causal)
        assert np.max(np.abs(dv.sum(0) - do.sum(0))) <= 1e-12


def pin_key_shift(grad):
    """Adding one vector to every key moves each score row by a constant, so
    P, and with it every gradient, is unchanged (each dS row sums to 0)."""
    for causal in (False, True):
        q, k, v, do = _case(4, 19, 5, 3)
        g0 = grad(q, k, v, do, 0.6, causal)
        g1 = grad(q, k + _rng(5).normal(size=(1, 5)) * 3, v, do, 0.6, causal)
        for a, b in zip(g0, g1):
            assert np.max(np.abs(a - b)) <= 1e-11


def pin_linear_in_do(grad):
    """The gradients are linear in dO."""
    q, k, v, do = _case(6, 17, 4, 4)
    do2 = _rng(7).normal(size=do.shape)
    for causal in (False, True):
        ga = grad(q, k, v, do, 0.5, causal)
        gb = grad(q, k, v, do2, 0.5, causal)
        gc = grad(q, k, v, 2.0 * do - 3.0 * do2, 0.5, causal)
        for a, b, c in zip(ga, gb, gc):
            assert np.max(np.abs(c - (2.0 * a - 3.0 * b))) <= 1e-12
        for z in grad(q, k, v, np.zeros_like(do), 0.5, causal):
            assert np.all(z == 0)


def pin_zero_query_closed_form(grad):
    """Q = 0: P is uniform over the visible keys.  Then dV_j = sum over the
    rows that see key j of dO_i / (number of keys row i sees), dK = 0, and
    dQ_i = scale / c_i * sum_j (dO_i . (v_j - vbar_i)) k_j over its keys."""
    n, d = 11, 4
    _, k, v, do = _case(8, n, d, 3)
    q = np.zeros((n, d))
    for causal in (False, True):
        dq, dk, dv = grad(q, k, v, do, 0.8, causal)
        assert np.max(np.abs(dk)) <= 1e-13
        for i in range(n):
            c = i + 1 if causal else n
            vbar = v[:c].mean(0)
            ref = 0.8 / c * sum((do[i] @ (v[j] - vbar)) * k[j] for j in range(c))
            assert np.max(np.abs(dq[i] - ref)) <= 1e-13
        for j in range(n):
            rows = range(j, n) if causal else range(n)
            ref = sum(do[i] / (i + 1 if causal else n) for i in rows)
            assert np.max(np.abs(dv[j] - ref)) <= 1e-13


def pin_causal_edges(grad):
    """Causal: row 0 sees only key 0 (P = 1, so dS row 0 = 0 and dQ_0 = 0);
    the last key is seen only by the last row, so dV_{n-1} = P[n-1, n-1]
    dO_{n-1} with P from the forward oracle's L."""
    n = 9
    q, k, v, do = _case(9, n, 4, 3)
    dq, _, dv = grad(q, k, v, do, 0.7, True)
    assert np.max(np.abs(dq[0])) <= 1e-14
    _, L = attention_ref(q, k, v, 0.7, True)
    p_last = math.exp(0.7 * float(q[-1] @ k[-1]) - L[-1])
    assert np.max(np.abs(dv[-1] - p_last * do[-1])) <= 1e-14


def pin_zero_values(grad):
    """V = 0: O = 0 and dP = 0, so dS = 0 and dQ = dK = 0, while dV = P^T dO
    is not zero."""
    q, k, _, do = _case(10, 13, 4, 3)
    v = np.zeros((13, 3))
    for causal in (False, True):
        dq, dk, dv = grad(q, k, v, do, 0.5, causal)
        assert np.max(np.abs(dq)) <= 1e-15 and np.max(np.abs(dk)) <= 1e-15
        assert np.max(np.abs(dv)) > 1e-3


BWD_PINS = [pin_finite_differences, pin_torch_autograd, pin_dv_sums_to_do, pin_key_shift,
            pin_linear_in_do, pin_zero_query_closed_form, pin_causal_edges, pin_zero_values]


def _ref3(q, k, v, do, s, c):
    return attention_bwd_ref(q, k, v, do, s, c)[:3]


@pytest.mark.parametrize("pin", BWD_PINS, ids=lambda p: p.__name__)
def test_bwd_ref_pins(pin):
    pin(_ref3)


@pytest.mark.parametrize("pin", BWD_PINS, ids=lambda p: p.__name__)
@pytest.mark.parametrize("blocks", [(1, 1), (4, 3), (16, 16), (64, 128)])
def test_bwd_recompute_pins(pin, blocks):
    """STAGE 5's route: P recomputed per tile from Q, K and the stored L."""
    br, bc = blocks

    def grad(q, k, v, do, s, c):
        o, lse = forward_for_backward(q, k, v, s, c)
        return attention_bwd_recompute(q, k, v, do, o, lse, s, c, Br=br, Bc=bc)
    pin(grad)


@pytest.mark.parametrize("pin", BWD_PINS, ids=lambda p: p.__name__)
def test_bwd_varlen_pins(pin):
    """A single sequence between empty ones in a packed batch."""
    def grad(q, k, v, do, s, c):
        n = np.asarray(q).shape[0]
        cu = np.array([0, 0, n, n], dtype=np.int32)
        dq, dk, dv, _ = attention_bwd_ref_varlen(q[:, None], k[:, None], v[:, None],
                                                 do[:, None], cu, s, c)
        return dq[:, 0], dk[:, 0], dv[:, 0]
    pin(grad)


def test_bwd_varlen_sequences_are_independent():
    """Each packed sequence's gradients are those of the sequence alone."""
    r = _rng(11)
    lens = [3, 0, 5, 1, 4]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    tot, H, d = int(cu[-1]), 2, 4
    q, k, v, do = (r.normal(size=(tot, H, d)) for _ in range(4))
    for causal in (False, True):
        dq, dk, dv, delta = attention_bwd_ref_varlen(q, k, v, do, cu, 0.9, causal)
        for s in range(len(lens)):
            a, b = cu[s], cu[s + 1]
            for h in range(H):
                g = attention_bwd_ref(q[a:b, h], k[a:b, h], v[a:b, h], do[a:b, h], 0.9, causal)
                for mine, ref in zip((dq[a:b, h], dk[a:b, h], dv[a:b, h], delta[h, a:b]), g):
                    assert np.max(np.abs(mine - ref), initial=0.0) <= 1e-14


def test_bwd_delta_is_rowsum_do_o():
    """delta = rowsum(dO * O) with O from the forward oracle."""
    q, k, v, do = _case(12, 21, 6, 4)
    for causal in (False, True):
        o, _ = attention_ref(q, k, v, 0.3, causal)
        delta = attention_bwd_ref(q, k, v, do, 0.3, causal)[3]
        assert np.max(np.abs(delta - np.sum(do * o, axis=1))) <= 1e-14


def test_bwd_recompute_equals_definition():
    """Tiling and recomputation do not change the result (float64 noise),
    for causal, full and band masks and ragged block sizes."""
    q, k, v, do = _case(13, 150, 16, 16, qk=1.5)
    for causal, window in ((False, None), (True, None), (False, (20, 7))):
        ref = attention_bwd_ref(q, k, v, do, 0.25, causal, window=window)[:3]
        o, lse = forward_for_backward(q, k, v, 0.25, causal, window=window)
        for br, bc in [(1, 1), (7, 3), (16, 64), (64, 16), (128, 128), (150, 150)]:
            got = attention_bwd_recompute(q, k, v, do, o, lse, 0.25, causal, Br=br, Bc=bc,
                                          window=window)
            for a, b in zip(got, ref):
                assert np.max(np.abs(a - b)) <= 1e-12


@pytest.mark.parametrize("window", [(0, 0), (2, 1), (-1, 3), (4, -1), (64, 64)])
def test_bwd_window_against_torch(window):
    """The band (DEMO 6's |i - j| <= 64 and others) as an explicit boolean
    mask in torch's float64 autograd."""
    n = 80
    q, k, v, do = _case(14, n, 8, 5)
    dq, dk, dv, _ = attention_bwd_ref(q, k, v, do, 0.5, False, window=window)
    wl, wr = window
    i, j = np.arange(n)[:, None], np.arange(n)[None, :]
    keep = np.ones((n, n), dtype=bool)
    if wl >= 0:
        keep &= j >= i - wl
    if wr >= 0:
        keep &= j <= i + wr
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    out = torch.nn.functional.scaled_dot_product_attention(
        tq[None, None], tk[None, None], tv[None, None], attn_mask=torch.tensor(keep), scale=0.5)[0, 0]
    out.backward(torch.tensor(do, dtype=torch.float64))
    for mine, ref in ((dq, tq.grad), (dk, tk.grad), (dv, tv.grad)):
        assert np.max(np.abs(mine - ref.numpy())) <= 1e-12


def test_bwd_batched_leading_dims():
    """[B, H, N, D] is a loop over (b, h) heads with nothing shared."""
    r = _rng(15)
    q, k, v, do = (r.normal(size=(2, 3, 9, 4)) for _ in range(4))
    got = attention_bwd_ref(q, k, v, do, 0.5, True)
    for b in range(2):
        for h in range(3):
            ref = attention_bwd_ref(q[b, h], k[b, h], v[b, h], do[b, h], 0.5, True)
            for a, c in zip(got, ref):
                assert np.array_equal(a[b, h], c)


@pytest.mark.parametrize("pin", BWD_PINS, ids=lambda p: p.__name__)
def test_bwd_sampled_pins(pin):
    """Every row and key taken one at a time, in reversed order."""
    from oracle import attention_bwd_sampled

    def grad(q, k, v, do, s, c):
        n = np.asarray(q).shape[0]
        idx = np.arange(n)[::-1]
        dq, dk, dv = attention_bwd_sampled(q, k, v, do, s, c, idx, idx)
        return dq[::-1], dk[::-1], dv[::-1]
    pin(grad)


def test_bwd_sampled_band_matches_definition():
    from oracle import attention_bwd_sampled
    q, k, v, do = _case(16, 90, 8, 5)
    for causal, window in ((False, (10, 3)), (True, None), (False, (-1, 7))):
        ref = attention_bwd_ref(q, k, v, do, 0.5, causal, window=window)
        rows, keys = [0, 1, 44, 89], [0, 30, 88, 89]
        dq, dk, dv = attention_bwd_sampled(q, k, v, do, 0.5, causal, rows, keys, window=window)
        assert np.max(np.abs(dq - ref[0][rows])) <= 1e-13
        assert np.max(np.abs(dk - ref[1][keys])) <= 1e-13
        assert np.max(np.abs(dv - ref[2][keys])) <= 1e-13


# ------------------------------------------------ gradient magnitudes --
# attention_bwd_magnitudes gives, per gradient element, the sum of the
# absolute values of its terms: the scale of the per-element error bound in
# the GPU parity tests.  Pinned by the triangle inequality, by the case
# without cancellation (equality) and by a one-key closed form.

@pytest.mark.parametrize("causal, window", [(False, None), (True, None), (False, (5, 3))])
def test_bwd_magnitudes_bound_the_gradients(causal, window):
    rng = np.random.default_rng(11)
    q, k, v, do = (rng.standard_normal((2, 41, 16)) for _ in range(4))
    grads = attention_bwd_ref(q, k, v, do, 0.3, causal, window=window)[:3]
    mags = attention_bwd_magnitudes(q, k, v, do, 0.3, causal, window=window)
    for g, m in zip(grads, mags):
        assert g.shape == m.shape
        assert np.all(m >= 0)
        assert np.all(np.abs(g) <= m * (1 + 1e-12) + 1e-300)
        # a real bound, not a loose constant: somewhere within a factor 2
        assert np.max(np.abs(g) / np.maximum(m, 1e-300)) > 0.5


def test_bwd_magnitudes_equal_dv_without_cancellation():
    rng = np.random.default_rng(12)
    q, k, v = (rng.standard_normal((30, 8)) for _ in range(3))
    do = np.abs(rng.standard_normal((30, 8)))          # P >= 0, dO >= 0: no cancellation in dV
    dv = attention_bwd_ref(q, k, v, do, 0.5, True)[2]
    mv = attention_bwd_magnitudes(q, k, v, do, 0.5, True)[2]
    np.testing.assert_allclose(mv, dv, rtol=1e-13, atol=0)


def test_bwd_magnitudes_one_key_closed_form():
    """n = 1: P = 1, O = V, dP = dO.V = D, so dS = 0 and the gradients of Q, K
    vanish, while their magnitudes are scale (|dO.V| + sum |dO| |V|) |K| (and
    |Q|); M_dV = |dO|."""
    q = np.array([[0.5, -2.0, 1.0, 3.0]])
    k = np.array([[-1.0, 0.25, 2.0, -0.5]])
    v = np.array([[1.0, 1.0, -2.0, 0.5]])
    do = np.array([[1.0, -1.0, 0.5, 2.0]])
    scale = 0.7
    dq, dk, dv, _ = attention_bwd_ref(q, k, v, do, scale, False)
    mq, mk, mv = attention_bwd_magnitudes(q, k, v, do, scale, False)
    dpv = float((do @ v.T)[0, 0])                     # dO . V = D
    dabs = float(np.sum(np.abs(do) * np.abs(v)))
    np.testing.assert_allclose(dq, 0.0, atol=1e-15)
    np.testing.assert_allclose(dk, 0.0, atol=1e-15)
    np.testing.assert_allclose(mq, scale * (abs(dpv) + dabs) * np.abs(k), rtol=1e-15)
    np.testing.assert_allclose(mk, scale * (abs(dpv) + dabs) * np.abs(q), rtol=1e-15)
    np.testing.assert_allclose(mv, np.abs(do), rtol=1e-15)
    np.testing.assert_allclose(dv, do, rtol=1e-15)
