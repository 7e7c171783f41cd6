"""Pins for the CPU oracle: closed forms, brute force, library routines and
the pages' worked examples.  CPU only.

Each ``pin_*`` helper takes an attention implementation with the signature
``ref(q, k, v, scale, causal) -> (O, L)`` for ``[N, D]`` inputs, so that
``test_oracle_mutations.py`` can run the same pins against deliberately
broken copies of the oracle and show that every planted mistake is caught.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import (attention_ref, attention_ref_varlen, attention_rows,
                    attention_tiled, merge_partials)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------------------
# brute force in pure Python: no NumPy, no max shift, math.fsum everywhere.
# The textbook definition softmax_j = exp(s_j) / sum exp(s_j) is used as is;
# the inputs are small enough that nothing overflows.
# ---------------------------------------------------------------------------
def brute_force(q, k, v, scale, causal):
    n, d = len(q), len(q[0])
    dv = len(v[0])
    O, L = [], []
    for i in range(n):
        keys = [j for j in range(n) if not (causal and j > i)]
        w = [math.exp(scale * math.fsum(q[i][t] * k[j][t] for t in range(d)))
             for j in keys]
        z = math.fsum(w)
        O.append([math.fsum(w[a] * v[j][c] for a, j in enumerate(keys)) / z
                  for c in range(dv)])
        L.append(math.log(z))
    return O, L


# ---------------------------------------------------------------------------
# pins, parameterised by the implementation under test
# ---------------------------------------------------------------------------
def pin_brute_force(ref):
    for seed, (n, d) in enumerate([(1, 1), (2, 3), (3, 4), (5, 2), (8, 4),
                                   (7, 5)]):
        r = _rng(100 + seed)
        q, k, v = (r.normal(size=(n, d)) for _ in range(3))
        v = r.normal(size=(n, d + 1))  # D_v != D_qk catches a swapped operand
        for causal in (False, True):
            scale = 0.37
            O, L = ref(q, k, v, scale, causal)
            Ob, Lb = brute_force(q.tolist(), k.tolist(), v.tolist(), scale,
                                 causal)
            assert np.max(np.abs(O - np.array(Ob))) <= 1e-14
            assert np.max(np.abs(L - np.array(Lb))) <= 1e-14


def pin_n1_and_n2(ref):
    r = _rng(7)
    q, k, v = r.normal(size=(1, 6)), r.normal(size=(1, 6)), r.normal(size=(1, 6))
    O, L = ref(q, k, v, 0.5, False)
    assert np.allclose(O[0], v[0], atol=0, rtol=1e-15)      # one key: O = V_0
    assert abs(L[0] - 0.5 * float(q[0] @ k[0])) <= 1e-14    # L = the score
    # two keys: weight of key 1 is the logistic function of the difference
    q, k, v = r.normal(size=(2, 6)), r.normal(size=(2, 6)), r.normal(size=(2, 3))
    O, L = ref(q, k, v, 0.5, False)
    for i in range(2):
        s0, s1 = 0.5 * float(q[i] @ k[0]), 0.5 * float(q[i] @ k[1])
        w1 = 1.0 / (1.0 + math.exp(s0 - s1))
        assert np.allclose(O[i], (1 - w1) * v[0] + w1 * v[1], atol=1e-14)
        assert abs(L[i] - (max(s0, s1) + math.log1p(math.exp(-abs(s0 - s1))))) < 1e-14


def pin_zero_query(ref):
    """Q = 0 makes every score 0: O is the mean of the attended V rows and
    L = ln(#attended keys), for any scale."""
    r = _rng(3)
    n, d = 37, 8
    k, v = r.normal(size=(n, d)), r.normal(size=(n, 5))
    q = np.zeros((n, d))
    for causal in (False, True):
        O, L = ref(q, k, v, 1.7, causal)
        for i in range(n):
            cnt = i + 1 if causal else n
            assert np.allclose(O[i], v[:cnt].mean(axis=0), atol=1e-13)
            assert abs(L[i] - math.log(cnt)) <= 1e-13


def pin_identical_keys(ref):
    """All K rows equal: uniform weights, L = scale q.k + ln(#keys)."""
    r = _rng(4)
    n, d = 29, 8
    q, v = r.normal(size=(n, d)), r.normal(size=(n, 3))
    krow = r.normal(size=d)
    k = np.tile(krow, (n, 1))
    for causal in (False, True):
        O, L = ref(q, k, v, 0.3, causal)
        for i in range(n):
            cnt = i + 1 if causal else n
            assert np.allclose(O[i], v[:cnt].mean(axis=0), atol=1e-13)
            assert abs(L[i] - (0.3 * float(q[i] @ krow) + math.log(cnt))) <= 1e-12


def pin_shift_invariance(ref):
    """K -> K + 1 u^T adds scale q_i.u to all of row i's scores: O unchanged,
    L_i moves by exactly that amount."""
    r = _rng(5)
    n, d = 33, 8
    q, k, v = r.normal(size=(n, d)), r.normal(size=(n, d)), r.normal(size=(n, d))
    u = r.normal(size=d) * 3
    for causal in (False, True):
        O0, L0 = ref(q, k, v, 0.25, causal)
        O1, L1 = ref(q, k + u[None, :], v, 0.25, causal)
        assert np.max(np.abs(O1 - O0)) <= 1e-12
        assert np.max(np.abs((L1 - L0) - 0.25 * (q @ u))) <= 1e-11


def pin_permutation(ref):
    r = _rng(6)
    n, d = 21, 8
    q, k, v = r.normal(size=(n, d)), r.normal(size=(n, d)), r.normal(size=(n, 4))
    O, L = ref(q, k, v, 0.4, False)
    p = r.permutation(n)
    Ok, Lk = ref(q, k[p], v[p], 0.4, False)      # keys/values jointly
    assert np.max(np.abs(Ok - O)) <= 1e-13 and np.max(np.abs(Lk - L)) <= 1e-13
    Oq, Lq = ref(q[p], k, v, 0.4, False)         # queries
    assert np.max(np.abs(Oq - O[p])) <= 1e-13 and np.max(np.abs(Lq - L[p])) <= 1e-13


def pin_convex(ref):
    """Rows of P sum to one (V = ones gives O = 1) and O is a convex
    combination of the attended V rows."""
    r = _rng(8)
    n, d = 40, 8
    q, k = r.normal(size=(n, d)) * 2, r.normal(size=(n, d)) * 2
    for causal in (False, True):
        O, _ = ref(q, k, np.ones((n, 1)), 0.5, causal)
        assert np.max(np.abs(O - 1.0)) <= 1e-12
        v = r.normal(size=(n, 3))
        O, _ = ref(q, k, v, 0.5, causal)
        for i in range(n):
            att = v[: i + 1] if causal else v
            assert np.all(O[i] >= att.min(axis=0) - 1e-12)
            assert np.all(O[i] <= att.max(axis=0) + 1e-12)


def pin_torch_library(ref):
    """torch's own CPU scaled_dot_product_attention (float64) and logsumexp."""
    r = _rng(9)
    n, d = 50, 16
    q, k, v = r.normal(size=(n, d)), r.normal(size=(n, d)), r.normal(size=(n, d))
    for causal in (False, True):
        O, L = ref(q, k, v, 0.2, causal)
        tq, tk, tv = (torch.from_numpy(x)[None, None] for x in (q, k, v))
        To = torch.nn.functional.scaled_dot_product_attention(
            tq, tk, tv, is_causal=causal, scale=0.2)[0, 0].numpy()
        s = 0.2 * (torch.from_numpy(q) @ torch.from_numpy(k).T)
        if causal:
            s = s.masked_fill(torch.ones(n, n, dtype=torch.bool).triu(1),
                              float("-inf"))
        TL = torch.logsumexp(s, dim=-1).numpy()
        assert np.max(np.abs(O - To)) <= 1e-12
        assert np.max(np.abs(L - TL)) <= 1e-12


def pin_overflow_demo9(ref):
    """The four scores printed by DEMO 9 overflow exp() without the max
    shift; the oracle must give the finite closed form."""
    with open(os.path.join(GOLDEN, "demo9_overflow.json")) as f:
        scores = json.load(f)["scores"]
    n, d = 4, 64
    q = np.zeros((n, d))
    q[:, 0] = 1.0
    k = np.zeros((n, d))
    k[:, 0] = scores             # row i's scores are exactly the page's list
    v = np.eye(n, d)             # O row = the weight vector
    O, L = ref(q, k, v, 1.0, False)
    smax = max(scores)
    z = math.fsum(math.exp(s - smax) for s in scores)
    w = [math.exp(s - smax) / z for s in scores]
    assert np.all(np.isfinite(O)) and np.all(np.isfinite(L))
    assert np.max(np.abs(O[0, :n] - np.array(w))) <= 1e-15
    assert abs(L[0] - (810.0 + math.log1p(math.exp(-5) + math.exp(-10) + math.exp(-20)))) <= 1e-12


ALL_PINS = [pin_brute_force, pin_n1_and_n2, pin_zero_query, pin_identical_keys,
            pin_shift_invariance, pin_permutation, pin_convex,
            pin_torch_library, pin_overflow_demo9]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_attention_ref_pins(pin):
    pin(attention_ref)


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
@pytest.mark.parametrize("blocks", [(1, 1), (4, 3), (16, 16), (64, 128)])
def test_attention_tiled_pins(pin, blocks):
    br, bc = blocks
    pin(lambda q, k, v, s, c: attention_tiled(q, k, v, s, c, Br=br, Bc=bc))


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_attention_rows_pins(pin):
    def ref(q, k, v, s, c):
        rows = np.arange(np.asarray(q).shape[0])[::-1]   # reversed order
        O, L = attention_rows(q, k, v, s, c, rows)
        return O[::-1], L[::-1]
    pin(ref)


def _varlen_as_dense(q, k, v, s, c):
    """Run a single-sequence varlen call (with an empty sequence before and
    after it) on [N, D] inputs."""
    n = np.asarray(q).shape[0]
    cu = np.array([0, 0, n, n], dtype=np.int32)
    O, L = attention_ref_varlen(np.asarray(q)[:, None], np.asarray(k)[:, None],
                                np.asarray(v)[:, None], cu, s, c)
    return O[:, 0], L[0]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_attention_varlen_pins(pin):
    pin(_varlen_as_dense)


def test_varlen_sequences_are_independent():
    """Per-sequence closed form (Q = 0) and brute force in a packed batch:
    a sequence must never see another's keys."""
    r = _rng(11)
    lens = [3, 0, 5, 1, 4]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    tot, H, d = int(cu[-1]), 2, 4
    q = np.zeros((tot, H, d))
    k, v = r.normal(size=(tot, H, d)), r.normal(size=(tot, H, 3))
    for causal in (False, True):
        O, L = attention_ref_varlen(q, k, v, cu, 0.9, causal)
        for s in range(len(lens)):
            a, b = cu[s], cu[s + 1]
            for i in range(b - a):
                cnt = i + 1 if causal else b - a
                for h in range(H):
                    assert np.allclose(O[a + i, h], v[a:a + cnt, h].mean(0), atol=1e-13)
                    assert abs(L[h, a + i] - math.log(cnt)) <= 1e-13
    q = r.normal(size=(tot, H, d))
    for causal in (False, True):
        O, L = attention_ref_varlen(q, k, v, cu, 0.9, causal)
        for s in range(len(lens)):
            a, b = cu[s], cu[s + 1]
            for h in range(H):
                if b == a:
                    continue
                Ob, Lb = brute_force(q[a:b, h].tolist(), k[a:b, h].tolist(),
                                     v[a:b, h].tolist(), 0.9, causal)
                assert np.max(np.abs(O[a:b, h] - np.array(Ob))) <= 1e-14
                assert np.max(np.abs(L[h, a:b] - np.array(Lb))) <= 1e-14


def test_batched_leading_dims():
    """[B, H, N, D] is a loop over (b, h) heads with nothing shared."""
    r = _rng(12)
    q, k, v = (r.normal(size=(2, 3, 9, 4)) for _ in range(3))
    O, L = attention_ref(q, k, v, 0.5, True)
    for b in range(2):
        for h in range(3):
            Ob, Lb = brute_force(q[b, h].tolist(), k[b, h].tolist(),
                                 v[b, h].tolist(), 0.5, True)
            assert np.max(np.abs(O[b, h] - np.array(Ob))) <= 1e-14
            assert np.max(np.abs(L[b, h] - np.array(Lb))) <= 1e-14


def test_block_size_invariance():
    """STAGE 3/4 and DEMO 3/6: the tiled loop computes the same function as
    the one-pass definition -- any block size, float64 noise only."""
    r = _rng(13)
    n, d = 200, 16
    q, k, v = r.normal(size=(n, d)) * 2, r.normal(size=(n, d)) * 2, r.normal(size=(n, d))
    for causal in (False, True):
        O, L = attention_ref(q, k, v, 0.25, causal)
        for br, bc in [(1, 1), (7, 3), (16, 64), (64, 16), (128, 128), (n, n)]:
            Ot, Lt = attention_tiled(q, k, v, 0.25, causal, Br=br, Bc=bc)
            assert np.max(np.abs(Ot - O)) <= 1e-12
            assert np.max(np.abs(Lt - L)) <= 1e-12
    # DEMO 6's exactness claim at its own size: allclose with atol 1e-10
    q, k, v = r.normal(size=(512, 64)) / 8, r.normal(size=(512, 64)) / 8, r.normal(size=(512, 64))
    O, _ = attention_ref(q, k, v, 1.0, False)
    Ot, _ = attention_tiled(q, k, v, 1.0, False, Br=64, Bc=64)
    assert np.allclose(O, Ot, atol=1e-10)


def test_no_rescale_variant_is_wrong():
    """STAGE 4 / DEMO 2: dropping the exp(m_old - m_new) rescale leaves the
    running sum l mixing terms taken against different maxima, so L (which
    carries log l) is wrong, and so are the weights that make O."""
    r = _rng(14)
    n, d = 64, 8
    q, k = r.normal(size=(n, d)) * 2, r.normal(size=(n, d)) * 2
    v = np.eye(n)                 # O row = the effective weight vector
    O, L = attention_ref(q, k, v, 1.0, False)
    Ob, Lb = attention_tiled(q, k, v, 1.0, False, Br=16, Bc=8, rescale=False)
    assert np.max(np.abs(Lb - L)) > 1e-1
    assert np.max(np.abs(Ob - O)) > 1e-2


def test_rows_match_full():
    r = _rng(15)
    n, d = 300, 8
    q, k, v = r.normal(size=(n, d)), r.normal(size=(n, d)), r.normal(size=(n, d))
    rows = [0, 1, 127, 128, 255, 299]
    for causal in (False, True):
        O, L = attention_ref(q, k, v, 0.3, causal)
        Or, Lr = attention_rows(q, k, v, 0.3, causal, rows)
        assert np.max(np.abs(Or - O[rows])) <= 1e-14
        assert np.max(np.abs(Lr - L[rows])) <= 1e-14


def test_bf16_inputs_are_upcast_exactly():
    """bf16 tensors enter the oracle as their exact float64 values."""
    r = torch.Generator().manual_seed(0)
    x = torch.randn(4, 8, generator=r).to(torch.bfloat16)
    O, L = attention_ref(x, x, x, 0.5, False)
    O2, L2 = attention_ref(x.double().numpy(), x.double().numpy(),
                           x.double().numpy(), 0.5, False)
    assert np.array_equal(O, O2) and np.array_equal(L, L2)


# ---------------------------------------------------------------------------
# key ranges and the split-key merge
# ---------------------------------------------------------------------------
def _split_points(n, g, rng):
    cuts = np.sort(rng.choice(np.arange(1, n), size=g - 1, replace=False)) if g > 1 else []
    return [0, *[int(c) for c in cuts], n]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("parts", [1, 2, 3, 7])
def test_merge_of_key_ranges_is_full_attention(causal, parts):
    """Attention over disjoint key ranges, merged, is attention over all keys
    (the identity behind split-key attention), to float64 noise."""
    r = _rng(20 + parts)
    n, d = 61, 8
    q, k, v = r.normal(size=(n, d)) * 2, r.normal(size=(n, d)) * 2, r.normal(size=(n, 5))
    rows = np.arange(n)
    cuts = _split_points(n, parts, r)
    O_p, L_p = zip(*[attention_rows(q, k, v, 0.4, causal, rows, a, b)
                     for a, b in zip(cuts[:-1], cuts[1:])])
    O, L = merge_partials(np.stack(O_p), np.stack(L_p))
    Of, Lf = attention_ref(q, k, v, 0.4, causal)
    assert np.max(np.abs(O - Of)) <= 1e-13 and np.max(np.abs(L - Lf)) <= 1e-12
    # part order does not matter
    perm = r.permutation(len(O_p))
    O2, L2 = merge_partials(np.stack(O_p)[perm], np.stack(L_p)[perm])
    assert np.max(np.abs(O2 - Of)) <= 1e-13 and np.max(np.abs(L2 - Lf)) <= 1e-12


def test_key_range_brute_force():
    """A key sub-range is plain attention over those keys (brute force)."""
    r = _rng(30)
    n, d = 7, 3
    q, k, v = r.normal(size=(n, d)), r.normal(size=(n, d)), r.normal(size=(n, 2))
    for causal in (False, True):
        for a, b in [(0, 7), (2, 5), (3, 4), (5, 7)]:
            O, L = attention_rows(q, k, v, 0.8, causal, np.arange(n), a, b)
            for i in range(n):
                keys = [j for j in range(a, b) if not (causal and j > i)]
                if not keys:
                    assert L[i] == -np.inf and np.all(O[i] == 0)
                    continue
                w = [math.exp(0.8 * math.fsum(q[i][t] * k[j][t] for t in range(d))) for j in keys]
                z = math.fsum(w)
                assert abs(L[i] - math.log(z)) <= 1e-14
                for c in range(2):
                    ref = math.fsum(w[x] * v[j][c] for x, j in enumerate(keys)) / z
                    assert abs(O[i][c] - ref) <= 1e-14


def test_merge_special_cases():
    r = _rng(31)
    o = r.normal(size=(4, 6, 3))
    l = r.normal(size=(4, 6))
    # one part: identity
    O, L = merge_partials(o[:1], l[:1])
    assert np.allclose(O, o[0], atol=1e-15) and np.allclose(L, l[0], atol=1e-15)
    # empty parts (L = -inf) are ignored
    l2 = l.copy()
    l2[1] = -np.inf
    O, L = merge_partials(o, l2)
    O3, L3 = merge_partials(o[[0, 2, 3]], l[[0, 2, 3]])
    assert np.allclose(O, O3, atol=1e-14) and np.allclose(L, L3, atol=1e-14)
    # all parts empty: O = 0, L = -inf
    O, L = merge_partials(o, np.full_like(l, -np.inf))
    assert np.all(O == 0) and np.all(L == -np.inf)
    # two equal parts: O unchanged, L + ln 2
    O, L = merge_partials(np.stack([o[0], o[0]]), np.stack([l[0], l[0]]))
    assert np.allclose(O, o[0], atol=1e-14) and np.allclose(L, l[0] + math.log(2), atol=1e-14)
    # huge L values do not overflow
    O, L = merge_partials(np.stack([o[0], o[1]]), np.stack([l[0] + 800, l[1] + 810]))
    assert np.all(np.isfinite(O)) and np.all(np.isfinite(L))


# ---------------------------------------------------------------------------
# the local band (DEMO 6's |i - j| <= 64, and general (wl, wr) windows)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("window", [(0, 0), (1, 2), (3, 0), (0, 5), (-1, 1), (2, -1)])
def test_window_brute_force(window):
    r = _rng(40)
    n, d = 8, 3
    q, k, v = r.normal(size=(n, d)), r.normal(size=(n, d)), r.normal(size=(n, 2))
    wl, wr = window
    O, L = attention_ref(q, k, v, 0.6, False, window=window)
    for i in range(n):
        keys = [j for j in range(n) if (wl < 0 or j >= i - wl) and (wr < 0 or j <= i + wr)]
        w = [math.exp(0.6 * math.fsum(q[i][t] * k[j][t] for t in range(d))) for j in keys]
        z = math.fsum(w)
        assert abs(L[i] - math.log(z)) <= 1e-14
        for c in range(2):
            assert abs(O[i][c] - math.fsum(w[x] * v[j][c] for x, j in enumerate(keys)) / z) <= 1e-14


def test_window_closed_forms():
    r = _rng(41)
    n, d = 50, 8
    q, k, v = r.normal(size=(n, d)), r.normal(size=(n, d)), r.normal(size=(n, d))
    # (0, 0): every row sees only its own key: O = V, L = scale q.k
    O, L = attention_ref(q, k, v, 0.3, False, window=(0, 0))
    assert np.max(np.abs(O - v)) <= 1e-14
    assert np.max(np.abs(L - 0.3 * np.sum(q * k, axis=1))) <= 1e-13
    # (-1, 0) is the causal mask; (-1, -1) is no mask
    Oc, Lc = attention_ref(q, k, v, 0.3, True)
    Ow, Lw = attention_ref(q, k, v, 0.3, False, window=(-1, 0))
    assert np.array_equal(Oc, Ow) and np.array_equal(Lc, Lw)
    Of, Lf = attention_ref(q, k, v, 0.3, False)
    Ow, Lw = attention_ref(q, k, v, 0.3, False, window=(-1, -1))
    assert np.array_equal(Of, Ow) and np.array_equal(Lf, Lw)
    # Q = 0 under a band: O = mean of the V rows inside the band
    O, L = attention_ref(np.zeros((n, d)), k, v, 0.3, False, window=(3, 5))
    for i in range(n):
        lo, hi = max(0, i - 3), min(n, i + 6)
        assert np.allclose(O[i], v[lo:hi].mean(0), atol=1e-13)
        assert abs(L[i] - math.log(hi - lo)) <= 1e-13


def test_window_demo6_band():
    """DEMO 6's local window: softmax over |i - j| <= 64 only -- a different
    function from exact attention (the page's point), equal to the band
    written out as a mask."""
    r = _rng(42)
    n, d = 512, 64
    q, k, v = r.normal(size=(n, d)) / 8, r.normal(size=(n, d)) / 8, r.normal(size=(n, d))
    O, _ = attention_ref(q, k, v, 1.0, False, window=(64, 64))
    s = q @ k.T
    band = np.abs(np.subtract.outer(np.arange(n), np.arange(n))) <= 64
    e = np.exp(np.where(band, s, -np.inf) - np.where(band, s, -np.inf).max(1, keepdims=True))
    assert np.max(np.abs(O - (e / e.sum(1, keepdims=True)) @ v)) <= 1e-13
    Of, _ = attention_ref(q, k, v, 1.0, False)
    assert np.max(np.abs(O - Of)) > 1e-3          # not the same function
