"""Float64 CPU oracle for the gradients of O = softmax(scale * Q K^T) V.

TEST INFRASTRUCTURE ONLY: imported by ``tests/`` and ``bench.py``'s
CPU-baseline leg, never by the product path.  It shares no code with the
CUDA library.

Sources (page titles and sections):

* "FlashAttention -- for programmers, not researchers."
  (flash_attention_from_scratch.py), STAGE 5: the backward pass does not
  keep the (n, n) probability matrix of the forward pass; it recomputes the
  score tiles from the per-row statistics the forward pass stored, paying
  one extra score matmul.  DEMO 5 prints the resulting memory / FLOP trade.
* "FlashAttention" (dao-ailab/flash-attention docs page), "Application in
  Backward Pass (5 MMAs)": the five contractions S = Q K^T, dP = dO V^T,
  dV = P^T dO, dK = dS^T Q, dQ = dS K.

Readings where the pages are silent (each is listed in the design notes):

* dS is the derivative of the row softmax: with D_i = sum_c dO[i,c] O[i,c]
  (= sum_j P[i,j] dP[i,j]), dS = P * (dP - D_i), elementwise.  The scale
  enters dQ and dK once, since S = scale * (Q K^T).
* the per-row statistic the forward pass stores is L = m + log l, so the
  recomputed probabilities are P = exp(scale * Q K^T - L) on unmasked
  entries and 0 on masked ones;
* rows with no unmasked key (never the case for the masks used here) give
  zero gradients.
"""

from __future__ import annotations

import numpy as np

from .attention import _attend, _f64


def _mask(n: int, rows: np.ndarray, causal: bool, window) -> np.ndarray:
    """Boolean [r, n]: True where key j is visible to the query at row_pos."""
    keys = np.arange(n)[None, :]
    r = rows[:, None]
    keep = np.ones((rows.shape[0], n), dtype=bool)
    if causal:
        keep &= keys <= r
    if window is not None:
        wl, wr = window
        if wl >= 0:
            keep &= keys >= r - wl
        if wr >= 0:
            keep &= keys <= r + wr
    return keep


def _bwd_head(q, k, v, do, scale: float, causal: bool, window=None):
    """Gradients of one head, from the plain definition (explicit P).

    q, k: [n, d]; v, do: [n, dv].  Returns (dq, dk, dv, delta) in float64,
    with delta[i] = sum_c dO[i, c] O[i, c].
    """
    n = q.shape[0]
    if n == 0:
        return np.zeros_like(q), np.zeros_like(k), np.zeros_like(v), np.zeros(0)
    keep = _mask(n, np.arange(n), causal, window)
    s = np.where(keep, scale * (q @ k.T), -np.inf)
    m = s.max(axis=1, keepdims=True)
    live = np.isfinite(m[:, 0])
    e = np.where(keep, np.exp(s - np.where(live[:, None], m, 0.0)), 0.0)
    l = e.sum(axis=1, keepdims=True)
    p = np.where(live[:, None], e / np.where(live[:, None], l, 1.0), 0.0)
    o = p @ v
    dv = p.T @ do                                   # dV = P^T dO
    dp = do @ v.T                                   # dP = dO V^T
    delta = np.sum(do * o, axis=1)                  # D_i = rowsum(dO * O)
    ds = p * (dp - delta[:, None])                  # softmax derivative
    dq = scale * (ds @ k)                           # dQ = scale dS K
    dk = scale * (ds.T @ q)                         # dK = scale dS^T Q
    return dq, dk, dv, delta


def attention_bwd_ref(q, k, v, do, scale: float, causal: bool, window=None):
    """Gradients (dQ, dK, dV) of sum(O * dO) for O = attention(Q, K, V).

    Any leading batch dimensions; q, k: ``[..., N, D]``, v, do:
    ``[..., N, Dv]``.  Returns float64 (dq, dk, dv, delta) with
    ``delta = rowsum(dO * O)`` of shape ``[..., N]``.
    """
    qf, kf, vf, dof = _f64(q), _f64(k), _f64(v), _f64(do)
    lead = qf.shape[:-2]
    n, d = qf.shape[-2:]
    dvd = vf.shape[-1]
    nb = int(np.prod(lead, dtype=np.int64))
    qf, kf = qf.reshape(nb, n, d), kf.reshape(nb, n, d)
    vf, dof = vf.reshape(nb, n, dvd), dof.reshape(nb, n, dvd)
    dq, dk, dv = np.zeros_like(qf), np.zeros_like(kf), np.zeros_like(vf)
    delta = np.zeros((qf.shape[0], n))
    for h in range(qf.shape[0]):
        dq[h], dk[h], dv[h], delta[h] = _bwd_head(qf[h], kf[h], vf[h], dof[h], float(scale),
                                                  causal, window)
    return (dq.reshape(*lead, n, d), dk.reshape(*lead, n, d), dv.reshape(*lead, n, dvd),
            delta.reshape(*lead, n))


def attention_bwd_magnitudes(q, k, v, do, scale: float, causal: bool, window=None):
    """Per-element magnitudes of the gradient sums, for error bounds.

    Each gradient element is a sum of products (the five contractions of
    "Application in Backward Pass (5 MMAs)"); rounding a factor of every
    term by a relative u moves the sum by at most u times the sum of the
    terms' absolute values.  These are those sums, from the same P and dP as
    ``_bwd_head``, with every factor replaced by its absolute value, D_i
    included (a sum itself, D_i = sum_c dO[i,c] O[i,c]):

        M_dV = P^T |dO|,   |D|_i = sum_c |dO[i,c]| |O[i,c]|,
        M_dS = P (|dP| + |D|_i),
        M_dQ = scale M_dS |K|,   M_dK = scale M_dS^T |Q|.

    By the triangle inequality |dQ| <= M_dQ, |dK| <= M_dK, |dV| <= M_dV
    elementwise.  Same shapes and leading dimensions as attention_bwd_ref.
    """
    qf, kf, vf, dof = _f64(q), _f64(k), _f64(v), _f64(do)
    lead = qf.shape[:-2]
    n, d = qf.shape[-2:]
    dvd = vf.shape[-1]
    nb = int(np.prod(lead, dtype=np.int64))
    qf, kf = qf.reshape(nb, n, d), kf.reshape(nb, n, d)
    vf, dof = vf.reshape(nb, n, dvd), dof.reshape(nb, n, dvd)
    mq, mk, mv = np.zeros_like(qf), np.zeros_like(kf), np.zeros_like(vf)
    for h in range(nb):
        if n == 0:
            continue
        keep = _mask(n, np.arange(n), causal, window)
        s = np.where(keep, scale * (qf[h] @ kf[h].T), -np.inf)
        m = s.max(axis=1, keepdims=True)
        live = np.isfinite(m[:, 0])
        e = np.where(keep, np.exp(s - np.where(live[:, None], m, 0.0)), 0.0)
        l = e.sum(axis=1, keepdims=True)
        p = np.where(live[:, None], e / np.where(live[:, None], l, 1.0), 0.0)
        o = p @ vf[h]
        dp = dof[h] @ vf[h].T
        dabs = np.sum(np.abs(dof[h]) * np.abs(o), axis=1)
        mds = p * (np.abs(dp) + dabs[:, None])
        mv[h] = p.T @ np.abs(dof[h])
        mq[h] = scale * (mds @ np.abs(kf[h]))
        mk[h] = scale * (mds.T @ np.abs(qf[h]))
    return mq.reshape(*lead, n, d), mk.reshape(*lead, n, d), mv.reshape(*lead, n, dvd)


def attention_bwd_ref_varlen(q, k, v, do, cu_seqlens, scale: float, causal: bool):
    """Varlen gradients: ``[total, H, D]`` packing, sequence s owns tokens
    ``cu[s] .. cu[s+1]-1`` and attends only within itself.  Returns
    (dq, dk, dv) as ``[total, H, D]`` and delta as ``[H, total]``."""
    qf, kf, vf, dof = _f64(q), _f64(k), _f64(v), _f64(do)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    dq, dk, dv = np.zeros_like(qf), np.zeros_like(kf), np.zeros_like(vf)
    delta = np.zeros((qf.shape[1], qf.shape[0]))
    for s in range(len(cu) - 1):
        a, b = int(cu[s]), int(cu[s + 1])
        for h in range(qf.shape[1]):
            g = _bwd_head(qf[a:b, h], kf[a:b, h], vf[a:b, h], dof[a:b, h], float(scale), causal)
            dq[a:b, h], dk[a:b, h], dv[a:b, h], delta[h, a:b] = g
    return dq, dk, dv, delta


def attention_bwd_recompute(q, k, v, do, o, lse, scale: float, causal: bool, Br: int = 64,
                            Bc: int = 64, window=None):
    """The backward pass of STAGE 5 for one head: P is never kept; each
    (query block, key block) tile of it is recomputed from Q, K and the
    stored L as exp(scale Q_i K_j^T - L_i), then the five contractions run
    tile by tile: dV_j += P^T dO_i, dP = dO_i V_j^T, dS = P (dP - D_i),
    dK_j += scale dS^T Q_i, dQ_i += scale dS K_j.  D_i = rowsum(dO_i O_i)
    uses the stored O.

    q, k: [n, d]; v, do, o: [n, dv]; lse: [n].  Returns (dq, dk, dv).
    """
    qf, kf, vf, dof, of, lf = (_f64(x) for x in (q, k, v, do, o, lse))
    n = qf.shape[0]
    dq, dk, dv = np.zeros_like(qf), np.zeros_like(kf), np.zeros_like(vf)
    delta = np.sum(dof * of, axis=1)
    for j0 in range(0, n, Bc):
        kj, vj = kf[j0:j0 + Bc], vf[j0:j0 + Bc]
        cols = np.arange(j0, min(n, j0 + Bc))
        for i0 in range(0, n, Br):
            rows = np.arange(i0, min(n, i0 + Br))
            keep = _mask(n, rows, causal, window)[:, cols]
            if not keep.any():
                continue
            s = scale * (qf[rows] @ kj.T)
            with np.errstate(over="ignore", invalid="ignore"):
                p = np.where(keep, np.exp(s - lf[rows][:, None]), 0.0)
            dv[cols] += p.T @ dof[rows]
            dp = dof[rows] @ vj.T
            ds = p * (dp - delta[rows][:, None])
            dk[cols] += scale * (ds.T @ qf[rows])
            dq[rows] += scale * (ds @ kj)
    return dq, dk, dv


def forward_for_backward(q, k, v, scale: float, causal: bool, window=None):
    """O and L of one head (the forward oracle), as the backward pass's
    stored inputs."""
    qf, kf, vf = _f64(q), _f64(k), _f64(v)
    return _attend(qf, kf, vf, float(scale), causal, np.arange(qf.shape[0]), window=window)


def _visible_col(n: int, j: int, causal: bool, window) -> np.ndarray:
    """Boolean [n]: rows i that see key j."""
    i = np.arange(n)
    keep = np.ones(n, dtype=bool)
    if causal:
        keep &= j <= i
    if window is not None:
        wl, wr = window
        if wl >= 0:
            keep &= j >= i - wl
        if wr >= 0:
            keep &= j <= i + wr
    return keep


def attention_bwd_sampled(q, k, v, do, scale: float, causal: bool, rows, keys, window=None):
    """dQ at the query rows ``rows`` and dK, dV at the keys ``keys`` of ONE
    head, without forming any (n, n) matrix: O and L of every row come from
    the forward definition, then each requested row of dQ and column of dK,
    dV is the definition above restricted to it (dQ_i = scale sum_j dS_ij K_j,
    dK_j = scale sum_i dS_ij Q_i, dV_j = sum_i P_ij dO_i).

    q, k: [n, d]; v, do: [n, dv].  Returns (dq [len(rows), d],
    dk [len(keys), d], dv [len(keys), dv]) in float64.
    """
    qf, kf, vf, dof = _f64(q), _f64(k), _f64(v), _f64(do)
    n = qf.shape[0]
    o, lse = _attend(qf, kf, vf, float(scale), causal, np.arange(n), window=window)
    delta = np.sum(dof * o, axis=1)
    rows, keys = np.asarray(rows, dtype=np.int64), np.asarray(keys, dtype=np.int64)
    dq = np.zeros((len(rows), qf.shape[1]))
    for t, i in enumerate(rows):
        keep = _mask(n, np.array([i]), causal, window)[0]
        with np.errstate(over="ignore", invalid="ignore"):
            p = np.where(keep, np.exp(scale * (kf @ qf[i]) - lse[i]), 0.0)
        ds = p * (vf @ dof[i] - delta[i])
        dq[t] = scale * (ds @ kf)
    dk = np.zeros((len(keys), kf.shape[1]))
    dv = np.zeros((len(keys), vf.shape[1]))
    for t, j in enumerate(keys):
        keep = _visible_col(n, int(j), causal, window)
        with np.errstate(over="ignore", invalid="ignore"):
            p = np.where(keep, np.exp(scale * (qf @ kf[j]) - lse), 0.0)
        ds = p * (dof @ vf[j] - delta)
        dv[t] = p @ dof
        dk[t] = scale * (ds @ qf)
    return dq, dk, dv
