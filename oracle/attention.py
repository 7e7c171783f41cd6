"""Float64 CPU oracle for O = softmax(scale * Q K^T) V and L = log-sum-exp.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py``'s CPU-baseline leg, never by the product path.  It shares no
code with the CUDA library.

Sources (page titles and sections):

* "FlashAttention -- for programmers, not researchers."
  (flash_attention_from_scratch.py):
  - STAGE 1: softmax with the row maximum subtracted before ``exp`` (overflow
    safety that cancels in the ratio);
  - STAGE 2: standard attention -- materialise the (n, n) scores, take the
    softmax along each row, multiply by V;
  - STAGE 3: online softmax -- running max ``m`` and running sum ``l``, the
    sum rescaled by ``exp(m_old - m_new)`` when the max grows;
  - STAGE 4: FlashAttention -- Q row blocks on the outer loop, K/V column
    blocks on the inner loop, ``l`` AND the output rescaled whenever ``m``
    moves, one division by ``l`` at the end.
* "Kernel visualization: Flash Attention 2":
  - "Iteration j = 0": the score is ``scale`` times the dot product
    (scale applied after the dot product);
  - "Write the data back to HBM": the outputs are ``O = O_acc / l`` and the
    single array ``L = m + log(l)`` (natural log).

Readings where the pages are silent (each is listed in the design notes):

* causal: key ``j`` is masked for query ``i`` when ``j > i`` (indices local
  to a sequence);
* a row with no unmasked key gets ``O = 0`` and ``L = -inf``;
* varlen: Q, K, V, O are ``[total, H, D]`` packed token-major, L is
  ``[H, total]``, sequence ``s`` owns tokens ``cu[s] .. cu[s+1]-1`` and
  attends only within itself.
"""

from __future__ import annotations

import numpy as np


def _f64(x) -> np.ndarray:
    """Up-cast an array (NumPy, or a CPU torch tensor of any float dtype) to
    float64 exactly."""
    if hasattr(x, "detach"):  # torch tensor: bf16 has no NumPy dtype
        import torch

        return x.detach().to(device="cpu", dtype=torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def _attend(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float,
            causal: bool, row_pos: np.ndarray, key_lo: int = 0, key_hi=None,
            window=None):
    """One head of standard attention for the query rows ``q`` whose
    positions in the sequence are ``row_pos``, over the keys at positions
    ``key_lo <= j < key_hi`` only (all keys by default; the causal mask uses
    absolute positions).  ``window=(wl, wr)`` keeps key j for row i only if
    ``i - wl <= j <= i + wr`` (a negative bound is unbounded) -- the local
    band of DEMO 6, where ``|i - j| <= 64``.

    q: [r, d]; k, v: [n, d]; returns (O [r, d], L [r]) in float64.
    """
    r, d = q.shape
    n = k.shape[0]
    key_hi = n if key_hi is None else min(int(key_hi), n)
    key_lo = max(0, int(key_lo))
    o = np.zeros((r, v.shape[1]), dtype=np.float64)
    lse = np.full(r, -np.inf, dtype=np.float64)
    if r == 0 or n == 0:
        return o, lse
    # STAGE 2: the full score block, scaled after the dot product.
    s = scale * (q @ k.T)
    key_pos = np.arange(n)
    outside = (key_pos < key_lo) | (key_pos >= key_hi)
    s = np.where(outside[None, :], -np.inf, s)
    if causal:
        s = np.where(key_pos[None, :] > row_pos[:, None], -np.inf, s)
    if window is not None:
        wl, wr = window
        if wl >= 0:
            s = np.where(key_pos[None, :] < row_pos[:, None] - wl, -np.inf, s)
        if wr >= 0:
            s = np.where(key_pos[None, :] > row_pos[:, None] + wr, -np.inf, s)
    # STAGE 1: subtract the row max, exponentiate, normalise.
    m = s.max(axis=1)
    live = np.isfinite(m)
    m_shift = np.where(live, m, 0.0)
    e = np.exp(s - m_shift[:, None])
    l = e.sum(axis=1)
    o[live] = (e[live] @ v) / l[live, None]
    lse[live] = m[live] + np.log(l[live])
    return o, lse


def attention_ref(q, k, v, scale: float, causal: bool, window=None):
    """Standard attention over ``[..., N, D]`` inputs (any leading dims),
    optionally restricted to the local band ``window=(wl, wr)``.

    Returns ``(O [..., N, D], L [..., N])`` in float64.  One (N, N) float64
    score block exists at a time.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    lead = q.shape[:-2]
    n, d = q.shape[-2:]
    qf = q.reshape(-1, n, d)
    kf = k.reshape(-1, k.shape[-2], d)
    vf = v.reshape(-1, v.shape[-2], v.shape[-1])
    o = np.empty((qf.shape[0], n, vf.shape[-1]))
    lse = np.empty((qf.shape[0], n))
    pos = np.arange(n)
    for h in range(qf.shape[0]):
        o[h], lse[h] = _attend(qf[h], kf[h], vf[h], float(scale), causal, pos,
                               window=window)
    return o.reshape(*lead, n, vf.shape[-1]), lse.reshape(*lead, n)


def attention_rows(q, k, v, scale: float, causal: bool, rows, key_lo: int = 0,
                   key_hi=None, window=None):
    """Standard attention for selected query rows of ONE head, optionally
    over a sub-range of the keys ``[key_lo, key_hi)`` (positions absolute).

    q, k, v: ``[N, D]``; ``rows``: integer positions.  Used to check outputs
    of workloads too large for the full oracle, one row at a time, and the
    partial results of a split key range.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    rows = np.asarray(rows, dtype=np.int64)
    return _attend(q[rows], k, v, float(scale), causal, rows, key_lo, key_hi, window)


def merge_partials(o_parts, l_parts):
    """Combine attention results computed over disjoint key ranges.

    o_parts: ``[G, ..., D]`` -- each part normalised over its own keys;
    l_parts: ``[G, ...]`` -- each part's log-sum-exp (``-inf`` for a part with
    no key).  This is STAGE 3's online-softmax update applied part by part:
    carry a running max ``m`` and running sum ``l`` of exp(score - m) plus the
    unnormalised output; when a part raises the max, rescale what was carried
    by exp(m_old - m_new); normalise once at the end.  Returns ``(O, L)``.
    """
    o_parts = np.asarray(o_parts, dtype=np.float64)
    l_parts = np.asarray(l_parts, dtype=np.float64)
    m = np.full(l_parts.shape[1:], -np.inf)
    l = np.zeros(l_parts.shape[1:])
    acc = np.zeros(o_parts.shape[1:])
    for g in range(l_parts.shape[0]):
        lg = l_parts[g]
        m_new = np.maximum(m, lg)
        live = np.isfinite(m_new)
        m_use = np.where(live, m_new, 0.0)
        carry = np.where(np.isfinite(m), np.exp(m - m_use), 0.0)   # rescale of the carry
        w = np.where(np.isfinite(lg), np.exp(lg - m_use), 0.0)     # this part's sum, on m_use
        l = carry * l + w
        acc = carry[..., None] * acc + w[..., None] * o_parts[g]
        m = m_new
    live = l > 0
    o = np.zeros_like(acc)
    o[live] = acc[live] / l[live, None]
    lse = np.full(l.shape, -np.inf)
    lse[live] = m[live] + np.log(l[live])
    return o, lse


def attention_ref_varlen(q, k, v, cu_seqlens, scale: float, causal: bool):
    """Standard attention over a packed batch of variable-length sequences.

    q, k, v: ``[total, H, D]``; ``cu_seqlens``: ``num_seqs + 1`` prefix
    offsets.  Returns ``(O [total, H, D], L [H, total])`` in float64.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    total, nh, _ = q.shape
    o = np.zeros((total, nh, v.shape[-1]))
    lse = np.full((nh, total), -np.inf)
    for s in range(len(cu) - 1):
        a, b = int(cu[s]), int(cu[s + 1])
        pos = np.arange(b - a)
        for h in range(nh):
            o[a:b, h], lse[h, a:b] = _attend(q[a:b, h], k[a:b, h], v[a:b, h],
                                             float(scale), causal, pos)
    return o, lse


def attention_tiled(q, k, v, scale: float, causal: bool, Br: int = 64,
                    Bc: int = 64, rescale: bool = True):
    """The tiled FlashAttention-2 forward loop of STAGE 3/4, for ONE head.

    Query blocks of ``Br`` rows on the outer loop; for each, key/value blocks
    of ``Bc`` rows stream through while each row carries its running max
    ``m``, running sum ``l`` and unnormalised output ``acc``.  When the max
    grows, ``l`` and ``acc`` are multiplied by ``exp(m_old - m_new)`` (taken
    as 0 while ``m_old`` is still -inf).  ``rescale=False`` drops that
    multiplication -- the bug STAGE 4 warns about -- and exists only so the
    tests can show it is caught.

    q, k, v: ``[N, D]``.  Returns ``(O [N, D], L [N])`` in float64.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    n = q.shape[0]
    o = np.zeros((n, v.shape[1]))
    lse = np.full(n, -np.inf)
    for i0 in range(0, n, Br):
        qi = q[i0:i0 + Br]
        rows = np.arange(i0, i0 + qi.shape[0])
        acc = np.zeros((qi.shape[0], v.shape[1]))
        m = np.full(qi.shape[0], -np.inf)
        l = np.zeros(qi.shape[0])
        for j0 in range(0, n, Bc):
            kj, vj = k[j0:j0 + Bc], v[j0:j0 + Bc]
            s = scale * (qi @ kj.T)
            if causal:
                cols = np.arange(j0, j0 + kj.shape[0])
                s = np.where(cols[None, :] > rows[:, None], -np.inf, s)
            m_new = np.maximum(m, s.max(axis=1))
            m_use = np.where(np.isfinite(m_new), m_new, 0.0)
            p = np.exp(s - m_use[:, None])
            if rescale:
                alpha = np.where(np.isfinite(m), np.exp(m - m_use), 0.0)
                l = alpha * l + p.sum(axis=1)
                acc = alpha[:, None] * acc + p @ vj
            else:
                l = l + p.sum(axis=1)
                acc = acc + p @ vj
            m = m_new
        live = l > 0
        o[i0:i0 + Br][live] = acc[live] / l[live, None]
        lse[i0:i0 + Br][live] = m[live] + np.log(l[live])
    return o, lse
