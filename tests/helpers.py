"""Shared helpers for the GPU parity tests: run the CUDA path through the C
ABI, compare with the oracle element by element, report the worst index.

Tolerances (max abs error against the float64 oracle on the same inputs):
  float32:                 O <= 1e-4, L <= 1e-5
  bf16 in, fp32 O:         O <= 1e-2, L <= 5e-3
  bf16 in, bf16 O:         O <= 1e-2 + half a bf16 ulp of |O_ref|, L <= 5e-3
"""

from __future__ import annotations

import numpy as np
import torch

import exact_attention_24_gb300 as fa

TOL = {
    fa.FA_F32: (1e-4, 1e-5),
    fa.FA_BF16_OUT_F32: (1e-2, 5e-3),
    fa.FA_BF16: (1e-2, 5e-3),
}


def half_ulp_bf16(x: np.ndarray) -> np.ndarray:
    """Half the spacing of bf16 numbers at |x| (8 significant bits)."""
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax > 0, 2.0 ** (e - 8), 0.0)


def out_dtype(code):
    return torch.bfloat16 if code == fa.FA_BF16 else torch.float32


def run_dense(q, k, v, causal, code, scale, stream=None):
    """q, k, v: CUDA tensors [B, H, N, D].  Returns (O, L) CUDA tensors."""
    B, H, N, D = q.shape
    O = torch.full((B, H, N, D), float("nan"), dtype=out_dtype(code), device=q.device)
    L = torch.full((B, H, N), float("nan"), dtype=torch.float32, device=q.device)
    st = fa.fa_fwd(q, k, v, O, L, B, H, N, D, scale, int(causal), code, stream)
    assert st == fa.FA_OK, fa.fa_status_string(st) + " / " + fa.fa_last_cuda_error()
    st = fa.fa_check_device_error(stream)
    assert st == fa.FA_OK, fa.fa_status_string(st)
    return O, L


def run_varlen(q, k, v, cu, max_seqlen, causal, code, scale, stream=None):
    total, H, D = q.shape
    O = torch.full((total, H, D), float("nan"), dtype=out_dtype(code), device=q.device)
    L = torch.full((H, total), float("nan"), dtype=torch.float32, device=q.device)
    cu_d = torch.as_tensor(np.asarray(cu), dtype=torch.int32).to(q.device)
    st = fa.fa_fwd_varlen(q, k, v, O, L, cu_d, len(cu) - 1, total, max_seqlen,
                          H, D, scale, int(causal), code, stream)
    assert st == fa.FA_OK, fa.fa_status_string(st)
    st = fa.fa_check_device_error(stream)
    assert st == fa.FA_OK, fa.fa_status_string(st)
    return O, L


def to_f64(x) -> np.ndarray:
    return x.detach().to("cpu", torch.float64).numpy()


def assert_close(got_o, got_l, ref_o, ref_l, code, what="", l_extra=0.0):
    """Element-by-element comparison; the message names the worst index.
    ``l_extra`` widens the L bound where the stored float32 value cannot
    resolve the base tolerance (|L| in the hundreds)."""
    tol_o, tol_l = TOL[code]
    tol_l = tol_l + l_extra
    got_o, got_l = np.asarray(got_o), np.asarray(got_l)
    assert got_o.shape == ref_o.shape and got_l.shape == ref_l.shape
    assert np.all(np.isfinite(got_o)), f"{what}: non-finite O at {np.argwhere(~np.isfinite(got_o))[:4]}"
    lfin = np.isfinite(ref_l)
    assert np.all(np.isfinite(got_l[lfin])), f"{what}: non-finite L where the oracle's is finite"
    assert np.all(got_l[~lfin] == -np.inf), f"{what}: L must be -inf for rows with no key"
    err_o = np.abs(got_o - ref_o)
    bound = tol_o + (half_ulp_bf16(ref_o) if code == fa.FA_BF16 else 0.0)
    excess = err_o - bound
    i = np.unravel_index(np.argmax(excess), excess.shape)
    assert excess[i] <= 0, (f"{what}: O err {err_o[i]:.3e} > {np.asarray(bound)[i] if np.ndim(bound) else bound:.3e} "
                            f"at {tuple(int(x) for x in i)} (got {got_o[i]:.6f}, ref {ref_o[i]:.6f})")
    err_l = np.abs(np.where(lfin, got_l - ref_l, 0.0))
    j = np.unravel_index(np.argmax(err_l), err_l.shape)
    assert err_l[j] <= tol_l, (f"{what}: L err {err_l[j]:.3e} > {tol_l:.1e} at "
                               f"{tuple(int(x) for x in j)} (got {got_l[j]:.6f}, ref {ref_l[j]:.6f})")
    return float(err_o.max()), float(err_l.max())


def sample_rows(n: int, count: int, seed: int, tile: int = 128) -> np.ndarray:
    """Rows to check at full size: the first and last rows, every tile
    boundary pair, and random rows, sorted and unique."""
    rng = np.random.default_rng(seed)
    fixed = {0, 1, n - 1, n - 2}
    for t in range(tile, n, tile):
        fixed.update({t - 1, t})
    fixed = sorted(x for x in fixed if 0 <= x < n)
    if len(fixed) > count // 2:
        fixed = list(rng.choice(fixed, count // 2, replace=False))
    rand = rng.integers(0, n, size=max(0, count - len(fixed)))
    return np.unique(np.concatenate([fixed, rand]).astype(np.int64))
