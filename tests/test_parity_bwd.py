"""GPU parity of the backward pass (fa_bwd through the C ABI) against the
float64 oracle on the same seeded inputs, element by element.

The kernel is given the oracle's O and L, stored in the library's types
(O in the input dtype, L float32), so these tests check the backward
kernels alone.  The expected gradients come from the oracle's own
definition on Q, K, V, dO.

Tolerance: the pages state none for gradients.  Two bounds, both enforced
where the full oracle is run:

* the forward bounds, applied relative to each gradient tensor's scale:
  max abs error <= tol * max(1, max |ref|), with tol = 1e-4 for float32 and
  1e-2 for bf16 inputs;
* per element, from the arithmetic: every gradient element is a sum of
  products, and rounding a factor of each term by a relative u moves it by
  at most u times the sum of the terms' magnitudes, M
  (oracle.attention_bwd_magnitudes).  With bf16 inputs P and dS enter the
  tensor-core contractions rounded to bf16 (2^-9 each) and D_i is computed
  from O stored in bf16 (2^-9 of sum |dO||O|): error <= 2^-7 M, four times
  that unit.  Float32 throughout: 2e-5 M.  Measured worst cases on GB300:
  3.5e-3 M (tensor cores, dV), 6e-4 M (bf16 on the FFMA kernels), 7.3e-7 M
  (float32).  Rows whose gradients are small against the tensor's largest
  are held to their own terms this way.

Half a bf16 ulp of |ref| is added when the gradient is stored as bf16.
"""

import numpy as np
import pytest
import torch

import exact_attention_24_gb300 as fa
from exact_attention_24_gb300 import build as fa_build
from exact_attention_24_gb300.workloads import Workload, make_inputs
from helpers import half_ulp_bf16, to_f64
from oracle import (attention_bwd_magnitudes, attention_bwd_ref, attention_bwd_ref_varlen,
                    attention_bwd_sampled, attention_ref, attention_ref_varlen)

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
GRAD_TOL = {fa.FA_F32: 1e-4, fa.FA_BF16_OUT_F32: 1e-2, fa.FA_BF16: 1e-2}
# per element, relative to the sum of the terms' magnitudes (see the module text)
GRAD_REL = {fa.FA_F32: 2e-5, fa.FA_BF16_OUT_F32: 2.0 ** -7, fa.FA_BF16: 2.0 ** -7}
BF16_CODES = (fa.FA_BF16_OUT_F32, fa.FA_BF16)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    fa_build.build()
    fa.load_library()
    yield
    fa.fa_set_options(fa.FA_KERNEL_AUTO, 0, 0)


@pytest.fixture(params=["auto", "simt"])
def kernel(request):
    code = fa.FA_KERNEL_AUTO if request.param == "auto" else fa.FA_KERNEL_SIMT
    assert fa.fa_set_options(code, 0, 0) == fa.FA_OK
    yield request.param
    fa.fa_set_options(fa.FA_KERNEL_AUTO, 0, 0)


def _bwd_inputs(B, H, N, D, dtype, causal, seed, qk_mult=1.0):
    """Seeded Q, K, V, dO (storage dtype) and the oracle's O, L for them."""
    w = Workload("bwd", B, H, N, D, dtype, causal, seed, qk_mult)
    q, k, v = make_inputs(w)
    do = make_inputs(Workload("dO", B, H, N, D, dtype, causal, seed + 50_000))[0]
    o, lse = attention_ref(q, k, v, w.scale, causal)
    return w, q, k, v, do, torch.from_numpy(o).to(q.dtype), torch.from_numpy(lse).float()


def run_bwd(q, k, v, o, do, lse, causal, code, scale):
    B, H, N, D = q.shape
    odt = torch.bfloat16 if code == fa.FA_BF16 else torch.float32
    grads = [torch.full((B, H, N, D), float("nan"), dtype=odt, device=q.device) for _ in range(3)]
    nbytes = fa.fa_bwd_workspace_size(B, H, N)
    ws = torch.full((max(nbytes, 16) // 4,), float("nan"), dtype=torch.float32, device=q.device)
    st = fa.fa_bwd(q, k, v, o, do, lse, *grads, B, H, N, D, scale, int(causal), code, ws, nbytes,
                   None)
    assert st == fa.FA_OK, fa.fa_status_string(st) + " / " + fa.fa_last_cuda_error()
    assert fa.fa_check_device_error(None) == fa.FA_OK
    return grads


def assert_grads(got, ref, code, what, mags=None):
    """Both bounds of the module text; the per-element one when the oracle's
    magnitudes `mags` (dQ, dK, dV) are given."""
    for idx, (name, g, r) in enumerate(zip(("dQ", "dK", "dV"), got, ref)):
        g = np.asarray(g)
        assert g.shape == r.shape, (what, name)
        assert np.all(np.isfinite(g)), f"{what}: non-finite {name}"
        ulp = half_ulp_bf16(r) if code == fa.FA_BF16 else 0.0
        bound = GRAD_TOL[code] * max(1.0, float(np.max(np.abs(r), initial=0.0))) + ulp
        excess = np.abs(g - r) - bound
        i = np.unravel_index(np.argmax(excess), excess.shape)
        assert excess[i] <= 0, (f"{what}: {name} err {abs(g[i] - r[i]):.3e} at "
                                f"{tuple(int(x) for x in i)} (got {g[i]:.6f}, ref {r[i]:.6f})")
        if mags is None:
            continue
        m = np.asarray(mags[idx])
        assert m.shape == r.shape, (what, name)
        # a floor of 1e-30 leaves exact zeros (masked rows) held to exactly zero error
        excess = np.abs(g - r) - (GRAD_REL[code] * m + ulp + 1e-30)
        i = np.unravel_index(np.argmax(excess), excess.shape)
        assert excess[i] <= 0, (f"{what}: {name} err {abs(g[i] - r[i]):.3e} > {GRAD_REL[code]:.1e} x "
                                f"M = {m[i]:.3e} at {tuple(int(x) for x in i)}")


SHAPES = [(1, 1, 1, 64), (1, 1, 3, 128), (1, 1, 127, 64), (1, 2, 129, 128), (1, 1, 257, 64),
          (2, 2, 300, 128), (1, 1, 700, 64), (1, 3, 1000, 128)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_small_bf16(kernel, shape, causal):
    B, H, N, D = shape
    w, q, k, v, do, o, lse = _bwd_inputs(B, H, N, D, "bf16", causal, seed=3 * N + D)
    ref = attention_bwd_ref(q, k, v, do, w.scale, causal)[:3]
    mags = attention_bwd_magnitudes(q, k, v, do, w.scale, causal)
    dev = [x.to(DEV) for x in (q, k, v, o, do, lse)]
    for code in BF16_CODES:
        got = run_bwd(*dev, causal, code, w.scale)
        assert_grads([to_f64(x) for x in got], ref, code, f"{kernel} {shape} c={causal} dt={code}", mags)


@pytest.mark.parametrize("shape", [(1, 1, 1, 64), (1, 1, 5, 128), (2, 2, 300, 64),
                                   (1, 2, 513, 128)], ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_small_f32(kernel, shape, causal):
    B, H, N, D = shape
    w, q, k, v, do, o, lse = _bwd_inputs(B, H, N, D, "f32", causal, seed=5 * N + D)
    ref = attention_bwd_ref(q, k, v, do, w.scale, causal)[:3]
    mags = attention_bwd_magnitudes(q, k, v, do, w.scale, causal)
    got = run_bwd(*[x.to(DEV) for x in (q, k, v, o, do, lse)], causal, fa.FA_F32, w.scale)
    assert_grads([to_f64(x) for x in got], ref, fa.FA_F32, f"{kernel} {shape} c={causal}", mags)


def test_bwd_sharp_softmax(kernel):
    """Q, K doubled (the sharp-softmax workload's recipe): P is nearly
    one-hot, large entries of dS."""
    w, q, k, v, do, o, lse = _bwd_inputs(1, 2, 640, 64, "bf16", True, seed=77, qk_mult=2.0)
    ref = attention_bwd_ref(q, k, v, do, w.scale, True)[:3]
    mags = attention_bwd_magnitudes(q, k, v, do, w.scale, True)
    got = run_bwd(*[x.to(DEV) for x in (q, k, v, o, do, lse)], True, fa.FA_BF16_OUT_F32, w.scale)
    assert_grads([to_f64(x) for x in got], ref, fa.FA_BF16_OUT_F32, f"{kernel} sharp", mags)


def test_bwd_deterministic(kernel):
    """No atomics: two calls give bitwise the same gradients."""
    w, q, k, v, do, o, lse = _bwd_inputs(2, 2, 1000, 128, "bf16", True, seed=3)
    dev = [x.to(DEV) for x in (q, k, v, o, do, lse)]
    a = run_bwd(*dev, True, fa.FA_BF16, w.scale)
    b = run_bwd(*dev, True, fa.FA_BF16, w.scale)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_bwd_from_own_forward(kernel):
    """The usual pairing: L and O from fa_fwd itself feed fa_bwd."""
    w, q, k, v, do, _, _ = _bwd_inputs(1, 2, 900, 128, "bf16", True, seed=11)
    qd, kd, vd, dod = (x.to(DEV) for x in (q, k, v, do))
    O, L = fa.attention(qd, kd, vd, causal=True, scale=w.scale)
    got = run_bwd(qd, kd, vd, O, dod, L, True, fa.FA_BF16_OUT_F32, w.scale)
    ref = attention_bwd_ref(q, k, v, do, w.scale, True)[:3]
    assert_grads([to_f64(x) for x in got], ref, fa.FA_BF16_OUT_F32, f"{kernel} own forward")


@pytest.mark.parametrize("shape", [(2, 16, 4096, 128, True), (4, 8, 1024, 64, False)],
                         ids=lambda s: "x".join(map(str, s)))
def test_bwd_full_size_sampled(shape):
    """Benchmark-sized problems (the C3 and C2 shapes) in the default kernel
    selection, checked on sampled rows of dQ and keys of dK, dV."""
    B, H, N, D, causal = shape
    w, q, k, v, do, o, lse = _bwd_inputs(B, H, N, D, "bf16", causal, seed=123)
    got = run_bwd(*[x.to(DEV) for x in (q, k, v, o, do, lse)], causal, fa.FA_BF16, w.scale)
    rng = np.random.default_rng(5)
    idx = np.unique(np.concatenate([[0, 1, 127, 128, N - 1], rng.integers(0, N, 20)]))
    for b, h in [(0, 0), (B - 1, H - 1)]:
        ref = attention_bwd_sampled(q[b, h], k[b, h], v[b, h], do[b, h], w.scale, causal, idx, idx)
        mine = [to_f64(got[0][b, h, idx]), to_f64(got[1][b, h, idx]), to_f64(got[2][b, h, idx])]
        assert_grads(mine, ref, fa.FA_BF16, f"full {shape} b={b} h={h}")


# ---------------------------------------------------------------- varlen --
def _varlen_bwd_inputs(lengths, H, D, causal, seed):
    w = Workload("vbwd", 0, H, 0, D, "bf16", causal, seed, lengths=tuple(lengths))
    q, k, v = make_inputs(w)
    do = make_inputs(Workload("vdO", 0, H, 0, D, "bf16", causal, seed + 50_000,
                              lengths=tuple(lengths)))[0]
    o, lse = attention_ref_varlen(q, k, v, w.cu_seqlens, w.scale, causal)
    return w, q, k, v, do, torch.from_numpy(o).to(q.dtype), torch.from_numpy(lse).float()


def run_bwd_varlen(w, q, k, v, o, do, lse, code):
    odt = torch.bfloat16 if code == fa.FA_BF16 else torch.float32
    grads = [torch.full(q.shape, float("nan"), dtype=odt, device=q.device) for _ in range(3)]
    nbytes = fa.fa_bwd_varlen_workspace_size(w.total, w.H)
    ws = torch.full((max(nbytes, 16) // 4,), float("nan"), dtype=torch.float32, device=q.device)
    cu = torch.as_tensor(w.cu_seqlens, dtype=torch.int32, device=q.device)
    st = fa.fa_bwd_varlen(q, k, v, o, do, lse, *grads, cu, len(w.lengths), w.total, w.max_seqlen,
                          w.H, w.D, w.scale, int(w.causal), code, ws, nbytes, None)
    assert st == fa.FA_OK, fa.fa_status_string(st) + " / " + fa.fa_last_cuda_error()
    assert fa.fa_check_device_error(None) == fa.FA_OK
    return grads


def _varlen_magnitudes(q, k, v, do, cu, scale, causal):
    """attention_bwd_magnitudes of every (sequence, head) of a packed batch,
    in its [total, H, D] layout."""
    out = [np.zeros(tuple(x.shape), dtype=np.float64) for x in (q, k, v)]
    for s in range(len(cu) - 1):
        a, b = int(cu[s]), int(cu[s + 1])
        for h in range(q.shape[1]):
            ms = attention_bwd_magnitudes(q[a:b, h], k[a:b, h], v[a:b, h], do[a:b, h], scale, causal)
            for dst, m in zip(out, ms):
                dst[a:b, h] = m
    return out


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_varlen_small(kernel, D, causal):
    lengths = [0, 1, 127, 128, 129, 300, 5, 0, 260]
    w, q, k, v, do, o, lse = _varlen_bwd_inputs(lengths, 2, D, causal, seed=D + int(causal))
    ref = attention_bwd_ref_varlen(q, k, v, do, w.cu_seqlens, w.scale, causal)[:3]
    mags = _varlen_magnitudes(q, k, v, do, w.cu_seqlens, w.scale, causal)
    dev = [x.to(DEV) for x in (q, k, v, o, do, lse)]
    for code in BF16_CODES:
        got = run_bwd_varlen(w, *dev, code)
        assert_grads([to_f64(x) for x in got], ref, code, f"{kernel} varlen D={D} c={causal} dt={code}",
                     mags)


def test_bwd_varlen_f32(kernel):
    lengths = [3, 0, 200, 64]
    w = Workload("vbwd32", 0, 3, 0, 64, "f32", True, 9, lengths=tuple(lengths))
    q, k, v = make_inputs(w)
    do = make_inputs(Workload("vdO32", 0, 3, 0, 64, "f32", True, 99, lengths=tuple(lengths)))[0]
    o, lse = attention_ref_varlen(q, k, v, w.cu_seqlens, w.scale, True)
    o, lse = torch.from_numpy(o).float(), torch.from_numpy(lse).float()
    ref = attention_bwd_ref_varlen(q, k, v, do, w.cu_seqlens, w.scale, True)[:3]
    got = run_bwd_varlen(w, *[x.to(DEV) for x in (q, k, v, o, do, lse)], fa.FA_F32)
    assert_grads([to_f64(x) for x in got], ref, fa.FA_F32, f"{kernel} varlen f32")


def test_bwd_varlen_full_size_sampled():
    """The 16-sequence packed workload (lengths uniform in [128, 4096]) in the
    default kernel selection, on sampled rows and keys of three sequences."""
    from exact_attention_24_gb300.workloads import C5
    w, q, k, v, do, o, lse = _varlen_bwd_inputs(C5.lengths, C5.H, C5.D, True, seed=C5.seed)
    got = run_bwd_varlen(w, *[x.to(DEV) for x in (q, k, v, o, do, lse)], fa.FA_BF16)
    cu = w.cu_seqlens
    rng = np.random.default_rng(7)
    for s, h in [(0, 0), (7, 9), (15, 15)]:
        a, b = int(cu[s]), int(cu[s + 1])
        n = b - a
        idx = np.unique(np.concatenate([[0, n - 1], rng.integers(0, n, 12)]))
        ref = attention_bwd_sampled(q[a:b, h], k[a:b, h], v[a:b, h], do[a:b, h], w.scale, True, idx, idx)
        mine = [to_f64(got[0][a + idx, h]), to_f64(got[1][a + idx, h]), to_f64(got[2][a + idx, h])]
        assert_grads(mine, ref, fa.FA_BF16, f"varlen full s={s} h={h}")


# ------------------------------------------------------------ local band --
def run_bwd_window(q, k, v, o, do, lse, wl, wr, code, scale):
    B, H, N, D = q.shape
    odt = torch.bfloat16 if code == fa.FA_BF16 else torch.float32
    grads = [torch.full((B, H, N, D), float("nan"), dtype=odt, device=q.device) for _ in range(3)]
    nbytes = fa.fa_bwd_workspace_size(B, H, N)
    ws = torch.full((max(nbytes, 16) // 4,), float("nan"), dtype=torch.float32, device=q.device)
    st = fa.fa_bwd_window(q, k, v, o, do, lse, *grads, B, H, N, D, scale, wl, wr, code, ws, nbytes,
                          None)
    assert st == fa.FA_OK, fa.fa_status_string(st) + " / " + fa.fa_last_cuda_error()
    assert fa.fa_check_device_error(None) == fa.FA_OK
    return grads


def _window_inputs(B, H, N, D, window, seed):
    w = Workload("wbwd", B, H, N, D, "bf16", False, seed)
    q, k, v = make_inputs(w)
    do = make_inputs(Workload("wdO", B, H, N, D, "bf16", False, seed + 50_000))[0]
    o, lse = attention_ref(q, k, v, w.scale, False, window=window)
    return w, q, k, v, do, torch.from_numpy(o).to(q.dtype), torch.from_numpy(lse).float()


BWD_WINDOWS = [(1, 2, 1000, 64, 64, 64), (1, 1, 777, 128, 100, 30), (2, 1, 600, 128, 0, 0),
               (1, 1, 2048, 128, 300, -1), (1, 2, 1500, 64, 5, 200), (1, 1, 513, 64, 127, 129),
               (1, 1, 1024, 128, 256, 0), (1, 1, 300, 128, 1000, 1000)]


@pytest.mark.parametrize("case", BWD_WINDOWS, ids=lambda c: "x".join(map(str, c)))
def test_bwd_window_matches_oracle(kernel, case):
    B, H, N, D, wl, wr = case
    w, q, k, v, do, o, lse = _window_inputs(B, H, N, D, (wl, wr), seed=N + wl + 7)
    ref = attention_bwd_ref(q, k, v, do, w.scale, False, window=(wl, wr))[:3]
    mags = attention_bwd_magnitudes(q, k, v, do, w.scale, False, window=(wl, wr))
    dev = [x.to(DEV) for x in (q, k, v, o, do, lse)]
    for code in BF16_CODES:
        got = run_bwd_window(*dev, wl, wr, code, w.scale)
        assert_grads([to_f64(x) for x in got], ref, code, f"{kernel} band {case} dt={code}", mags)


def test_bwd_window_special_cases_are_the_plain_paths(kernel):
    """(-1, 0) is the causal backward and (-1, -1) the full one, bit for bit."""
    for causal, window in ((True, (-1, 0)), (False, (-1, -1))):
        w, q, k, v, do, o, lse = _bwd_inputs(1, 2, 900, 128, "bf16", causal, seed=17)
        dev = [x.to(DEV) for x in (q, k, v, o, do, lse)]
        a = run_bwd(*dev, causal, fa.FA_BF16, w.scale)
        b = run_bwd_window(*dev, window[0], window[1], fa.FA_BF16, w.scale)
        for x, y in zip(a, b):
            assert torch.equal(x, y)


def test_bwd_window_sliding_full_size_sampled():
    """A causal 4096-key sliding window over 32K tokens (the sliding-window
    forward workload's shape, one head shown), sampled rows and keys."""
    B, H, N, D, wl, wr = 1, 2, 32768, 128, 4096, 0
    w = Workload("wbig", B, H, N, D, "bf16", False, 3)
    q, k, v = make_inputs(w)
    do = make_inputs(Workload("wbigdO", B, H, N, D, "bf16", False, 50_003))[0]
    qd, kd, vd, dod = (x.to(DEV) for x in (q, k, v, do))
    O = torch.empty_like(qd)
    L = torch.empty((B, H, N), dtype=torch.float32, device=DEV)
    assert fa.fa_fwd_window(qd, kd, vd, O, L, B, H, N, D, w.scale, wl, wr, fa.FA_BF16, None) == fa.FA_OK
    got = run_bwd_window(qd, kd, vd, O, dod, L, wl, wr, fa.FA_BF16, w.scale)
    rng = np.random.default_rng(9)
    idx = np.unique(np.concatenate([[0, 4095, 4096, N - 1], rng.integers(0, N, 12)]))
    for h in range(H):
        ref = attention_bwd_sampled(q[0, h], k[0, h], v[0, h], do[0, h], w.scale, False, idx, idx,
                                    window=(wl, wr))
        mine = [to_f64(got[0][0, h, idx]), to_f64(got[1][0, h, idx]), to_f64(got[2][0, h, idx])]
        assert_grads(mine, ref, fa.FA_BF16, f"sliding full size h={h}")
