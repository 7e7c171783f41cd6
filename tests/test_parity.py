"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle on
the same seeded inputs, element by element.

Small problems are compared in full (several tiles plus a ragged tail); the
five benchmark workloads are compared at full size on sampled rows that the
oracle computes one by one, in the launch configuration bench.py times
(default options: tensor-core kernel for bf16, one CTA per SM).
Every test runs under both kernel selections: ``auto`` (the tensor-core
kernel for bf16) and ``simt`` (the FFMA kernel for every dtype).
"""

import math

import numpy as np
import pytest
import torch

import exact_attention_24_gb300 as fa
from exact_attention_24_gb300 import build as fa_build
from exact_attention_24_gb300.workloads import (C1, C2, C3, C4, C5, WORKLOADS, Workload,
                                                default_scale, make_inputs)
from helpers import (assert_close, run_dense, run_varlen, sample_rows, to_f64)
from oracle import attention_ref, attention_ref_varlen, attention_rows

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
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


def _dense_case(B, H, N, D, dtype, causal, seed, qk_mult=1.0):
    w = Workload("case", B, H, N, D, dtype, causal, seed, qk_mult)
    q, k, v = make_inputs(w)
    return w, q, k, v


# ---------------------------------------------------------------- small --
SMALL_SHAPES = [
    (1, 1, 1, 64), (1, 2, 2, 128), (1, 1, 3, 64), (1, 1, 127, 128),
    (1, 1, 129, 64), (1, 1, 255, 128), (1, 2, 256, 64), (1, 1, 257, 128),
    (2, 3, 1000, 64), (2, 3, 1000, 128), (1, 2, 640, 128),
]


@pytest.mark.parametrize("shape", SMALL_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("causal", [False, True])
def test_small_dense_bf16(kernel, shape, causal):
    B, H, N, D = shape
    w, q, k, v = _dense_case(B, H, N, D, "bf16", causal, seed=N + D)
    ref_o, ref_l = attention_ref(q, k, v, w.scale, causal)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    for code in BF16_CODES:
        O, L = run_dense(qd, kd, vd, causal, code, w.scale)
        assert_close(to_f64(O), to_f64(L), ref_o, ref_l, code, f"{kernel} {shape} c={causal} dt={code}")


@pytest.mark.parametrize("shape", [(1, 1, 1, 64), (1, 1, 3, 128), (2, 2, 300, 64),
                                   (1, 2, 513, 128)], ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("causal", [False, True])
def test_small_dense_f32(kernel, shape, causal):
    B, H, N, D = shape
    w, q, k, v = _dense_case(B, H, N, D, "f32", causal, seed=7 * N + D)
    ref_o, ref_l = attention_ref(q, k, v, w.scale, causal)
    O, L = run_dense(q.to(DEV), k.to(DEV), v.to(DEV), causal, fa.FA_F32, w.scale)
    assert_close(to_f64(O), to_f64(L), ref_o, ref_l, fa.FA_F32, f"{shape} c={causal}")


@pytest.mark.parametrize("lengths", [(1, 129, 0, 300), (128, 256, 5), (0, 0, 700),
                                     (2, 3, 1, 130, 257, 77)], ids=str)
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_small_varlen(kernel, lengths, D, causal):
    w = Workload("vl", 0, 3, 0, D, "bf16", causal, seed=sum(lengths) + D,
                 lengths=tuple(lengths))
    q, k, v = make_inputs(w)
    cu = w.cu_seqlens
    ref_o, ref_l = attention_ref_varlen(q, k, v, cu, w.scale, causal)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    for code in BF16_CODES:
        O, L = run_varlen(qd, kd, vd, cu, w.max_seqlen, causal, code, w.scale)
        assert_close(to_f64(O), to_f64(L), ref_o, ref_l, code, f"{kernel} {lengths} c={causal}")


# ------------------------------------------------------- full workloads --
def test_c1_full(kernel):
    q, k, v = make_inputs(C1)
    ref_o, ref_l = attention_ref(q, k, v, C1.scale, C1.causal)
    O, L = run_dense(q.to(DEV), k.to(DEV), v.to(DEV), C1.causal, fa.FA_F32, C1.scale)
    assert_close(to_f64(O), to_f64(L), ref_o, ref_l, fa.FA_F32, "C1")


def test_c2_full(kernel):
    q, k, v = make_inputs(C2)
    ref_o, ref_l = attention_ref(q, k, v, C2.scale, C2.causal)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    for code in BF16_CODES:
        O, L = run_dense(qd, kd, vd, C2.causal, code, C2.scale)
        assert_close(to_f64(O), to_f64(L), ref_o, ref_l, code, f"C2 dt={code}")


@pytest.mark.parametrize("w", [C3, C4], ids=lambda w: w.name)
def test_full_size_sampled_rows(kernel, w):
    q, k, v = make_inputs(w)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    outs = {code: run_dense(qd, kd, vd, w.causal, code, w.scale) for code in BF16_CODES}
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    for idx, (b, h) in enumerate(heads):
        rows = sample_rows(w.N, 24, seed=idx)
        ref_o, ref_l = attention_rows(q[b, h], k[b, h], v[b, h], w.scale, w.causal, rows)
        for code, (O, L) in outs.items():
            assert_close(to_f64(O[b, h, rows]), to_f64(L[b, h, rows]), ref_o, ref_l,
                         code, f"{w.name} b={b} h={h} dt={code}")


def test_c5_varlen_sampled_rows(kernel):
    w = C5
    q, k, v = make_inputs(w)
    cu = w.cu_seqlens
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    outs = {code: run_varlen(qd, kd, vd, cu, w.max_seqlen, w.causal, code, w.scale)
            for code in BF16_CODES}
    # every (sequence, head) pair: the compact order walks heads in groups
    # sized for L2, so each position within a group is covered
    for s in range(len(w.lengths)):
        a, n = int(cu[s]), int(w.lengths[s])
        for h in range(w.H):
            rows = sample_rows(n, 12, seed=100 * s + h)
            ref_o, ref_l = attention_rows(q[a:a + n, h], k[a:a + n, h], v[a:a + n, h],
                                          w.scale, w.causal, rows)
            for code, (O, L) in outs.items():
                assert_close(to_f64(O[a + rows, h]), to_f64(L[h, a + rows]), ref_o, ref_l,
                             code, f"C5 seq={s} h={h} dt={code}")


# ------------------------------------------------ closed forms on the GPU --
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", [64, 128])
def test_zero_query_closed_form(kernel, causal, D):
    """Q = 0: O = mean of the attended V rows, L = ln(#attended keys)."""
    N = 300
    g = torch.Generator().manual_seed(5)
    k = torch.randn(1, 2, N, D, generator=g).to(torch.bfloat16)
    v = torch.randn(1, 2, N, D, generator=g).to(torch.bfloat16)
    q = torch.zeros_like(k)
    O, L = run_dense(q.to(DEV), k.to(DEV), v.to(DEV), causal, fa.FA_BF16_OUT_F32,
                     default_scale(D))
    vf = v.double().numpy()
    cnt = np.arange(1, N + 1) if causal else np.full(N, N)
    exp_o = (np.cumsum(vf, axis=2) / np.arange(1, N + 1)[:, None]) if causal else \
        np.broadcast_to(vf.mean(axis=2, keepdims=True), vf.shape)
    exp_l = np.broadcast_to(np.log(cnt), (1, 2, N))
    assert_close(to_f64(O), to_f64(L), exp_o, exp_l, fa.FA_BF16_OUT_F32, "Q=0")


def test_overflow_scores_f32(kernel):
    """The page's DEMO 9 scores (800, 810, 805, 790) must give finite, exact
    softmax weights on the GPU too (float32 path)."""
    scores = [800.0, 810.0, 805.0, 790.0]
    D = 64
    q = torch.zeros(1, 1, 4, D)
    q[..., 0] = 1.0
    k = torch.zeros(1, 1, 4, D)
    k[0, 0, :, 0] = torch.tensor(scores)
    v = torch.zeros(1, 1, 4, D)
    v[0, 0, :, :4] = torch.eye(4)
    O, L = run_dense(q.to(DEV), k.to(DEV), v.to(DEV), False, fa.FA_F32, 1.0)
    z = sum(math.exp(s - 810.0) for s in scores)
    w = np.array([math.exp(s - 810.0) / z for s in scores])
    exp_o = np.zeros((1, 1, 4, D))
    exp_o[0, 0, :, :4] = w
    exp_l = np.full((1, 1, 4), 810.0 + math.log(z))
    # |L| ~ 810: one float32 ulp there is 2^-14 = 6.1e-5, so the 1e-5 bound
    # (set for |L| of order 1) is widened by one ulp of the stored value.
    assert_close(to_f64(O), to_f64(L), exp_o, exp_l, fa.FA_F32, "DEMO 9",
                 l_extra=float(np.spacing(np.float32(810.0))))


def test_overflow_scores_bf16(kernel):
    """Large scores in bf16 (exactly representable): 800, 808, 804, 792."""
    scores = [800.0, 808.0, 804.0, 792.0]
    D = 128
    q = torch.zeros(1, 1, 4, D, dtype=torch.bfloat16)
    q[..., 0] = 1.0
    k = torch.zeros(1, 1, 4, D, dtype=torch.bfloat16)
    k[0, 0, :, 0] = torch.tensor(scores, dtype=torch.bfloat16)
    v = torch.zeros(1, 1, 4, D, dtype=torch.bfloat16)
    v[0, 0, :, :4] = torch.eye(4, dtype=torch.bfloat16)
    O, L = run_dense(q.to(DEV), k.to(DEV), v.to(DEV), False, fa.FA_BF16_OUT_F32, 1.0)
    z = sum(math.exp(s - 808.0) for s in scores)
    exp_o = np.zeros((1, 1, 4, D))
    exp_o[0, 0, :, :4] = [math.exp(s - 808.0) / z for s in scores]
    exp_l = np.full((1, 1, 4), 808.0 + math.log(z))
    assert_close(to_f64(O), to_f64(L), exp_o, exp_l, fa.FA_BF16_OUT_F32, "large scores",
                 l_extra=float(np.spacing(np.float32(808.0))))


# ---------------------------------------------------- hygiene / safety --
def test_outputs_written_only_in_bounds(kernel):
    """Canary regions around O and L must stay untouched."""
    B, H, N, D = 1, 2, 333, 128
    w, q, k, v = _dense_case(B, H, N, D, "bf16", True, seed=3)
    pad = 4096
    for code in BF16_CODES:
        odt = torch.bfloat16 if code == fa.FA_BF16 else torch.float32
        obuf = torch.full((2 * pad + B * H * N * D,), float("nan"), dtype=odt, device=DEV)
        lbuf = torch.full((2 * pad + B * H * N,), float("nan"), dtype=torch.float32, device=DEV)
        o_view = obuf[pad:pad + B * H * N * D]
        l_view = lbuf[pad:pad + B * H * N]
        st = fa.fa_fwd(q.to(DEV), k.to(DEV), v.to(DEV), o_view, l_view, B, H, N, D,
                       w.scale, 1, code, None)
        assert st == fa.FA_OK
        assert fa.fa_check_device_error(None) == fa.FA_OK
        for buf in (obuf, lbuf):
            assert torch.isnan(buf[:pad].float()).all() and torch.isnan(buf[-pad:].float()).all()
        assert torch.isfinite(o_view.float()).all() and torch.isfinite(l_view).all()


def test_deterministic(kernel):
    w, q, k, v = _dense_case(2, 4, 1100, 128, "bf16", True, seed=11)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    O1, L1 = run_dense(qd, kd, vd, True, fa.FA_BF16, w.scale)
    O2, L2 = run_dense(qd, kd, vd, True, fa.FA_BF16, w.scale)
    assert torch.equal(O1, O2) and torch.equal(L1, L2)


def test_grid_size_does_not_change_results():
    """The persistent tensor-core kernel gives bitwise the same result for any
    grid size: each output row is produced by one CTA in a fixed order."""
    w, q, k, v = _dense_case(1, 5, 1500, 128, "bf16", True, seed=12)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    res = []
    for grid in (0, 1, 7, 300):
        fa.fa_set_options(fa.FA_KERNEL_AUTO, grid, 0)
        res.append(run_dense(qd, kd, vd, True, fa.FA_BF16, w.scale))
    fa.fa_set_options(fa.FA_KERNEL_AUTO, 0, 0)
    for O, L in res[1:]:
        assert torch.equal(O, res[0][0]) and torch.equal(L, res[0][1])


@pytest.mark.parametrize("code", [fa.FA_F32, fa.FA_BF16])
def test_ffma_row_grouping_does_not_change_results(code):
    """The FFMA kernel gives small grids one row per warp (8-row CTAs) and
    larger ones 8 rows per warp (64-row CTAs); each row's arithmetic is the
    same, so one head computed alone (4 blocks of 64 rows: under-filled) and
    as head 0 of a 64-head batch (256 blocks) agree bitwise."""
    dt = "f32" if code == fa.FA_F32 else "bf16"
    w, q, k, v = _dense_case(1, 64, 256, 64, dt, True, seed=13)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    assert fa.fa_set_options(fa.FA_KERNEL_SIMT, 0, 0) == fa.FA_OK
    try:
        O_all, L_all = run_dense(qd, kd, vd, True, code, w.scale)
        O_one, L_one = run_dense(*(x[:, :1].contiguous() for x in (qd, kd, vd)), True, code, w.scale)
    finally:
        fa.fa_set_options(fa.FA_KERNEL_AUTO, 0, 0)
    assert torch.equal(O_one[:, 0], O_all[:, 0]) and torch.equal(L_one[:, 0], L_all[:, 0])
    ref_o, ref_l = attention_ref(q[0, 0], k[0, 0], v[0, 0], w.scale, True)
    assert_close(to_f64(O_one[0, 0]), to_f64(L_one[0, 0]), ref_o, ref_l, code, "FFMA one row a warp")


def test_invalid_cu_seqlens_reported_on_device(kernel):
    """A decreasing cu_seqlens is caught on the device: the sequence is
    skipped and fa_check_device_error reports FA_ERR_INVALID_ARG."""
    H, D = 2, 64
    total = 300
    q = torch.randn(total, H, D, device=DEV).to(torch.bfloat16)
    O = torch.zeros(total, H, D, device=DEV, dtype=torch.bfloat16)
    L = torch.zeros(H, total, device=DEV)
    cu = torch.tensor([0, 200, 100, 300], dtype=torch.int32, device=DEV)
    st = fa.fa_fwd_varlen(q, q, q, O, L, cu, 3, total, 300, H, D, 0.125, 1, fa.FA_BF16, None)
    assert st == fa.FA_OK
    assert fa.fa_check_device_error(None) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_check_device_error(None) == fa.FA_OK  # cleared
    # the library is still usable
    run_varlen(q, q, q, np.array([0, 100, 300]), 200, True, fa.FA_BF16, 0.125)


def test_watchdog_timeout_reports_and_recovers():
    """A wait that nothing satisfies runs out after its limit, is reported as
    FA_ERR_DEVICE_TIMEOUT, and leaves the context usable."""
    assert fa.fa_watchdog_selftest(50_000_000, None) == fa.FA_OK
    assert fa.fa_check_device_error(None) == fa.FA_ERR_DEVICE_TIMEOUT
    assert fa.fa_check_device_error(None) == fa.FA_OK
    w, q, k, v = _dense_case(1, 1, 200, 64, "bf16", True, seed=1)
    O, L = run_dense(q.to(DEV), k.to(DEV), v.to(DEV), True, fa.FA_BF16_OUT_F32, w.scale)
    ref_o, ref_l = attention_ref(q, k, v, w.scale, True)
    assert_close(to_f64(O), to_f64(L), ref_o, ref_l, fa.FA_BF16_OUT_F32, "after watchdog")


# ------------------------------------------------------------ split keys --
def run_splitkv(q, k, v, causal, code, scale, splits):
    B, H, N, D = q.shape
    O = torch.full((B, H, N, D), float("nan"), dtype=torch.bfloat16 if code == fa.FA_BF16 else torch.float32,
                   device=q.device)
    L = torch.full((B, H, N), float("nan"), dtype=torch.float32, device=q.device)
    nbytes = fa.fa_fwd_splitkv_workspace_size(B, H, N, D, splits)
    ws = torch.full((max(nbytes, 16) // 4,), float("nan"), dtype=torch.float32, device=q.device)
    st = fa.fa_fwd_splitkv(q, k, v, O, L, B, H, N, D, scale, int(causal), code, splits, ws, nbytes, None)
    assert st == fa.FA_OK, fa.fa_status_string(st) + " / " + fa.fa_last_cuda_error()
    assert fa.fa_check_device_error(None) == fa.FA_OK
    return O, L


@pytest.mark.parametrize("case", [(1, 1, 4096, 128, True, 8), (1, 2, 3000, 64, False, 3),
                                  (2, 1, 1000, 128, True, 0), (1, 1, 300, 64, True, 5),
                                  (1, 3, 777, 128, False, 2), (1, 1, 2048, 64, True, 16)],
                         ids=lambda c: "x".join(map(str, c)))
def test_splitkv_matches_oracle(case):
    B, H, N, D, causal, splits = case
    w, q, k, v = _dense_case(B, H, N, D, "bf16", causal, seed=N + splits)
    ref_o, ref_l = attention_ref(q, k, v, w.scale, causal)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    for code in BF16_CODES:
        O, L = run_splitkv(qd, kd, vd, causal, code, w.scale, splits)
        assert_close(to_f64(O), to_f64(L), ref_o, ref_l, code, f"split {case} dt={code}")


def test_splitkv_small_grid_runs_consecutive_items():
    """With a small persistent grid each CTA runs many split items in a row,
    among them items whose first query tile has no keys in its range (the
    last of 16 key ranges of a short causal block) followed by items whose
    first tile does.  Results match the oracle and do not depend on the grid."""
    w, q, k, v = _dense_case(1, 2, 2048, 64, "bf16", True, seed=31)
    ref_o, ref_l = attention_ref(q, k, v, w.scale, True)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    res = []
    try:
        for grid in (1, 3, 0):
            fa.fa_set_options(fa.FA_KERNEL_AUTO, grid, 0)
            res.append(run_splitkv(qd, kd, vd, True, fa.FA_BF16_OUT_F32, w.scale, 16))
    finally:
        fa.fa_set_options(fa.FA_KERNEL_AUTO, 0, 0)
    for O, L in res:
        assert_close(to_f64(O), to_f64(L), ref_o, ref_l, fa.FA_BF16_OUT_F32, "split, small grid")
        assert torch.equal(O, res[-1][0]) and torch.equal(L, res[-1][1])


def test_splitkv_one_split_is_the_dense_path():
    w, q, k, v = _dense_case(1, 2, 1500, 128, "bf16", True, seed=9)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    O1, L1 = run_splitkv(qd, kd, vd, True, fa.FA_BF16, w.scale, 1)
    O2, L2 = run_dense(qd, kd, vd, True, fa.FA_BF16, w.scale)
    assert torch.equal(O1, O2) and torch.equal(L1, L2)


def test_splitkv_merge_agrees_with_oracle_merge():
    """The GPU merge of the GPU's own partials against the oracle's merge of
    the oracle's partials over the same key ranges (C4-like sharp softmax)."""
    from oracle import merge_partials
    w, q, k, v = _dense_case(1, 1, 2048, 64, "bf16", True, seed=4, qk_mult=2.0)
    O, L = run_splitkv(q.to(DEV), k.to(DEV), v.to(DEV), True, fa.FA_BF16_OUT_F32, w.scale, 4)
    rows = sample_rows(2048, 64, seed=3)
    ref_o, ref_l = attention_rows(q[0, 0], k[0, 0], v[0, 0], w.scale, True, rows)
    assert_close(to_f64(O[0, 0, rows]), to_f64(L[0, 0, rows]), ref_o, ref_l, fa.FA_BF16_OUT_F32, "merge")
    # the oracle's own split-and-merge over 128-key-aligned ranges agrees too
    cuts = [0, 512, 1024, 1536, 2048]
    parts = [attention_rows(q[0, 0], k[0, 0], v[0, 0], w.scale, True, rows, a, b)
             for a, b in zip(cuts[:-1], cuts[1:])]
    mo, ml = merge_partials(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
    assert np.max(np.abs(mo - ref_o)) < 1e-12 and np.max(np.abs(ml - ref_l)) < 1e-12


# ------------------------------------------------------------ local band --
def run_window(q, k, v, wl, wr, code, scale):
    B, H, N, D = q.shape
    O = torch.full((B, H, N, D), float("nan"), dtype=torch.bfloat16 if code == fa.FA_BF16 else torch.float32,
                   device=q.device)
    L = torch.full((B, H, N), float("nan"), dtype=torch.float32, device=q.device)
    st = fa.fa_fwd_window(q, k, v, O, L, B, H, N, D, scale, wl, wr, code, None)
    assert st == fa.FA_OK, fa.fa_status_string(st) + " / " + fa.fa_last_cuda_error()
    assert fa.fa_check_device_error(None) == fa.FA_OK
    return O, L


WINDOW_CASES = [(1, 2, 1000, 64, 64, 64), (1, 1, 777, 128, 100, 30), (2, 1, 600, 128, 0, 0),
                (1, 1, 2048, 128, 300, -1), (1, 2, 1500, 64, 5, 200), (1, 1, 513, 64, 127, 129),
                (1, 1, 1024, 128, 256, 0), (1, 1, 300, 128, 1000, 1000)]


@pytest.mark.parametrize("case", WINDOW_CASES, ids=lambda c: "x".join(map(str, c)))
def test_window_matches_oracle(kernel, case):
    B, H, N, D, wl, wr = case
    w, q, k, v = _dense_case(B, H, N, D, "bf16", False, seed=N + wl)
    ref_o, ref_l = attention_ref(q, k, v, w.scale, False, window=(wl, wr))
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    for code in BF16_CODES:
        O, L = run_window(qd, kd, vd, wl, wr, code, w.scale)
        assert_close(to_f64(O), to_f64(L), ref_o, ref_l, code, f"{kernel} window {case} dt={code}")


def test_window_demo6_band_f32(kernel):
    """DEMO 6's local window |i - j| <= 64 at its own size (n = 512, d = 64),
    float32 path."""
    w, q, k, v = _dense_case(1, 1, 512, 64, "f32", False, seed=6)
    ref_o, ref_l = attention_ref(q, k, v, w.scale, False, window=(64, 64))
    O, L = run_window(q.to(DEV), k.to(DEV), v.to(DEV), 64, 64, fa.FA_F32, w.scale)
    assert_close(to_f64(O), to_f64(L), ref_o, ref_l, fa.FA_F32, "DEMO 6 band")


def test_window_special_cases_are_the_plain_paths(kernel):
    w, q, k, v = _dense_case(1, 2, 1100, 128, "bf16", True, seed=8)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    Oc, Lc = run_dense(qd, kd, vd, True, fa.FA_BF16, w.scale)
    Ow, Lw = run_window(qd, kd, vd, -1, 0, fa.FA_BF16, w.scale)
    assert torch.equal(Oc, Ow) and torch.equal(Lc, Lw)
    On, Ln = run_dense(qd, kd, vd, False, fa.FA_BF16, w.scale)
    Ow, Lw = run_window(qd, kd, vd, -1, -1, fa.FA_BF16, w.scale)
    assert torch.equal(On, Ow) and torch.equal(Ln, Lw)


def test_window_full_size_sampled_rows():
    """A causal local window (keys i-512 .. i) at the C3 shape."""
    w = C3
    q, k, v = make_inputs(w)
    O, L = run_window(q.to(DEV), k.to(DEV), v.to(DEV), 512, 0, fa.FA_BF16_OUT_F32, w.scale)
    for b, h in [(0, 0), (1, 15), (0, 7)]:
        rows = sample_rows(w.N, 48, seed=b * 16 + h)
        ref_o, ref_l = attention_rows(q[b, h], k[b, h], v[b, h], w.scale, False, rows, window=(512, 0))
        assert_close(to_f64(O[b, h, rows]), to_f64(L[b, h, rows]), ref_o, ref_l,
                     fa.FA_BF16_OUT_F32, f"band C3 b={b} h={h}")


@pytest.mark.parametrize("name", ["B2_H16_N4096_D128_bf16_band64",
                                  "B1_H16_N32768_D128_bf16_sliding4096"])
def test_window_bench_workloads_sampled_rows(name):
    """The band workloads the benchmark times, at full size and in the same
    launch (bf16 O), on sampled rows."""
    w = WORKLOADS[name]
    q, k, v = make_inputs(w)
    O, L = run_window(q.to(DEV), k.to(DEV), v.to(DEV), w.window[0], w.window[1], fa.FA_BF16,
                      w.scale)
    assert not torch.isnan(O.float()).any() and not torch.isnan(L).any()
    for b, h in [(0, 0), (w.B - 1, w.H - 1), (0, w.H // 2)]:
        rows = sample_rows(w.N, 40, seed=b * 16 + h)
        ref_o, ref_l = attention_rows(q[b, h], k[b, h], v[b, h], w.scale, False, rows,
                                      window=w.window)
        assert_close(to_f64(O[b, h, rows]), to_f64(L[b, h, rows]), ref_o, ref_l, fa.FA_BF16,
                     f"{name} b={b} h={h}")


def test_window_argument_checks():
    q = torch.zeros(1, 1, 16, 64, dtype=torch.bfloat16, device=DEV)
    O = torch.zeros_like(q)
    L = torch.zeros(1, 1, 16, device=DEV)
    assert fa.fa_fwd_window(q, q, q, O, L, 1, 1, 16, 64, 0.1, -2, 0, fa.FA_BF16, None) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd_window(q, q, q, O, L, 1, 1, 16, 64, 0.1, 0, -5, fa.FA_BF16, None) == fa.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("code", [fa.FA_BF16, fa.FA_BF16_OUT_F32])
def test_output_only_16_byte_aligned(kernel, code):
    """The epilogue stores 32 bytes at a time when O is 32-byte aligned and
    16 bytes otherwise; both give the same bits."""
    w, q, k, v = _dense_case(1, 2, 700, 128, "bf16", True, seed=44)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    O1, L1 = run_dense(qd, kd, vd, True, code, w.scale)
    odt = torch.bfloat16 if code == fa.FA_BF16 else torch.float32
    pad = 16 // torch.tensor([], dtype=odt).element_size()
    flat = torch.full((O1.numel() + 64,), float("nan"), dtype=odt, device=DEV)
    base = (-flat.data_ptr() // flat.element_size()) % (32 // flat.element_size())  # 32-aligned start
    O2 = flat[base + pad: base + pad + O1.numel()].view(O1.shape)
    assert O2.data_ptr() % 32 == 16
    L2 = torch.full_like(L1, float("nan"))
    st = fa.fa_fwd(qd, kd, vd, O2, L2, 1, 2, 700, 128, w.scale, 1, code, None)
    assert st == fa.FA_OK and fa.fa_check_device_error(None) == fa.FA_OK
    assert torch.equal(O1, O2) and torch.equal(L1, L2)
