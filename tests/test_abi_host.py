"""Host-side checks of the C-ABI library: it loads, exports every symbol that
include/fa.h declares, and rejects bad arguments before touching CUDA.
CPU only -- no call here launches a kernel: every call either fails
validation or (on a machine without a GPU) fails to find a device.  Fake
addresses are used only in calls that must be rejected before any launch."""

import os
import re

import pytest
import torch

import exact_attention_24_gb300 as fa
from exact_attention_24_gb300 import build as fa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    fa_build.build()
    return fa.load_library()


def _declared_symbols():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            names += re.findall(r"FA_API\s+[\w\s\*]*?\b(fa_\w+)\s*\(", text)
    return names


def test_exports_every_declared_symbol(lib):
    declared = _declared_symbols()
    assert set(declared) >= set(fa.EXPORTED_SYMBOLS)
    for name in declared:
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(5):
        assert fa.fa_status_string(code).startswith("FA_")
    assert "unknown" in fa.fa_status_string(99)


A = 1 << 20          # fake, 16-byte aligned "device" addresses: never touched
STEP = 1 << 30


def _ptrs():
    return [A + i * STEP for i in range(5)]


def test_rejects_unsupported_head_dim(lib):
    q, k, v, o, l = _ptrs()
    for D in (32, 96, 256):
        assert fa.fa_fwd(q, k, v, o, l, 1, 1, 16, D, 0.1, 0, fa.FA_BF16, 0) == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_fwd(q, k, v, o, l, 1, 1, 16, 0, 0.1, 0, fa.FA_BF16, 0) == fa.FA_ERR_INVALID_ARG


def test_rejects_bad_arguments(lib):
    q, k, v, o, l = _ptrs()
    bad = fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd(q, k, v, o, l, -1, 1, 16, 64, 0.1, 0, fa.FA_BF16, 0) == bad
    assert fa.fa_fwd(q, k, v, o, l, 1, -1, 16, 64, 0.1, 0, fa.FA_BF16, 0) == bad
    assert fa.fa_fwd(q, k, v, o, l, 1, 1, -16, 64, 0.1, 0, fa.FA_BF16, 0) == bad
    assert fa.fa_fwd(q, k, v, o, l, 1, 1, 16, 64, float("nan"), 0, fa.FA_BF16, 0) == bad
    assert fa.fa_fwd(q, k, v, o, l, 1, 1, 16, 64, float("inf"), 0, fa.FA_BF16, 0) == bad
    assert fa.fa_fwd(q, k, v, o, l, 1, 1, 16, 64, 0.1, 2, fa.FA_BF16, 0) == bad
    assert fa.fa_fwd(q, k, v, o, l, 1, 1, 16, 64, 0.1, 0, 7, 0) == bad
    # null and misaligned pointers
    assert fa.fa_fwd(0, k, v, o, l, 1, 1, 16, 64, 0.1, 0, fa.FA_BF16, 0) == bad
    assert fa.fa_fwd(q, k, v, 0, l, 1, 1, 16, 64, 0.1, 0, fa.FA_BF16, 0) == bad
    assert fa.fa_fwd(q + 8, k, v, o, l, 1, 1, 16, 64, 0.1, 0, fa.FA_BF16, 0) == bad
    assert fa.fa_fwd(q, k, v, o, l + 4, 1, 1, 16, 64, 0.1, 0, fa.FA_BF16, 0) == bad
    # outputs overlapping inputs or each other
    assert fa.fa_fwd(q, k, v, q + 64, l, 1, 1, 16, 64, 0.1, 0, fa.FA_BF16, 0) == bad
    assert fa.fa_fwd(q, k, v, o, o + 16, 1, 1, 16, 64, 0.1, 0, fa.FA_BF16, 0) == bad
    # inputs may alias one another.  The fake pointers would reach a kernel
    # once validation passes, so this runs only where no GPU exists.
    if not torch.cuda.is_available():
        st = fa.fa_fwd(q, q, q, o, l, 1, 1, 16, 64, 0.1, 0, fa.FA_BF16, 0)
        assert st == fa.FA_ERR_CUDA


def test_zero_sizes_are_noops(lib):
    for B, H, N in [(0, 1, 16), (1, 0, 16), (1, 1, 0)]:
        assert fa.fa_fwd(0, 0, 0, 0, 0, B, H, N, 64, 0.1, 1, fa.FA_BF16, 0) == fa.FA_OK
    assert fa.fa_fwd_varlen(0, 0, 0, 0, 0, 0, 0, 0, 0, 4, 128, 0.1, 1, fa.FA_BF16, 0) == fa.FA_OK


def test_varlen_argument_checks(lib):
    q, k, v, o, l = _ptrs()
    cu = A + 5 * STEP
    bad = fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd_varlen(q, k, v, o, l, cu, -1, 100, 50, 2, 64, 0.1, 1, fa.FA_BF16, 0) == bad
    assert fa.fa_fwd_varlen(q, k, v, o, l, cu, 2, -1, 50, 2, 64, 0.1, 1, fa.FA_BF16, 0) == bad
    assert fa.fa_fwd_varlen(q, k, v, o, l, cu, 2, 100, -5, 2, 64, 0.1, 1, fa.FA_BF16, 0) == bad
    assert fa.fa_fwd_varlen(q, k, v, o, l, 0, 2, 100, 50, 2, 64, 0.1, 1, fa.FA_BF16, 0) == bad
    assert fa.fa_fwd_varlen(q, k, v, o, l, cu + 2, 2, 100, 50, 2, 64, 0.1, 1, fa.FA_BF16, 0) == bad
    assert fa.fa_fwd_varlen(q, k, v, o, l, cu, 2, 100, 50, 2, 80, 0.1, 1, fa.FA_BF16, 0) == fa.FA_ERR_UNSUPPORTED


def test_options_roundtrip(lib):
    before = fa.fa_get_options()
    try:
        assert fa.fa_set_options(fa.FA_KERNEL_SIMT, 7, 12345) == fa.FA_OK
        assert fa.fa_get_options() == {"kernel": 1, "grid_ctas": 7, "wait_limit_ns": 12345}
        assert fa.fa_set_options(9, 0, 0) == fa.FA_ERR_INVALID_ARG
        assert fa.fa_set_options(0, -1, 0) == fa.FA_ERR_INVALID_ARG
        # fp32 with the tensor-core kernel forced is unsupported
        fa.fa_set_options(fa.FA_KERNEL_TC, 0, 0)
        q, k, v, o, l = _ptrs()
        assert fa.fa_fwd(q, k, v, o, l, 1, 1, 16, 64, 0.1, 0, fa.FA_F32, 0) in (
            fa.FA_ERR_UNSUPPORTED, fa.FA_ERR_CUDA)
    finally:
        fa.fa_set_options(before["kernel"], before["grid_ctas"], before["wait_limit_ns"])


def test_watchdog_limit_checked(lib):
    assert fa.fa_watchdog_selftest(0, 0) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_watchdog_selftest(2_000_000_000, 0) == fa.FA_ERR_INVALID_ARG


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU behaviour")
def test_valid_call_without_gpu_fails_loudly(lib):
    """With no CUDA device the library reports FA_ERR_CUDA; it never computes
    on the CPU instead."""
    q, k, v, o, l = _ptrs()
    assert fa.fa_fwd(q, k, v, o, l, 1, 1, 16, 64, 0.1, 0, fa.FA_BF16, 0) == fa.FA_ERR_CUDA
    assert fa.fa_last_cuda_error() != "no error"   # the runtime's reason is kept
    assert fa.fa_check_device_error(0) == fa.FA_ERR_CUDA


@pytest.mark.skipif(torch.cuda.is_available(), reason="fake addresses are for GPU-less hosts only")
def test_bf16_case_the_tensor_cores_cannot_take_is_reported(lib):
    """A bf16 problem the tensor-core kernels do not take (here: more work
    items than their 32-bit numbering allows) returns FA_ERR_UNSUPPORTED to
    the caller, decided on the host before any CUDA call -- it is never run on
    the FFMA kernel instead.  Without a GPU, any CUDA call would have turned
    the result into FA_ERR_CUDA."""
    far = [(i + 1) << 47 for i in range(10)]   # fake, far apart: nothing overlaps
    q, k, v, o, l = far[:5]
    H, N = 1 << 22, 1 << 16                   # 256 blocks x 2^22 heads = 2^30 items
    for kernel in (fa.FA_KERNEL_AUTO, fa.FA_KERNEL_TC):
        assert fa.fa_set_options(kernel, 0, 0) == fa.FA_OK
        try:
            for code in (fa.FA_BF16, fa.FA_BF16_OUT_F32):
                for causal in (0, 1):
                    assert fa.fa_fwd(q, k, v, o, l, 1, H, N, 64, 0.1, causal, code, 0) == \
                        fa.FA_ERR_UNSUPPORTED
            # backward: 2^11 key blocks x 2^20 heads = 2^31 blocks
            Hb, Nb = 1 << 20, 1 << 18
            nws = fa.fa_bwd_workspace_size(1, Hb, Nb)
            assert fa.fa_bwd(*far[:9], 1, Hb, Nb, 64, 0.1, 1, fa.FA_BF16, far[9], nws, 0) == \
                fa.FA_ERR_UNSUPPORTED
            # one item fewer is taken (and, with no GPU, then fails in CUDA)
            assert fa.fa_fwd(q, k, v, o, l, 1, H - 1, N, 64, 0.1, 1, fa.FA_BF16, 0) == fa.FA_ERR_CUDA
        finally:
            fa.fa_set_options(fa.FA_KERNEL_AUTO, 0, 0)
    # float32 never reaches the tensor-core kernel
    assert fa.fa_set_options(fa.FA_KERNEL_TC, 0, 0) == fa.FA_OK
    try:
        assert fa.fa_fwd(q, k, v, o, l, 1, 1, 16, 64, 0.1, 0, fa.FA_F32, 0) == fa.FA_ERR_UNSUPPORTED
    finally:
        fa.fa_set_options(fa.FA_KERNEL_AUTO, 0, 0)


def test_product_package_does_not_import_oracle():
    """The oracle is test infrastructure: nothing in the product package may
    import or load it."""
    pkg = os.path.join(ROOT, "exact_attention_24_gb300")
    pat = re.compile(r"^\s*(import\s+oracle|from\s+oracle)|oracle/|oracle\.", re.M)
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert not pat.search(text), f


def test_splitkv_argument_checks(lib):
    q, k, v, o, l = _ptrs()
    ws = A + 6 * STEP
    bad = fa.FA_ERR_INVALID_ARG
    args = (q, k, v, o, l, 1, 1, 1024, 128, 0.1, 1)
    assert fa.fa_fwd_splitkv(*args, fa.FA_BF16, 65, ws, 1 << 30, 0) == bad
    assert fa.fa_fwd_splitkv(*args, fa.FA_BF16, -1, ws, 1 << 30, 0) == bad
    assert fa.fa_fwd_splitkv(*args, fa.FA_F32, 3, ws, 1 << 30, 0) == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_fwd_splitkv(*args, fa.FA_BF16, 3, 0, 1 << 30, 0) == bad        # no workspace
    assert fa.fa_fwd_splitkv(*args, fa.FA_BF16, 3, ws + 8, 1 << 30, 0) == bad   # misaligned
    need = fa.fa_fwd_splitkv_workspace_size(1, 1, 1024, 128, 3)
    assert fa.fa_fwd_splitkv(*args, fa.FA_BF16, 3, ws, need - 1, 0) == bad      # too small
    assert fa.fa_fwd_splitkv(*args, fa.FA_BF16, 3, q, need, 0) == bad           # overlaps Q


def test_splitkv_workspace_size(lib):
    # partial O in fp32 then partial L, each padded to 256 bytes
    assert fa.fa_fwd_splitkv_workspace_size(1, 1, 1024, 128, 3) == 3 * 1024 * 128 * 4 + 3 * 1024 * 4
    assert fa.fa_fwd_splitkv_workspace_size(2, 3, 1000, 64, 4) == \
        -(-4 * 6 * 1000 * 64 * 4 // 256) * 256 + -(-4 * 6 * 1000 * 4 // 256) * 256
    assert fa.fa_fwd_splitkv_workspace_size(1, 1, 1024, 128, 1) == 0     # one split: none needed
    assert fa.fa_fwd_splitkv_workspace_size(1, 1, 300, 64, 9) == \
        fa.fa_fwd_splitkv_workspace_size(1, 1, 300, 64, 3)                # capped at ceil(N/128)
    assert fa.fa_fwd_splitkv_workspace_size(1, 1, 1024, 96, 3) == 0      # unsupported D
    assert fa.fa_fwd_splitkv_workspace_size(0, 1, 1024, 128, 3) == 0


# ------------------------------------------------------------ backward --
def _bwd_ptrs():
    return [A + i * STEP for i in range(10)]   # Q K V O dO L dQ dK dV workspace


def test_bwd_workspace_size(lib):
    assert fa.fa_bwd_workspace_size(2, 16, 4096) == 2 * 16 * 4096 * 4
    assert fa.fa_bwd_workspace_size(1, 1, 3) == 256          # rounded up to 256
    for B, H, N in [(0, 1, 16), (1, 0, 16), (1, 1, 0), (-1, 1, 16)]:
        assert fa.fa_bwd_workspace_size(B, H, N) == 0


def test_bwd_argument_checks(lib):
    q, k, v, o, do, l, dq, dk, dv, ws = _bwd_ptrs()
    nws = fa.fa_bwd_workspace_size(1, 1, 16)
    bad, uns = fa.FA_ERR_INVALID_ARG, fa.FA_ERR_UNSUPPORTED

    def call(*, B=1, H=1, N=16, D=64, scale=0.1, causal=0, dtype=fa.FA_BF16, p=None, w=ws,
             nw=nws):
        args = list(p or (q, k, v, o, do, l, dq, dk, dv))
        return fa.fa_bwd(*args, B, H, N, D, scale, causal, dtype, w, nw, 0)

    assert call(B=-1) == bad and call(H=-1) == bad and call(N=-4) == bad
    assert call(D=0) == bad and call(D=96) == uns and call(D=256) == uns
    assert call(scale=float("nan")) == bad and call(causal=2) == bad and call(dtype=9) == bad
    # null or misaligned pointers, short or missing workspace
    for i in range(9):
        p = [q, k, v, o, do, l, dq, dk, dv]
        p[i] = 0
        assert call(p=p) == bad
        p[i] = [q, k, v, o, do, l, dq, dk, dv][i] + 8
        assert call(p=p) == bad
    assert call(w=0) == bad and call(w=ws + 4) == bad and call(nw=nws - 4) == bad
    # outputs overlapping inputs, each other or the workspace
    assert call(p=[q, k, v, o, do, l, q + 64, dk, dv]) == bad
    assert call(p=[q, k, v, o, do, l, dq, dq + 64, dv]) == bad
    assert call(p=[q, k, v, o, do, l, dq, dk, l]) == bad
    assert call(p=[q, k, v, o, do, l, dq, dk, ws]) == bad
    assert call(w=do + 32) == bad
    # empty problems are no-ops and touch nothing
    for B, H, N in [(0, 1, 16), (1, 0, 16), (1, 1, 0)]:
        assert fa.fa_bwd(0, 0, 0, 0, 0, 0, 0, 0, 0, B, H, N, 64, 0.1, 1, fa.FA_BF16, 0, 0,
                         0) == fa.FA_OK
    if not torch.cuda.is_available():   # valid arguments reach CUDA, which is absent
        assert call() == fa.FA_ERR_CUDA
        assert call(dtype=fa.FA_F32) == fa.FA_ERR_CUDA


def test_bwd_varlen_argument_checks(lib):
    q, k, v, o, do, l, dq, dk, dv, ws = _bwd_ptrs()
    cu = A + 11 * STEP
    nws = fa.fa_bwd_varlen_workspace_size(100, 2)
    assert nws == 1024 and fa.fa_bwd_varlen_workspace_size(0, 2) == 0
    bad = fa.FA_ERR_INVALID_ARG

    def call(*, c=cu, ns=2, tot=100, mx=50, H=2, D=64, p=None, w=ws, nw=nws):
        args = list(p or (q, k, v, o, do, l, dq, dk, dv))
        return fa.fa_bwd_varlen(*args, c, ns, tot, mx, H, D, 0.1, 1, fa.FA_BF16, w, nw, 0)

    assert call(ns=-1) == bad and call(tot=-1) == bad and call(mx=-3) == bad and call(H=-1) == bad
    assert call(c=0) == bad and call(c=cu + 2) == bad
    assert call(D=80) == fa.FA_ERR_UNSUPPORTED
    assert call(w=0) == bad and call(nw=4 * 100 * 2 - 4) == bad   # one float short
    assert call(p=[q, k, v, o, do, l, q + 64, dk, dv]) == bad
    assert fa.fa_bwd_varlen(0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 2, 64, 0.1, 1, fa.FA_BF16, 0, 0,
                            0) == fa.FA_OK
    if not torch.cuda.is_available():
        assert call() == fa.FA_ERR_CUDA


def test_bwd_window_argument_checks(lib):
    q, k, v, o, do, l, dq, dk, dv, ws = _bwd_ptrs()
    nws = fa.fa_bwd_workspace_size(1, 1, 16)
    bad = fa.FA_ERR_INVALID_ARG
    args = (q, k, v, o, do, l, dq, dk, dv, 1, 1, 16, 64, 0.1)
    assert fa.fa_bwd_window(*args, -2, 0, fa.FA_BF16, ws, nws, 0) == bad
    assert fa.fa_bwd_window(*args, 3, -7, fa.FA_BF16, ws, nws, 0) == bad
    assert fa.fa_bwd_window(*args, 3, 3, fa.FA_BF16, 0, nws, 0) == bad
    if not torch.cuda.is_available():
        assert fa.fa_bwd_window(*args, 3, 3, fa.FA_BF16, ws, nws, 0) == fa.FA_ERR_CUDA


def test_host_forward_argument_checks(lib):
    """fa_fwd_host rejects bad arguments before any copy is enqueued: chunk
    counts outside 1..64, null host buffers and every fa_fwd check of the
    device staging buffers."""
    qd, kd, vd, od, ld = _ptrs()
    qh, kh, vh, oh, lh = (A + (10 + i) * STEP for i in range(5))
    bad = fa.FA_ERR_INVALID_ARG
    dims = (2, 3, 100, 64, 0.1, 1, fa.FA_BF16)
    for chunks in (0, -1, 65):
        assert fa.fa_fwd_host(qh, kh, vh, oh, lh, qd, kd, vd, od, ld, *dims, chunks, 0) == bad
    assert fa.fa_fwd_host(0, kh, vh, oh, lh, qd, kd, vd, od, ld, *dims, 4, 0) == bad
    assert fa.fa_fwd_host(qh, kh, vh, oh, 0, qd, kd, vd, od, ld, *dims, 4, 0) == bad
    assert fa.fa_fwd_host(qh, kh, vh, oh, lh, qd, kd, vd, 0, ld, *dims, 4, 0) == bad
    assert fa.fa_fwd_host(qh, kh, vh, oh, lh, qd + 8, kd, vd, od, ld, *dims, 4, 0) == bad
    assert fa.fa_fwd_host(qh, kh, vh, oh, lh, qd, kd, vd, qd + 64, ld, *dims, 4, 0) == bad
    assert fa.fa_fwd_host(qh, kh, vh, oh, lh, qd, kd, vd, od, ld, 2, 3, 100, 96, 0.1, 1,
                          fa.FA_BF16, 4, 0) == fa.FA_ERR_UNSUPPORTED
    # empty batches are no-ops, host pointers unused
    assert fa.fa_fwd_host(0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 3, 100, 64, 0.1, 1, fa.FA_BF16, 4, 0) == fa.FA_OK
