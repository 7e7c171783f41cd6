"""The allocation-free split-key entry point, fa_fwd_splitkv_noalloc, for
callers that may not allocate device memory (a plugin inside a host program
that owns the device-memory budget, a latency-critical caller that must not
call cudaMalloc/cudaFree, C code handed only its buffers).

Two calls in a row, each through the C ABI, checked against the existing
fa_fwd_splitkv (which takes a caller workspace) on the same inputs, and on
sampled rows against the float64 oracle, with the parity tolerances of the
other GPU tests.  Collected last on purpose.
"""

import numpy as np
import pytest
import torch

import exact_attention_24_gb300 as fa
from exact_attention_24_gb300 import build as fa_build
from exact_attention_24_gb300.workloads import Workload, make_inputs
from helpers import TOL, assert_close, half_ulp_bf16, sample_rows, to_f64
from oracle import attention_rows

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    fa_build.build()
    fa.load_library()
    fa.fa_set_options(fa.FA_KERNEL_AUTO, 0, 0)


def _outputs(w, code):
    odt = torch.bfloat16 if code == fa.FA_BF16 else torch.float32
    O = torch.full((w.B, w.H, w.N, w.D), float("nan"), dtype=odt, device=DEV)
    L = torch.full((w.B, w.H, w.N), float("nan"), dtype=torch.float32, device=DEV)
    return O, L


def _with_workspace(q, k, v, w, code, splits):
    O, L = _outputs(w, code)
    nbytes = fa.fa_fwd_splitkv_workspace_size(w.B, w.H, w.N, w.D, splits)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=DEV)
    st = fa.fa_fwd_splitkv(q, k, v, O, L, w.B, w.H, w.N, w.D, w.scale, int(w.causal), code,
                           splits, ws, nbytes, None)
    assert st == fa.FA_OK, fa.fa_status_string(st)
    assert fa.fa_check_device_error(None) == fa.FA_OK
    return O, L


def _noalloc(q, k, v, w, code, splits):
    O, L = _outputs(w, code)
    st = fa.fa_fwd_splitkv_noalloc(q, k, v, O, L, w.B, w.H, w.N, w.D, w.scale, int(w.causal),
                                   code, splits, None)
    assert st == fa.FA_OK, fa.fa_status_string(st) + " / " + fa.fa_last_cuda_error()
    assert fa.fa_check_device_error(None) == fa.FA_OK
    return O, L


def _check(got, ref, code, what):
    tol_o, tol_l = TOL[code]
    go, gl = to_f64(got[0]), to_f64(got[1])
    ro, rl = to_f64(ref[0]), to_f64(ref[1])
    bound = tol_o + (half_ulp_bf16(ro) if code == fa.FA_BF16 else 0.0)
    assert np.all(np.isfinite(go)) and np.all(np.isfinite(gl)), what
    assert np.all(np.abs(go - ro) <= bound), f"{what}: O differs by {np.max(np.abs(go - ro)):.3e}"
    assert np.max(np.abs(gl - rl)) <= tol_l, f"{what}: L differs by {np.max(np.abs(gl - rl)):.3e}"


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    cases = [
        (Workload("a", 1, 2, 4096, 128, "bf16", True, 21), fa.FA_BF16, 4),
        (Workload("b", 2, 1, 1500, 64, "bf16", False, 22), fa.FA_BF16_OUT_F32, 3),
    ]
    for w, code, splits in cases:   # two different calls in a row
        need = fa.fa_fwd_splitkv_workspace_size(w.B, w.H, w.N, w.D, splits)
        # more than one split, so both calls really go through their scratch
        assert 0 < need <= fa.FA_NOALLOC_SCRATCH_BYTES
        qh, kh, vh = make_inputs(w)
        q, k, v = qh.to(DEV), kh.to(DEV), vh.to(DEV)
        ref = _with_workspace(q, k, v, w, code, splits)
        got = _noalloc(q, k, v, w, code, splits)
        _check(got, ref, code, f"{w.name} splits={splits}")
        # and against the float64 oracle on sampled rows of every head
        for b in range(w.B):
            for h in range(w.H):
                rows = sample_rows(w.N, 24, seed=31 * b + h)
                ro, rl = attention_rows(qh[b, h], kh[b, h], vh[b, h], w.scale, w.causal, rows)
                assert_close(to_f64(got[0][b, h, rows]), to_f64(got[1][b, h, rows]), ro, rl, code,
                             f"{w.name} b={b} h={h} vs oracle")


def test_noalloc_rejects_sizes_beyond_its_scratch():
    w = Workload("big", 1, 16, 16384, 128, "bf16", True, 23)
    assert fa.fa_fwd_splitkv_workspace_size(w.B, w.H, w.N, w.D, 8) > fa.FA_NOALLOC_SCRATCH_BYTES
    q = torch.zeros((w.B, w.H, w.N, w.D), dtype=torch.bfloat16, device=DEV)
    O, L = _outputs(w, fa.FA_BF16)
    st = fa.fa_fwd_splitkv_noalloc(q, q, q, O, L, w.B, w.H, w.N, w.D, w.scale, 1, fa.FA_BF16, 8,
                                   None)
    assert st == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_check_device_error(None) == fa.FA_OK
