"""Forward and backward passes over tensors of more than 2^31 elements (4.3 GB
each in bf16): every offset past element 2^31 must be computed in 64 bits.
Heads on both sides of that boundary are checked against the oracle.

Inputs are drawn on the GPU by the seeded device generator of the workloads
module; the oracle gets the sampled heads' slices copied to the host.  The
backward pass takes O and L from the library's own forward pass, as a
training step would; the oracle recomputes its forward pass per head.
Memory: about 35 GB of device memory per case.
"""

import numpy as np
import pytest
import torch

import exact_attention_24_gb300 as fa
from exact_attention_24_gb300 import build as fa_build
from exact_attention_24_gb300.workloads import Workload, make_inputs_device
from helpers import assert_close, half_ulp_bf16, to_f64
from oracle import attention_bwd_sampled, attention_ref

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
GRAD_TOL = 1e-2           # as for the other bf16 gradient checks
TWO31 = 1 << 31


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    fa_build.build()
    fa.load_library()
    yield
    fa.fa_set_options(fa.FA_KERNEL_AUTO, 0, 0)
    torch.cuda.empty_cache()


@pytest.fixture(params=["auto", "simt"])
def kernel(request):
    code = fa.FA_KERNEL_AUTO if request.param == "auto" else fa.FA_KERNEL_SIMT
    assert fa.fa_set_options(code, 0, 0) == fa.FA_OK
    yield request.param
    fa.fa_set_options(fa.FA_KERNEL_AUTO, 0, 0)
    torch.cuda.empty_cache()


def _check_grads(got, ref, what):
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        assert np.all(np.isfinite(g)), f"{what}: non-finite {name}"
        bound = GRAD_TOL * max(1.0, float(np.max(np.abs(r)))) + half_ulp_bf16(r)
        excess = np.abs(g - r) - bound
        i = np.unravel_index(np.argmax(excess), excess.shape)
        assert excess[i] <= 0, f"{what}: {name} err {abs(g[i] - r[i]):.3e} at {tuple(int(x) for x in i)}"


def _ok(st):
    assert st == fa.FA_OK, fa.fa_status_string(st) + " / " + fa.fa_last_cuda_error()
    assert fa.fa_check_device_error(None) == fa.FA_OK


def test_dense_past_2_31_elements(kernel):
    # 64 x 1025 heads of 256 x 128: head u starts at element u * 2^15, so
    # head 65536 starts exactly at element 2^31
    B, H, N, D = 64, 1025, 256, 128
    w = Workload("large_dense", B, H, N, D, "bf16", True, 31)
    assert B * H * N * D > TWO31
    q, k, v, do = make_inputs_device(w, DEV, count=4)
    O = torch.full_like(q, float("nan"))
    L = torch.full((B, H, N), float("nan"), dtype=torch.float32, device=DEV)
    _ok(fa.fa_fwd(q, k, v, O, L, B, H, N, D, w.scale, 1, fa.FA_BF16, None))
    units = [0, 65535, 65536, B * H - 1]
    for u in units:
        b, h = divmod(u, H)
        qh, kh, vh = (x[b, h].cpu() for x in (q, k, v))
        ref_o, ref_l = attention_ref(qh, kh, vh, w.scale, True)
        assert_close(to_f64(O[b, h]), to_f64(L[b, h]), ref_o, ref_l, fa.FA_BF16,
                     f"{kernel} dense head {u} (element {u * N * D})")
    grads = [torch.full_like(q, float("nan")) for _ in range(3)]
    nbytes = fa.fa_bwd_workspace_size(B, H, N)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=DEV)
    _ok(fa.fa_bwd(q, k, v, O, do, L, *grads, B, H, N, D, w.scale, 1, fa.FA_BF16, ws, nbytes, None))
    idx = np.array([0, 1, 127, 128, N - 1])
    for u in units:
        b, h = divmod(u, H)
        ref = attention_bwd_sampled(q[b, h].cpu(), k[b, h].cpu(), v[b, h].cpu(), do[b, h].cpu(),
                                    w.scale, True, idx, idx)
        _check_grads([to_f64(g[b, h, idx]) for g in grads], ref, f"{kernel} dense bwd head {u}")


def test_packed_past_2_31_elements(kernel):
    # 4100 sequences of 256 tokens, 16 heads of 128: token t starts at
    # element 2048 t, so sequence 4096 starts exactly at element 2^31
    n, S, H, D = 256, 4100, 16, 128
    lengths = (n,) * S
    w = Workload("large_packed", 0, H, 0, D, "bf16", True, 32, lengths=lengths)
    assert w.total * H * D > TWO31
    q, k, v, do = make_inputs_device(w, DEV, count=4)
    cu = torch.as_tensor(w.cu_seqlens, dtype=torch.int32, device=DEV)
    O = torch.full_like(q, float("nan"))
    L = torch.full((H, w.total), float("nan"), dtype=torch.float32, device=DEV)
    _ok(fa.fa_fwd_varlen(q, k, v, O, L, cu, S, w.total, n, H, D, w.scale, 1, fa.FA_BF16, None))
    picks = [(0, 0), (4095, 15), (4096, 0), (S - 1, 15)]
    for s, h in picks:
        a = s * n
        qh, kh, vh = (x[a:a + n, h].cpu() for x in (q, k, v))
        ref_o, ref_l = attention_ref(qh, kh, vh, w.scale, True)
        assert_close(to_f64(O[a:a + n, h]), to_f64(L[h, a:a + n]), ref_o, ref_l, fa.FA_BF16,
                     f"{kernel} packed seq {s} head {h}")
    grads = [torch.full_like(q, float("nan")) for _ in range(3)]
    nbytes = fa.fa_bwd_varlen_workspace_size(w.total, H)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=DEV)
    _ok(fa.fa_bwd_varlen(q, k, v, O, do, L, *grads, cu, S, w.total, n, H, D, w.scale, 1,
                         fa.FA_BF16, ws, nbytes, None))
    idx = np.array([0, 1, 127, 128, n - 1])
    for s, h in picks:
        a = s * n
        ref = attention_bwd_sampled(q[a:a + n, h].cpu(), k[a:a + n, h].cpu(), v[a:a + n, h].cpu(),
                                    do[a:a + n, h].cpu(), w.scale, True, idx, idx)
        _check_grads([to_f64(g[a + idx, h]) for g in grads], ref, f"{kernel} packed bwd seq {s} head {h}")
