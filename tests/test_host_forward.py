"""fa_fwd_host: the forward pass on host tensors with the transfers
overlapped in runs of problems.  The outputs copied back must be bitwise
those of fa_fwd on the same data (each problem's result does not depend on
how the batch is cut), for several run counts, N with and without a
multiple of 4 (run boundaries keep L's slices aligned), bf16 and fp32."""

import pytest
import torch

import exact_attention_24_gb300 as fa
from exact_attention_24_gb300 import build as fa_build
from exact_attention_24_gb300.workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    fa_build.build()
    fa.load_library()


@pytest.mark.parametrize("shape", [(2, 5, 1000, 128, True, "bf16"), (3, 3, 257, 64, False, "bf16"),
                                   (1, 7, 130, 64, True, "f32"), (1, 1, 4096, 128, True, "bf16")],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("chunks", [1, 3, 8, 64])
def test_host_forward_matches_device_forward(shape, chunks):
    B, H, N, D, causal, dt = shape
    w = Workload("host", B, H, N, D, dt, causal, 41)
    q, k, v = make_inputs(w)
    code = fa.FA_F32 if dt == "f32" else fa.FA_BF16
    qh, kh, vh = (x.pin_memory() for x in (q, k, v))
    oh = torch.full(q.shape, float("nan"), dtype=q.dtype).pin_memory()
    lh = torch.full(q.shape[:-1], float("nan"), dtype=torch.float32).pin_memory()
    stage = [torch.empty_like(q, device=DEV) for _ in range(4)] + [torch.empty(q.shape[:-1], device=DEV)]
    stream = torch.cuda.current_stream()
    st = fa.fa_fwd_host(qh, kh, vh, oh, lh, *stage, B, H, N, D, w.scale, int(causal), code, chunks, stream)
    assert st == fa.FA_OK, fa.fa_status_string(st) + " / " + fa.fa_last_cuda_error()
    torch.cuda.synchronize()
    assert fa.fa_check_device_error(None) == fa.FA_OK
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    O = torch.empty_like(qd)
    L = torch.empty(q.shape[:-1], device=DEV)
    assert fa.fa_fwd(qd, kd, vd, O, L, B, H, N, D, w.scale, int(causal), code, None) == fa.FA_OK
    torch.cuda.synchronize()
    assert torch.equal(oh, O.cpu()) and torch.equal(lh, L.cpu())
    # the staging buffers hold the inputs and outputs of the pass
    assert torch.equal(stage[0].cpu(), q) and torch.equal(stage[3].cpu(), oh)


def test_host_forward_orders_after_earlier_stream_work():
    """The copies wait for work already on the stream: a device buffer still
    being written by an earlier kernel is not read too early, and the stream
    completes only after the last device-to-host copy."""
    B, H, N, D = 1, 8, 2048, 128
    w = Workload("host2", B, H, N, D, "bf16", True, 43)
    q, k, v = make_inputs(w)
    qh, kh, vh = (x.pin_memory() for x in (q, k, v))
    oh = torch.empty_like(q).pin_memory()
    lh = torch.empty(q.shape[:-1]).pin_memory()
    stage = [torch.empty_like(q, device=DEV) for _ in range(4)] + [torch.empty(q.shape[:-1], device=DEV)]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for x in stage:
            x.fill_(1.0)            # earlier work on the stream touching the staging area
        st = fa.fa_fwd_host(qh, kh, vh, oh, lh, *stage, B, H, N, D, w.scale, 1, fa.FA_BF16, 8, s)
        assert st == fa.FA_OK
        done = torch.cuda.Event()
        done.record(s)
    done.synchronize()
    O, L = fa.attention(q.to(DEV), k.to(DEV), v.to(DEV), causal=True, scale=w.scale)
    assert torch.equal(oh, O.cpu()) and torch.equal(lh, L.cpu())


def test_host_forward_with_pageable_memory():
    """Pageable (not pinned) host tensors give the same results; the copies
    then do not overlap, but correctness does not depend on pinning."""
    B, H, N, D = 2, 3, 300, 64
    w = Workload("host3", B, H, N, D, "bf16", False, 44)
    q, k, v = make_inputs(w)
    oh = torch.full(q.shape, float("nan"), dtype=q.dtype)
    lh = torch.full(q.shape[:-1], float("nan"), dtype=torch.float32)
    stage = [torch.empty_like(q, device=DEV) for _ in range(4)] + [torch.empty(q.shape[:-1], device=DEV)]
    st = fa.fa_fwd_host(q, k, v, oh, lh, *stage, B, H, N, D, w.scale, 0, fa.FA_BF16, 3, None)
    assert st == fa.FA_OK, fa.fa_status_string(st) + " / " + fa.fa_last_cuda_error()
    torch.cuda.synchronize()
    O, L = fa.attention(q.to(DEV), k.to(DEV), v.to(DEV), causal=False, scale=w.scale)
    assert torch.equal(oh, O.cpu()) and torch.equal(lh, L.cpu())
