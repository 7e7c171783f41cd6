"""The library inside CUDA graphs: each call sequence is run eagerly, captured
once, then replayed on new inputs copied into the same buffers; the replay
must give bitwise the results of an eager run on those inputs (the kernels
are deterministic).  Covers the dense, packed, band and split-key forward
passes, the backward passes and the FFMA kernel."""

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
    yield
    fa.fa_set_options(fa.FA_KERNEL_AUTO, 0, 0)


def _ok(st):
    assert st == fa.FA_OK, fa.fa_status_string(st) + " / " + fa.fa_last_cuda_error()


def _graph_matches_eager(inputs, outputs, step, new_inputs):
    """Run `step` eagerly on `new_inputs`, capture it with the original
    inputs in place, replay it on `new_inputs`, compare bitwise."""
    originals = [x.clone() for x in inputs]
    for x, y in zip(inputs, new_inputs):
        x.copy_(y)
    step()
    torch.cuda.synchronize()
    assert fa.fa_check_device_error(None) == fa.FA_OK
    expected = [o.clone() for o in outputs]
    for x, y in zip(inputs, originals):
        x.copy_(y)
    for o in outputs:
        o.fill_(float("nan")) if o.is_floating_point() else o.zero_()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # a warm-up on a side stream before capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        step()
    for x, y in zip(inputs, new_inputs):
        x.copy_(y)
    for o in outputs:
        o.fill_(float("nan")) if o.is_floating_point() else o.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert fa.fa_check_device_error(None) == fa.FA_OK
    for i, (o, e) in enumerate(zip(outputs, expected)):
        assert torch.equal(o, e), f"output {i} differs after graph replay"


def _dense(B, H, N, D, dtype, causal, seed):
    w = Workload("g", B, H, N, D, dtype, causal, seed)
    return w, [x.to(DEV) for x in make_inputs(w)] + [make_inputs(
        Workload("gdo", B, H, N, D, dtype, causal, seed + 7))[0].to(DEV)]


def test_dense_forward_and_backward_in_a_graph():
    w, (q, k, v, do) = _dense(1, 4, 1000, 128, "bf16", True, 21)
    _, new = _dense(1, 4, 1000, 128, "bf16", True, 22)
    B, H, N, D = q.shape
    O = torch.empty_like(q)
    L = torch.empty((B, H, N), dtype=torch.float32, device=DEV)
    grads = [torch.empty_like(q) for _ in range(3)]
    nbytes = fa.fa_bwd_workspace_size(B, H, N)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)

    def step():
        _ok(fa.fa_fwd(q, k, v, O, L, B, H, N, D, w.scale, 1, fa.FA_BF16, None))
        _ok(fa.fa_bwd(q, k, v, O, do, L, *grads, B, H, N, D, w.scale, 1, fa.FA_BF16, ws, nbytes, None))

    _graph_matches_eager([q, k, v, do], [O, L, *grads], step, new)


def test_packed_forward_and_backward_in_a_graph():
    lengths = (300, 0, 129, 700, 64)
    H, D = 3, 64
    w = Workload("gv", 0, H, 0, D, "bf16", True, 23, lengths=lengths)
    q, k, v = (x.to(DEV) for x in make_inputs(w))
    do = make_inputs(Workload("gvdo", 0, H, 0, D, "bf16", True, 24, lengths=lengths))[0].to(DEV)
    w2 = Workload("gv2", 0, H, 0, D, "bf16", True, 25, lengths=lengths)
    new = [x.to(DEV) for x in make_inputs(w2)] + [make_inputs(
        Workload("gvdo2", 0, H, 0, D, "bf16", True, 26, lengths=lengths))[0].to(DEV)]
    cu = torch.as_tensor(w.cu_seqlens, dtype=torch.int32, device=DEV)
    O = torch.empty_like(q)
    L = torch.empty((H, w.total), dtype=torch.float32, device=DEV)
    grads = [torch.empty_like(q) for _ in range(3)]
    nbytes = fa.fa_bwd_varlen_workspace_size(w.total, H)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    S = len(lengths)

    def step():
        _ok(fa.fa_fwd_varlen(q, k, v, O, L, cu, S, w.total, w.max_seqlen, H, D, w.scale, 1, fa.FA_BF16, None))
        _ok(fa.fa_bwd_varlen(q, k, v, O, do, L, *grads, cu, S, w.total, w.max_seqlen, H, D, w.scale, 1,
                             fa.FA_BF16, ws, nbytes, None))

    _graph_matches_eager([q, k, v, do], [O, L, *grads], step, new)


def test_band_forward_and_backward_in_a_graph():
    w, (q, k, v, do) = _dense(1, 2, 900, 128, "bf16", False, 27)
    _, new = _dense(1, 2, 900, 128, "bf16", False, 28)
    B, H, N, D = q.shape
    O = torch.empty_like(q)
    L = torch.empty((B, H, N), dtype=torch.float32, device=DEV)
    grads = [torch.empty_like(q) for _ in range(3)]
    nbytes = fa.fa_bwd_workspace_size(B, H, N)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)

    def step():
        _ok(fa.fa_fwd_window(q, k, v, O, L, B, H, N, D, w.scale, 64, 64, fa.FA_BF16, None))
        _ok(fa.fa_bwd_window(q, k, v, O, do, L, *grads, B, H, N, D, w.scale, 64, 64, fa.FA_BF16, ws,
                             nbytes, None))

    _graph_matches_eager([q, k, v, do], [O, L, *grads], step, new)


def test_split_key_forward_in_a_graph():
    w, (q, k, v, _) = _dense(1, 2, 3000, 64, "bf16", True, 29)
    _, new = _dense(1, 2, 3000, 64, "bf16", True, 30)
    B, H, N, D = q.shape
    O = torch.empty_like(q)
    L = torch.empty((B, H, N), dtype=torch.float32, device=DEV)
    nbytes = fa.fa_fwd_splitkv_workspace_size(B, H, N, D, 4)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)

    def step():
        _ok(fa.fa_fwd_splitkv(q, k, v, O, L, B, H, N, D, w.scale, 1, fa.FA_BF16, 4, ws, nbytes, None))

    _graph_matches_eager([q, k, v], [O, L], step, new[:3])


def test_ffma_forward_in_a_graph():
    w, (q, k, v, _) = _dense(1, 1, 256, 64, "f32", False, 31)
    _, new = _dense(1, 1, 256, 64, "f32", False, 32)
    B, H, N, D = q.shape
    O = torch.empty_like(q)
    L = torch.empty((B, H, N), dtype=torch.float32, device=DEV)

    def step():
        _ok(fa.fa_fwd(q, k, v, O, L, B, H, N, D, w.scale, 0, fa.FA_F32, None))

    _graph_matches_eager([q, k, v], [O, L], step, new[:3])
