"""GB300 (sm_103a) FlashAttention-2 forward pass: Python binding.

Thin ctypes marshalling over the C ABI declared in ``include/fa.h``; every
step of the computation runs in the CUDA kernels of ``libfa_gb300.so``.
There is no CPU or PyTorch fallback: if the library is missing, loading it
raises.  PyTorch is used only for device memory and streams.

Raw entry points (same names and argument order as the C ABI; tensor
arguments may be torch tensors or integer device addresses, the stream a
``torch.cuda.Stream``, an integer handle or ``None`` for torch's current
stream): ``fa_fwd``, ``fa_fwd_varlen``, ``fa_check_device_error``,
``fa_status_string``, ``fa_set_options``, ``fa_get_options``,
``fa_watchdog_selftest``.

Convenience: ``attention(q, k, v, ...)`` and ``attention_varlen(...)``
allocate O and L with torch and call the raw entry points.
"""

from __future__ import annotations

import ctypes
import math
import os

__all__ = [
    "FA_OK", "FA_ERR_INVALID_ARG", "FA_ERR_UNSUPPORTED", "FA_ERR_CUDA",
    "FA_ERR_DEVICE_TIMEOUT", "FA_F32", "FA_BF16", "FA_BF16_OUT_F32",
    "FA_KERNEL_AUTO", "FA_KERNEL_SIMT", "FA_KERNEL_TC", "FaError",
    "load_library", "library_path", "fa_fwd", "fa_fwd_window", "fa_fwd_varlen", "fa_fwd_splitkv",
    "fa_fwd_splitkv_workspace_size", "fa_fwd_splitkv_noalloc", "FA_NOALLOC_SCRATCH_BYTES",
    "fa_fwd_host",
    "fa_check_device_error", "fa_status_string", "fa_last_cuda_error", "fa_set_options",
    "fa_get_options", "fa_watchdog_selftest", "attention",
    "attention_varlen", "EXPORTED_SYMBOLS", "fa_bwd", "fa_bwd_workspace_size",
    "fa_bwd_varlen", "fa_bwd_varlen_workspace_size", "fa_bwd_window", "attention_bwd",
]

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, \
    FA_ERR_DEVICE_TIMEOUT = 0, 1, 2, 3, 4
FA_F32, FA_BF16, FA_BF16_OUT_F32 = 0, 1, 2
FA_KERNEL_AUTO, FA_KERNEL_SIMT, FA_KERNEL_TC = 0, 1, 2

EXPORTED_SYMBOLS = ("fa_fwd", "fa_fwd_window", "fa_fwd_varlen", "fa_fwd_splitkv",
                    "fa_fwd_splitkv_workspace_size", "fa_fwd_splitkv_noalloc", "fa_fwd_host",
                    "fa_bwd", "fa_bwd_workspace_size", "fa_bwd_window", "fa_bwd_varlen",
                    "fa_bwd_varlen_workspace_size", "fa_check_device_error",
                    "fa_status_string", "fa_last_cuda_error", "fa_set_options",
                    "fa_get_options", "fa_watchdog_selftest")

_PKG = os.path.dirname(os.path.abspath(__file__))
_lib = None


class FaError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        msg = fa_status_string(status)
        if status == FA_ERR_CUDA:
            msg += f" ({fa_last_cuda_error()})"
        super().__init__(f"{what}: {msg}" if what else msg)


class _Options(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("grid_ctas", ctypes.c_int32),
                ("wait_limit_ns", ctypes.c_uint64)]


def library_path() -> str:
    return os.path.join(_PKG, "libfa_gb300.so")


def load_library():
    """Load ``libfa_gb300.so`` (built by ``build.py``); raise if absent."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is not built; run `python -m exact_attention_24_gb300.build`")
    try:  # let torch load its CUDA runtime first so both share one copy
        import torch  # noqa: F401
    except ImportError:
        pass
    lib = ctypes.CDLL(path)
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, f32, i32,
                           i32, vp]
    lib.fa_fwd.restype = i32
    lib.fa_fwd_window.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, f32, i32,
                                  i32, i32, vp]
    lib.fa_fwd_window.restype = i32
    lib.fa_fwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32,
                                  i32, f32, i32, i32, vp]
    lib.fa_fwd_varlen.restype = i32
    lib.fa_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, f32,
                                   i32, i32, i32, vp, ctypes.c_size_t, vp]
    lib.fa_fwd_splitkv.restype = i32
    lib.fa_fwd_splitkv_workspace_size.argtypes = [i32, i32, i32, i32, i32]
    lib.fa_fwd_splitkv_workspace_size.restype = ctypes.c_size_t
    lib.fa_fwd_splitkv_noalloc.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, f32,
                                           i32, i32, i32, vp]
    lib.fa_fwd_splitkv_noalloc.restype = i32
    lib.fa_fwd_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, f32,
                                i32, i32, i32, vp]
    lib.fa_fwd_host.restype = i32
    lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, f32, i32,
                           i32, vp, ctypes.c_size_t, vp]
    lib.fa_bwd.restype = i32
    lib.fa_bwd_workspace_size.argtypes = [i32, i32, i32]
    lib.fa_bwd_workspace_size.restype = ctypes.c_size_t
    lib.fa_bwd_window.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, f32, i32,
                                  i32, i32, vp, ctypes.c_size_t, vp]
    lib.fa_bwd_window.restype = i32
    lib.fa_bwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                  f32, i32, i32, vp, ctypes.c_size_t, vp]
    lib.fa_bwd_varlen.restype = i32
    lib.fa_bwd_varlen_workspace_size.argtypes = [i32, i32]
    lib.fa_bwd_varlen_workspace_size.restype = ctypes.c_size_t
    lib.fa_check_device_error.argtypes = [vp]
    lib.fa_check_device_error.restype = i32
    lib.fa_status_string.argtypes = [i32]
    lib.fa_status_string.restype = ctypes.c_char_p
    lib.fa_last_cuda_error.argtypes = []
    lib.fa_last_cuda_error.restype = ctypes.c_char_p
    lib.fa_set_options.argtypes = [ctypes.POINTER(_Options)]
    lib.fa_set_options.restype = i32
    lib.fa_get_options.argtypes = [ctypes.POINTER(_Options)]
    lib.fa_get_options.restype = i32
    lib.fa_watchdog_selftest.argtypes = [ctypes.c_uint64, vp]
    lib.fa_watchdog_selftest.restype = i32
    _lib = lib
    return lib


def _ptr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream(s) -> int:
    if s is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(s, int):
        return s
    return int(s.cuda_stream)


def fa_status_string(status: int) -> str:
    return load_library().fa_status_string(int(status)).decode()


def fa_last_cuda_error() -> str:
    return load_library().fa_last_cuda_error().decode()


def fa_fwd(Q, K, V, O, L, B, H, N, D, scale, causal, dtype, stream=None) -> int:
    return load_library().fa_fwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(L),
                                 int(B), int(H), int(N), int(D), float(scale),
                                 int(causal), int(dtype), _stream(stream))


def fa_fwd_window(Q, K, V, O, L, B, H, N, D, scale, window_left, window_right, dtype,
                  stream=None) -> int:
    return load_library().fa_fwd_window(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(L),
                                        int(B), int(H), int(N), int(D), float(scale),
                                        int(window_left), int(window_right), int(dtype),
                                        _stream(stream))


def fa_fwd_varlen(Q, K, V, O, L, cu_seqlens, num_seqs, total_tokens,
                  max_seqlen, H, D, scale, causal, dtype, stream=None) -> int:
    return load_library().fa_fwd_varlen(
        _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(L), _ptr(cu_seqlens),
        int(num_seqs), int(total_tokens), int(max_seqlen), int(H), int(D),
        float(scale), int(causal), int(dtype), _stream(stream))


def fa_fwd_splitkv(Q, K, V, O, L, B, H, N, D, scale, causal, dtype, num_splits,
                   workspace, workspace_bytes, stream=None) -> int:
    return load_library().fa_fwd_splitkv(
        _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(L), int(B), int(H), int(N), int(D),
        float(scale), int(causal), int(dtype), int(num_splits), _ptr(workspace),
        int(workspace_bytes), _stream(stream))


def fa_fwd_host(Qh, Kh, Vh, Oh, Lh, Qd, Kd, Vd, Od, Ld, B, H, N, D, scale, causal, dtype,
                chunks, stream=None) -> int:
    """Forward pass on HOST tensors (pinned for overlap) through caller-owned
    device staging buffers, copies overlapped with the kernels of
    neighbouring runs of ``chunks`` (see include/fa.h)."""
    return load_library().fa_fwd_host(
        _ptr(Qh), _ptr(Kh), _ptr(Vh), _ptr(Oh), _ptr(Lh), _ptr(Qd), _ptr(Kd), _ptr(Vd), _ptr(Od),
        _ptr(Ld), int(B), int(H), int(N), int(D), float(scale), int(causal), int(dtype),
        int(chunks), _stream(stream))


def fa_fwd_splitkv_noalloc(Q, K, V, O, L, B, H, N, D, scale, causal, dtype, num_splits,
                           stream=None) -> int:
    """Split-key forward pass that allocates nothing: for callers that may
    not allocate device memory (see include/fa.h).  Partials go to the
    library's fixed scratch array (FA_NOALLOC_SCRATCH_BYTES)."""
    return load_library().fa_fwd_splitkv_noalloc(
        _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(L), int(B), int(H), int(N), int(D),
        float(scale), int(causal), int(dtype), int(num_splits), _stream(stream))


FA_NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024


def fa_fwd_splitkv_workspace_size(B, H, N, D, num_splits) -> int:
    return int(load_library().fa_fwd_splitkv_workspace_size(int(B), int(H), int(N), int(D),
                                                            int(num_splits)))


def fa_bwd(Q, K, V, O, dO, L, dQ, dK, dV, B, H, N, D, scale, causal, dtype, workspace,
           workspace_bytes, stream=None) -> int:
    return load_library().fa_bwd(
        _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(L), _ptr(dQ), _ptr(dK), _ptr(dV),
        int(B), int(H), int(N), int(D), float(scale), int(causal), int(dtype), _ptr(workspace),
        int(workspace_bytes), _stream(stream))


def fa_bwd_workspace_size(B, H, N) -> int:
    return int(load_library().fa_bwd_workspace_size(int(B), int(H), int(N)))


def fa_bwd_window(Q, K, V, O, dO, L, dQ, dK, dV, B, H, N, D, scale, window_left, window_right,
                  dtype, workspace, workspace_bytes, stream=None) -> int:
    return load_library().fa_bwd_window(
        _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(L), _ptr(dQ), _ptr(dK), _ptr(dV),
        int(B), int(H), int(N), int(D), float(scale), int(window_left), int(window_right),
        int(dtype), _ptr(workspace), int(workspace_bytes), _stream(stream))


def fa_bwd_varlen(Q, K, V, O, dO, L, dQ, dK, dV, cu_seqlens, num_seqs, total_tokens, max_seqlen,
                  H, D, scale, causal, dtype, workspace, workspace_bytes, stream=None) -> int:
    return load_library().fa_bwd_varlen(
        _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(L), _ptr(dQ), _ptr(dK), _ptr(dV),
        _ptr(cu_seqlens), int(num_seqs), int(total_tokens), int(max_seqlen), int(H), int(D),
        float(scale), int(causal), int(dtype), _ptr(workspace), int(workspace_bytes),
        _stream(stream))


def fa_bwd_varlen_workspace_size(total_tokens, H) -> int:
    return int(load_library().fa_bwd_varlen_workspace_size(int(total_tokens), int(H)))


def fa_check_device_error(stream=None) -> int:
    return load_library().fa_check_device_error(_stream(stream))


def fa_set_options(kernel=FA_KERNEL_AUTO, grid_ctas=0, wait_limit_ns=0) -> int:
    o = _Options(int(kernel), int(grid_ctas), int(wait_limit_ns))
    return load_library().fa_set_options(ctypes.byref(o))


def fa_get_options() -> dict:
    o = _Options()
    st = load_library().fa_get_options(ctypes.byref(o))
    if st != FA_OK:
        raise FaError(st, "fa_get_options")
    return {"kernel": o.kernel, "grid_ctas": o.grid_ctas,
            "wait_limit_ns": o.wait_limit_ns}


def fa_watchdog_selftest(limit_ns: int, stream=None) -> int:
    return load_library().fa_watchdog_selftest(int(limit_ns), _stream(stream))


# ------------------------------------------------------------ convenience --
def _dtype_code(q, out_dtype):
    import torch
    if q.dtype == torch.float32:
        if out_dtype not in (None, torch.float32):
            raise ValueError("float32 inputs produce a float32 O")
        return FA_F32, torch.float32
    if q.dtype == torch.bfloat16:
        if out_dtype in (None, torch.bfloat16):
            return FA_BF16, torch.bfloat16
        if out_dtype == torch.float32:
            return FA_BF16_OUT_F32, torch.float32
    raise ValueError(f"unsupported dtypes {q.dtype} -> {out_dtype}")


def attention(q, k, v, causal: bool = False, scale: float | None = None,
              out_dtype=None, stream=None, num_splits: int | None = None):
    """O, L for ``[B, H, N, D]`` CUDA tensors (contiguous, same dtype).

    ``num_splits`` (bf16 only) selects the split-key path: an int >= 1, or 0
    for the automatic choice; the workspace is allocated here with torch."""
    import torch
    B, H, N, D = q.shape
    code, odt = _dtype_code(q, out_dtype)
    if scale is None:
        scale = float(torch.tensor(1.0 / math.sqrt(D), dtype=torch.float32))
    O = torch.empty((B, H, N, D), dtype=odt, device=q.device)
    L = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if num_splits is None:
        st = fa_fwd(q, k, v, O, L, B, H, N, D, scale, int(causal), code, stream)
    else:
        nbytes = fa_fwd_splitkv_workspace_size(B, H, N, D, num_splits)
        ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
        st = fa_fwd_splitkv(q, k, v, O, L, B, H, N, D, scale, int(causal), code,
                            num_splits, ws, nbytes, stream)
    if st != FA_OK:
        raise FaError(st, "fa_fwd" if num_splits is None else "fa_fwd_splitkv")
    return O, L


def attention_bwd(q, k, v, o, do, lse, causal: bool = False, scale: float | None = None,
                  out_dtype=None, stream=None):
    """dQ, dK, dV for ``[B, H, N, D]`` CUDA tensors, given the forward
    pass's O and L (``attention``'s outputs) and dO; the workspace is
    allocated here with torch."""
    import torch
    B, H, N, D = q.shape
    code, odt = _dtype_code(q, out_dtype)
    if scale is None:
        scale = float(torch.tensor(1.0 / math.sqrt(D), dtype=torch.float32))
    grads = [torch.empty((B, H, N, D), dtype=odt, device=q.device) for _ in range(3)]
    nbytes = fa_bwd_workspace_size(B, H, N)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    st = fa_bwd(q, k, v, o, do, lse, *grads, B, H, N, D, scale, int(causal), code, ws, nbytes,
                stream)
    if st != FA_OK:
        raise FaError(st, "fa_bwd")
    return tuple(grads)


def attention_varlen(q, k, v, cu_seqlens, max_seqlen: int, causal: bool = False,
                     scale: float | None = None, out_dtype=None, stream=None):
    """O ``[total, H, D]``, L ``[H, total]`` for a packed batch."""
    import torch
    total, H, D = q.shape
    code, odt = _dtype_code(q, out_dtype)
    if scale is None:
        scale = float(torch.tensor(1.0 / math.sqrt(D), dtype=torch.float32))
    O = torch.empty((total, H, D), dtype=odt, device=q.device)
    L = torch.empty((H, total), dtype=torch.float32, device=q.device)
    st = fa_fwd_varlen(q, k, v, O, L, cu_seqlens, cu_seqlens.numel() - 1,
                       total, max_seqlen, H, D, scale, int(causal), code, stream)
    if st != FA_OK:
        raise FaError(st, "fa_fwd_varlen")
    return O, L
