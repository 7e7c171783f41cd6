"""The library from plain C: a C program (tests/c_abi/abi_demo.c) built with
gcc against include/fa.h and the shared library, allocating its own device
memory with the CUDA runtime, runs fa_fwd and fa_bwd in float32 (the FFMA
kernels), and in a second mode fa_fwd on bf16 inputs on the tensor-core
kernel; its outputs are compared here with the float64 oracle.  No torch on
that path."""

import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import exact_attention_24_gb300 as fa
from exact_attention_24_gb300 import build as fa_build
from exact_attention_24_gb300.workloads import Workload, make_inputs
from helpers import assert_close
from oracle import attention_bwd_ref, attention_ref

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = "/usr/local/cuda"


def _compile(tmp_path):
    lib = fa_build.build()
    exe = str(tmp_path / "abi_demo")
    cmd = ["gcc", "-O2", "-o", exe, os.path.join(ROOT, "tests", "c_abi", "abi_demo.c"),
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
           lib, "-L", os.path.join(CUDA, "lib64"), "-lcudart",
           "-Wl,-rpath," + os.path.dirname(lib) + ":" + os.path.join(CUDA, "lib64")]
    subprocess.run(cmd, check=True, capture_output=True)
    return exe


def test_c_program_builds(tmp_path):
    """gcc compiles and links the C caller against the header and library."""
    if shutil.which("gcc") is None:
        pytest.skip("no gcc")
    assert os.path.exists(_compile(tmp_path))


@pytest.mark.gpu
def test_c_program_matches_oracle(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    exe = _compile(tmp_path)
    B, H, N, D, causal = 1, 2, 150, 64, True
    w = Workload("c_abi", B, H, N, D, "f32", causal, 5)
    q, k, v = make_inputs(w)
    do = make_inputs(Workload("c_abi_dO", B, H, N, D, "f32", causal, 6))[0]
    inp, out = tmp_path / "in.bin", tmp_path / "out.bin"
    np.concatenate([x.numpy().ravel() for x in (q, k, v, do)]).astype(np.float32).tofile(inp)
    r = subprocess.run([exe, str(inp), str(out), str(B), str(H), str(N), str(D), str(int(causal)),
                        repr(w.scale)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    got = np.fromfile(out, dtype=np.float32).astype(np.float64)
    e, rows = B * H * N * D, B * H * N
    O, L = got[:e].reshape(B, H, N, D), got[e:e + rows].reshape(B, H, N)
    dq, dk, dv = (got[e + rows + i * e: e + rows + (i + 1) * e].reshape(B, H, N, D) for i in range(3))
    ref_o, ref_l = attention_ref(q, k, v, w.scale, causal)
    assert np.max(np.abs(O - ref_o)) <= 1e-4 and np.max(np.abs(L - ref_l)) <= 1e-5
    for g, ref in zip((dq, dk, dv), attention_bwd_ref(q, k, v, do, w.scale, causal)[:3]):
        assert np.max(np.abs(g - ref)) <= 1e-4 * max(1.0, float(np.max(np.abs(ref))))


@pytest.mark.gpu
def test_c_program_tensor_core_bf16_matches_oracle(tmp_path):
    """bf16 inputs on the tensor-core kernel from C: fp32 O and bf16 O, each
    with L, against the oracle on the same bf16-rounded inputs."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    exe = _compile(tmp_path)
    B, H, N, D, causal = 2, 2, 333, 128, True
    w = Workload("c_abi_bf16", B, H, N, D, "bf16", causal, 9)
    q, k, v = make_inputs(w)      # bf16 values: exact in the float32 file
    inp, out = tmp_path / "in.bin", tmp_path / "out.bin"
    np.concatenate([x.float().numpy().ravel() for x in (q, k, v, q)]).astype(np.float32).tofile(inp)
    r = subprocess.run([exe, str(inp), str(out), str(B), str(H), str(N), str(D), str(int(causal)),
                        repr(w.scale), "bf16"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    got = np.fromfile(out, dtype=np.float32).astype(np.float64)
    e, rows = B * H * N * D, B * H * N
    o32, l1 = got[:e].reshape(B, H, N, D), got[e:e + rows].reshape(B, H, N)
    o16, l2 = got[e + rows:2 * e + rows].reshape(B, H, N, D), got[2 * e + rows:].reshape(B, H, N)
    ref_o, ref_l = attention_ref(q, k, v, w.scale, causal)
    assert_close(o32, l1, ref_o, ref_l, fa.FA_BF16_OUT_F32, "C caller, fp32 O")
    assert_close(o16, l2, ref_o, ref_l, fa.FA_BF16, "C caller, bf16 O")
