"""Build the in-tree shared library ``libfa_gb300.so`` for sm_103a.

Each translation unit under ``csrc/`` is compiled by its own ``nvcc`` process
(in parallel), then linked against the CUDA toolkit's shared runtime (found
through an rpath).  The runtime loads the GPU driver lazily, so the library
loads on machines without one (the driver API entry point it needs,
``cuTensorMapEncodeTiled``, is looked up at run time through the runtime).

Usage: ``python -m exact_attention_24_gb300.build [--force] [--verbose]``.
"""

from __future__ import annotations

import concurrent.futures as cf
import glob
import hashlib
import os
import shutil
import subprocess
import sys

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG_DIR, "csrc")
ROOT = os.path.dirname(PKG_DIR)
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG_DIR, "_build")
LIB_NAME = "libfa_gb300.so"
LIB_PATH = os.path.join(PKG_DIR, LIB_NAME)

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-Xcompiler", "-fvisibility=hidden", f"-I{INCLUDE}"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"),
                 "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


# Sources that decide what one kernel family does, besides the shared
# headers, the ABI header and the API file (which picks kernels and launch
# parameters): a measurement of a family stays valid while these are unchanged.
KERNEL_SOURCES = {
    "fa_tc": ("fa_tc.cu",),
    "fa_simt": ("fa_simt.cu",),
    "fa_bwd": ("fa_bwd_tc.cu", "fa_bwd_simt.cu"),
}
_SHARED = ("device_common.cuh", "tc_common.cuh", "fa_internal.h", "fa_api.cu")


def _hash(paths) -> str:
    h = hashlib.sha256()
    for path in sorted(paths, key=os.path.basename):
        with open(path, "rb") as f:
            h.update(os.path.basename(path).encode())
            h.update(f.read())
    # the flags without the checkout's location, so that a copy of the tree
    # elsewhere (another machine) has the same digest
    h.update(" ".join(f.replace(INCLUDE, "<include>") for f in NVCC_FLAGS).encode())
    return h.hexdigest()[:16]


def _digest() -> str:
    """Digest of every source of the library (the build stamp)."""
    return _hash(glob.glob(os.path.join(CSRC, "*")) + glob.glob(os.path.join(INCLUDE, "*.h")))


def kernel_digest(kernel: str) -> str:
    """Digest of the sources one kernel family depends on (see KERNEL_SOURCES)."""
    names = KERNEL_SOURCES[kernel] + _SHARED
    return _hash([os.path.join(CSRC, n) for n in names] + glob.glob(os.path.join(INCLUDE, "*.h")))


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile (if sources changed) and return the library path."""
    stamp = os.path.join(BUILD_DIR, "stamp")
    digest = _digest()
    if (not force and os.path.exists(LIB_PATH) and os.path.exists(stamp)
            and open(stamp).read() == digest):
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    nvcc = _nvcc()

    def compile_one(src):
        obj = os.path.join(BUILD_DIR, os.path.basename(src) + ".o")
        cmd = [nvcc, *NVCC_FLAGS, "-c", src, "-o", obj]
        if verbose:
            cmd += ["-Xptxas", "-v"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            sys.stderr.write(r.stderr)
        return obj

    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = LIB_PATH + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", *objs, "-o", tmp,
           "-Xlinker", "-rpath=/usr/local/cuda/lib64"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    with open(stamp, "w") as f:
        f.write(digest)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="--verbose" in sys.argv))
