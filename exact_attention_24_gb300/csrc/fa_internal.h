// Internal host-side interface between the C-ABI layer (fa_api.cu) and the
// kernel launchers (fa_simt.cu, fa_tc.cu).  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/fa.h"

// Device error word layout: bits 31..24 = fa_status code, bits 15..0 = the
// site that recorded it (first writer wins).
#define FA_ERRWORD(code, site) ((((uint32_t)(code)) << 24) | ((uint32_t)(site) & 0xffffu))

struct FaProblem {
    const void *q;
    const void *k;
    const void *v;
    void *o;
    float *lse;
    const int32_t *cu_seqlens;  // null for a dense batch
    int varlen;
    int heads;        // H
    int units_bh;     // dense: B*H; varlen: num_seqs*H
    int num_seqs;     // varlen only
    int n;            // dense: N; varlen: max_seqlen
    int64_t total;    // dense: N (per-head L stride); varlen: total tokens
    int D;
    float scale;
    int causal;
    int wl, wr;       // key j visible to row i iff i - wl <= j <= i + wr (< 0: unbounded)
    int dtype;        // fa_dtype
    uint32_t *err;    // device error word
    int grid_ctas;    // 0 = one per SM
    uint64_t wait_limit_ns;
    int num_splits;   // split-key mode when > 1 (dense bf16 only)
    void *workspace;  // split-key partials (caller-owned device memory)
    size_t workspace_bytes;
    cudaStream_t stream;
};

// The backward pass (dense batch).  Row statistic delta = rowsum(dO * O)
// lives in the caller's workspace.
struct FaBwdProblem {
    const void *q, *k, *v, *o, *dout;
    const float *lse;
    void *dq, *dk, *dv;
    float *delta;     // float32 workspace, laid out like L
    const int32_t *cu_seqlens;  // null for a dense batch
    int varlen;
    int heads;        // H
    int num_seqs;     // varlen only
    int64_t total;    // varlen: total tokens (L / delta are [H, total])
    int units_bh;     // dense: B*H; varlen: num_seqs*H
    int n;            // dense: N; varlen: max_seqlen
    int D;
    float scale;
    int causal;
    int wl, wr;       // key j visible to row i iff i - wl <= j <= i + wr (< 0: unbounded)
    int dtype;        // fa_dtype
    uint32_t *err;
    int grid_ctas;
    uint64_t wait_limit_ns;
    cudaStream_t stream;
};

// Record `e` as the calling thread's last CUDA failure (see
// fa_last_cuda_error) and clear the runtime's sticky-free last error.
// Returns FA_ERR_CUDA so launchers can `return fa_cuda_fail(e);`.
fa_status fa_cuda_fail(cudaError_t e);

// Run `setup` (kernel attributes: dynamic shared memory and the like) once
// per device and kernel instantiation; `done` is that instantiation's mask
// of devices already set up.  Launches after the first then make no runtime
// calls besides the launch itself, so they can also be captured in a CUDA
// graph.  Returns the first failure of `setup`, which is retried next time.
template <typename F>
inline fa_status fa_once_per_device(std::atomic<uint64_t> &done, F &&setup) {
    int dev = 0;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fa_cuda_fail(e);
    const uint64_t bit = dev >= 0 && dev < 64 ? (uint64_t)1 << dev : 0;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return FA_OK;
    const fa_status st = setup();
    if (st == FA_OK && bit) done.fetch_or(bit, std::memory_order_release);
    return st;
}

// Streaming multiprocessors of the current device, cached per device; 0
// (with the failure recorded) if the device cannot be queried.
inline int fa_num_sms() {
    static std::atomic<int> cached[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64) {
        fa_cuda_fail(e != cudaSuccess ? e : cudaErrorInvalidDevice);
        return 0;
    }
    int sms = cached[dev].load(std::memory_order_relaxed);
    if (sms > 0) return sms;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) {
        fa_cuda_fail(e);
        return 0;
    }
    cached[dev].store(sms, std::memory_order_relaxed);
    return sms;
}

fa_status fa_launch_simt(const FaProblem &p);
// Backward pass: delta = rowsum(dO * O), then the FFMA or tensor-core
// gradient kernels (each launcher runs the delta kernel itself).
fa_status fa_launch_bwd_delta(const FaBwdProblem &p);
fa_status fa_launch_bwd_simt(const FaBwdProblem &p);
fa_status fa_launch_bwd_tc(const FaBwdProblem &p);
fa_status fa_launch_tc(const FaProblem &p);

// Split-key planning for the tensor-core kernel: the number of key-range
// splits used for `requested` (0 = automatic: enough work items to cover the
// SMs) and the workspace bytes they need.  Returns false if the device
// cannot be queried.
bool fa_tc_split_plan(int units_bh, int n, int D, int requested, int &splits, size_t &bytes);
fa_status fa_launch_watchdog_selftest(uint32_t *err, uint64_t limit_ns,
                                      cudaStream_t stream);
