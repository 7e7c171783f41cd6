// Internal host-side interface between the C-ABI layer (fa_api.cu) and the
// kernel launchers (fa_simt.cu, fa_tc.cu).  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

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

// Unique id of the CUDA context current on the calling thread -- the one the
// runtime's next call uses -- or 0 if there is none yet (or the driver cannot
// say).  Device addresses of module globals and kernel attributes belong to
// a context, not to a device number: a context made after cudaDeviceReset,
// or a host program's own driver-API context, loads this library's module
// afresh.  Every cache of such values is keyed by this id.
uint64_t fa_context_id();

// A small set of context ids (see fa_context_id), thread-safe.  When full,
// the oldest entry makes room: a forgotten context only repeats its set-up.
struct FaCtxSet {
    static constexpr int kCap = 16;
    std::mutex mu;
    uint64_t ids[kCap] = {};
    int next = 0;
    bool has(uint64_t id) {
        std::lock_guard<std::mutex> lk(mu);
        for (uint64_t x : ids)
            if (x == id) return true;
        return false;
    }
    void add(uint64_t id) {
        std::lock_guard<std::mutex> lk(mu);
        for (uint64_t x : ids)
            if (x == id) return;
        ids[next] = id;
        next = (next + 1) % kCap;
    }
};

// Run `setup` (kernel attributes: dynamic shared memory and the like) once
// per CUDA context and kernel instantiation; `done` is that instantiation's
// set of contexts already set up.  Launches after the first then make no
// runtime calls besides the launch itself, so they can also be captured in a
// CUDA graph.  Returns the first failure of `setup`, which is retried next
// time.
template <typename F>
inline fa_status fa_once_per_context(FaCtxSet &done, F &&setup) {
    const uint64_t id = fa_context_id();
    if (id && done.has(id)) return FA_OK;
    const fa_status st = setup();  // its runtime calls create the context if need be
    if (st == FA_OK) {
        const uint64_t now = id ? id : fa_context_id();
        if (now) done.add(now);
    }
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
// What the tensor-core launchers accept, decided on the host without any
// CUDA call: FA_OK, or FA_ERR_UNSUPPORTED for a dtype, head dimension, mode
// or size they do not take.
fa_status fa_tc_supports(const FaProblem &p);
fa_status fa_bwd_tc_supports(const FaBwdProblem &p);

// Split-key planning for the tensor-core kernel: the number of key-range
// splits used for `requested` (0 = automatic: enough work items to cover the
// SMs) and the workspace bytes they need.  Returns false if the device
// cannot be queried.
bool fa_tc_split_plan(int units_bh, int n, int D, int requested, int &splits, size_t &bytes);
fa_status fa_launch_watchdog_selftest(uint32_t *err, uint64_t limit_ns,
                                      cudaStream_t stream);
