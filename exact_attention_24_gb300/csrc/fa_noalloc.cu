// fa_fwd_splitkv_noalloc: the split-key forward pass for callers that cannot
// allocate device memory themselves -- for example a plugin loaded into a
// host program that owns the whole device-memory budget, a latency-critical
// caller for which cudaMalloc / cudaFree (which can synchronise the device)
// are off limits, or plain C code that is handed only its input and output
// buffers.  Instead of a caller-provided workspace, the partial results live
// in one fixed scratch array in this file.
#include <cuda_runtime.h>

#include <mutex>

#include "fa_internal.h"

// The split-key partials of fa_fwd_splitkv_noalloc.  Every GPU that loads
// this library holds these FA_NOALLOC_SCRATCH_BYTES until the process exits.
// All calls share it: calls that overlap on the GPU (different streams, or
// different host threads) race on it.  Nothing in it needs to start at zero:
// each call reads only the partials it wrote itself.
static __device__ __align__(256) unsigned char g_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxContexts = 16;
uint64_t g_scratch_ctx[kMaxContexts];
void *g_scratch_addr[kMaxContexts];
int g_scratch_next = 0;
std::mutex g_scratch_mu;

// Device address of the scratch array in the current CUDA context.  In host
// code `g_noalloc_scratch` names a host-side stand-in, not device memory, so
// the runtime is asked for the address -- once per context, on the first
// call made with that context current -- and the address is what the kernels
// get.  The address belongs to the context, not to the device number: a
// context made later (after cudaDeviceReset, or a host program's own
// driver-API context) loads the module afresh and gets its own lookup.
fa_status scratch_address(void **out) {
    const uint64_t id = fa_context_id();
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    for (int i = 0; id && i < kMaxContexts; ++i)
        if (g_scratch_ctx[i] == id) {
            *out = g_scratch_addr[i];
            return FA_OK;
        }
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);  // creates the context if needed
    if (e != cudaSuccess) return fa_cuda_fail(e);
    const uint64_t now = id ? id : fa_context_id();
    if (now) {
        g_scratch_ctx[g_scratch_next] = now;
        g_scratch_addr[g_scratch_next] = p;
        g_scratch_next = (g_scratch_next + 1) % kMaxContexts;
    }
    *out = p;
    return FA_OK;
}

}  // namespace

extern "C" fa_status fa_fwd_splitkv_noalloc(const void *Q, const void *K, const void *V, void *O,
                                            float *L, int B, int H, int N, int D, float scale,
                                            int causal, fa_dtype dtype, int num_splits,
                                            fa_stream_t stream) {
    const size_t need = fa_fwd_splitkv_workspace_size(B, H, N, D, num_splits);
    if (need > (size_t)FA_NOALLOC_SCRATCH_BYTES) return FA_ERR_UNSUPPORTED;
    void *ws = nullptr;
    if (need > 0) {
        const fa_status st = scratch_address(&ws);
        if (st != FA_OK) return st;
    }
    // Argument checks (and the single-split case, which needs no scratch)
    // are those of fa_fwd_splitkv.
    return fa_fwd_splitkv(Q, K, V, O, L, B, H, N, D, scale, causal, dtype, num_splits, ws,
                          ws ? (size_t)FA_NOALLOC_SCRATCH_BYTES : 0, stream);
}
