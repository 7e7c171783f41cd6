// C-ABI layer: argument validation, kernel selection, the device error word
// and the watchdog self-test.  Declarations and contracts live in
// include/fa.h.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <mutex>

#include "device_common.cuh"
#include "fa_internal.h"

// Module-global device error word (see FA_ERRWORD).  Kernels receive its
// address as a plain pointer so every translation unit can report into it.
static __device__ uint32_t g_fa_error_word;

namespace {

fa_options g_opts = {FA_KERNEL_AUTO, 0, 0};
constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;  // 2 s

// A small table from CUDA context id (fa_context_id) to a value that
// belongs to that context; thread-safe.  When full, the oldest entry makes
// room (its context only repeats the lookup).
template <typename T>
struct CtxTable {
    static constexpr int kCap = 16;
    std::mutex mu;
    uint64_t ids[kCap] = {};
    T vals[kCap] = {};
    int next = 0;
    bool get(uint64_t id, T &out) {
        std::lock_guard<std::mutex> lk(mu);
        for (int i = 0; i < kCap; ++i)
            if (id && ids[i] == id) {
                out = vals[i];
                return true;
            }
        return false;
    }
    void put(uint64_t id, const T &v) {
        if (!id) return;
        std::lock_guard<std::mutex> lk(mu);
        ids[next] = id;
        vals[next] = v;
        next = (next + 1) % kCap;
    }
};

CtxTable<uint32_t *> g_err_addr;

// Device address of the error word in the current context.  In host code
// the symbol names a host-side stand-in, so the runtime is asked for the
// address (which also creates the context if none is current yet), once per
// context.
uint32_t *err_word() {
    const uint64_t id = fa_context_id();
    uint32_t *addr = nullptr;
    if (g_err_addr.get(id, addr)) return addr;
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_fa_error_word);
    if (e != cudaSuccess) {
        fa_cuda_fail(e);
        return nullptr;
    }
    g_err_addr.put(id ? id : fa_context_id(), static_cast<uint32_t *>(p));
    return static_cast<uint32_t *>(p);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

// fa_fwd_host's copy streams and run events, created in a context on its
// first call there and kept for the process; g_pipe_mu also serialises the
// enqueueing.
constexpr int kMaxHostChunks = 64;
struct HostPipe {
    uint64_t ctx = 0;
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start = nullptr, end = nullptr;
    cudaEvent_t landed[kMaxHostChunks], computed[kMaxHostChunks];
};
constexpr int kMaxPipes = 16;
HostPipe g_pipes[kMaxPipes];
int g_pipes_used = 0;
std::mutex g_pipe_mu;

// The current context's pipe (g_pipe_mu held), or null after recording the
// failure.
HostPipe *host_pipe() {
    // the error word's lookup makes sure a context is current
    if (!err_word()) return nullptr;
    const uint64_t id = fa_context_id();
    if (!id) {
        fa_cuda_fail(cudaErrorDeviceUninitialized);
        return nullptr;
    }
    cudaError_t e = cudaSuccess;
    for (int i = 0; i < g_pipes_used; ++i)
        if (g_pipes[i].ctx == id) return &g_pipes[i];
    if (g_pipes_used == kMaxPipes) {
        fa_cuda_fail(cudaErrorNotSupported);
        return nullptr;
    }
    HostPipe hp;
    const unsigned ev = cudaEventDisableTiming;
    e = cudaStreamCreateWithFlags(&hp.in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&hp.out, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.start, ev);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.end, ev);
    for (int i = 0; e == cudaSuccess && i < kMaxHostChunks; ++i) {
        e = cudaEventCreateWithFlags(&hp.landed[i], ev);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.computed[i], ev);
    }
    if (e != cudaSuccess) {  // partial creations are kept and retried no further
        fa_cuda_fail(e);
        return nullptr;
    }
    hp.ctx = id;
    g_pipes[g_pipes_used] = hp;
    return &g_pipes[g_pipes_used++];
}

size_t in_bytes(int dtype) { return dtype == FA_F32 ? 4 : 2; }
size_t out_bytes(int dtype) { return dtype == FA_BF16 ? 2 : 4; }

// Shared checks of the two entry points.  `tokens` = rows per head summed
// over the batch (B*N, or total_tokens).
fa_status check_common(const void *Q, const void *K, const void *V, void *O, float *L,
                       int64_t heads, int64_t tokens, int D, float scale, int causal,
                       fa_dtype dtype) {
    if (D <= 0 || heads < 0 || tokens < 0) return FA_ERR_INVALID_ARG;
    if (dtype != FA_F32 && dtype != FA_BF16 && dtype != FA_BF16_OUT_F32)
        return FA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    if (!isfinite(scale)) return FA_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
    if (tokens > INT32_MAX || heads > INT32_MAX) return FA_ERR_UNSUPPORTED;
    const int64_t elems = heads * tokens * D;  // < 2^31 * 2^31 * 128 fits
    if (elems == 0) return FA_OK;
    if (!Q || !K || !V || !O || !L) return FA_ERR_INVALID_ARG;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(L))
        return FA_ERR_INVALID_ARG;
    const size_t ni = (size_t)elems * in_bytes(dtype);
    const size_t no = (size_t)elems * out_bytes(dtype);
    const size_t nl = (size_t)(heads * tokens) * sizeof(float);
    const void *ins[3] = {Q, K, V};
    for (const void *x : ins)
        if (overlaps(O, no, x, ni) || overlaps(L, nl, x, ni)) return FA_ERR_INVALID_ARG;
    if (overlaps(O, no, L, nl)) return FA_ERR_INVALID_ARG;
    return FA_OK;
}

// Kernel choice.  bf16 runs on the tensor-core kernel: a bf16 case that
// kernel cannot take is reported to the caller as FA_ERR_UNSUPPORTED, before
// any CUDA call, and never handed to the FFMA kernel in its place.  The FFMA
// kernel serves float32, and bf16 only when the caller asks for it
// (FA_KERNEL_SIMT).
fa_status dispatch(FaProblem &p) {
    const bool bf16 = p.dtype != FA_F32;
    const bool simt = g_opts.kernel == FA_KERNEL_SIMT || (g_opts.kernel == FA_KERNEL_AUTO && !bf16);
    if (!simt) {
        if (!bf16) return FA_ERR_UNSUPPORTED;
        const fa_status st = fa_tc_supports(p);
        if (st != FA_OK) return st;
    }
    p.err = err_word();
    if (!p.err) return FA_ERR_CUDA;
    p.grid_ctas = g_opts.grid_ctas;
    p.wait_limit_ns = g_opts.wait_limit_ns ? g_opts.wait_limit_ns : kDefaultWaitLimitNs;
    return simt ? fa_launch_simt(p) : fa_launch_tc(p);
}

__global__ void watchdog_selftest_kernel(uint32_t *err, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        fa::mbar_init(fa::smem_u32(&bar), 1);
        fa::fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        fa::WaitCtx w{err, &abort_flag, limit_ns};
        // Nothing arrives on this barrier: the wait must run out and report.
        (void)fa::mbar_wait(fa::smem_u32(&bar), 0, w, 0xfeu);
    }
    __syncthreads();
}

}  // namespace

static thread_local cudaError_t t_last_cuda_error = cudaSuccess;

fa_status fa_cuda_fail(cudaError_t e) {
    t_last_cuda_error = e;
    cudaGetLastError();
    return FA_ERR_CUDA;
}

uint64_t fa_context_id() {
    // cuCtxGetCurrent / cuCtxGetId through the runtime's driver entry points
    // (the library links the runtime only), looked up once
    struct Fns {
        PFN_cuCtxGetCurrent_v4000 current = nullptr;
        PFN_cuCtxGetId_v12000 id = nullptr;
    };
    static const Fns fns = []() {
        Fns f;
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            f.current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            f.id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
        cudaGetLastError();
        return f;
    }();
    if (!fns.current || !fns.id) return 0;
    CUcontext ctx = nullptr;
    if (fns.current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    unsigned long long id = 0;
    if (fns.id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

fa_status fa_launch_watchdog_selftest(uint32_t *err, uint64_t limit_ns, cudaStream_t s) {
    watchdog_selftest_kernel<<<1, 32, 0, s>>>(err, limit_ns);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? FA_OK : fa_cuda_fail(e);
}

extern "C" {

static fa_status fwd_dense(const void *Q, const void *K, const void *V, void *O, float *L, int B,
                           int H, int N, int D, float scale, int causal, int wl, int wr,
                           fa_dtype dtype, fa_stream_t stream) {
    if (B < 0 || H < 0 || N < 0) return FA_ERR_INVALID_ARG;
    const int64_t heads = (int64_t)B * H;
    fa_status st = check_common(Q, K, V, O, L, heads, N, D, scale, causal, dtype);
    if (st != FA_OK) return st;
    if (heads == 0 || N == 0) return FA_OK;
    FaProblem p{};
    p.q = Q;
    p.k = K;
    p.v = V;
    p.o = O;
    p.lse = L;
    p.cu_seqlens = nullptr;
    p.varlen = 0;
    p.heads = H;
    p.units_bh = (int)heads;
    p.num_seqs = 0;
    p.n = N;
    p.total = N;
    p.D = D;
    p.scale = scale;
    p.causal = causal;
    p.wl = wl;
    p.wr = wr;
    p.dtype = dtype;
    p.stream = static_cast<cudaStream_t>(stream);
    return dispatch(p);
}

fa_status fa_fwd(const void *Q, const void *K, const void *V, void *O, float *L, int B, int H,
                 int N, int D, float scale, int causal, fa_dtype dtype, fa_stream_t stream) {
    return fwd_dense(Q, K, V, O, L, B, H, N, D, scale, causal, -1, causal ? 0 : -1, dtype, stream);
}

fa_status fa_fwd_host(const void *Qh, const void *Kh, const void *Vh, void *Oh, float *Lh, void *Qd,
                      void *Kd, void *Vd, void *Od, float *Ld, int B, int H, int N, int D, float scale,
                      int causal, fa_dtype dtype, int chunks, fa_stream_t stream) {
    if (chunks < 1 || chunks > kMaxHostChunks || B < 0 || H < 0 || N < 0) return FA_ERR_INVALID_ARG;
    const int64_t units = (int64_t)B * H;
    fa_status st = check_common(Qd, Kd, Vd, Od, Ld, units, N, D, scale, causal, dtype);
    if (st != FA_OK) return st;
    if (units == 0 || N == 0) return FA_OK;
    if (!Qh || !Kh || !Vh || !Oh || !Lh) return FA_ERR_INVALID_ARG;
    // runs of whole problems; boundaries on multiples of g keep each run's L
    // slice (u0 * N floats in) 16-byte aligned
    const int64_t g = N % 4 == 0 ? 1 : (N % 2 == 0 ? 2 : 4);
    const int64_t blocks = (units + g - 1) / g;
    const int runs = (int)(chunks < blocks ? chunks : blocks);
    const size_t row_in = (size_t)N * D * in_bytes(dtype), row_out = (size_t)N * D * out_bytes(dtype);
    const size_t row_l = (size_t)N * sizeof(float);
    std::lock_guard<std::mutex> lk(g_pipe_mu);
    HostPipe *hp = host_pipe();
    if (!hp) return FA_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaEventRecord(hp->start, s);  // earlier work on `stream` first
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->in, hp->start, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->out, hp->start, 0);
    if (e != cudaSuccess) return fa_cuda_fail(e);
    for (int c = 0; c < runs && st == FA_OK; ++c) {
        const int64_t u0 = blocks * c / runs * g, u1 = std::min(units, blocks * (c + 1) / runs * g);
        const size_t n = (size_t)(u1 - u0);
        auto dev = [&](void *base, size_t row) { return static_cast<char *>(base) + (size_t)u0 * row; };
        auto host = [&](const void *base, size_t row) {
            return static_cast<const char *>(base) + (size_t)u0 * row;
        };
        e = cudaMemcpyAsync(dev(Qd, row_in), host(Qh, row_in), n * row_in, cudaMemcpyHostToDevice, hp->in);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(dev(Kd, row_in), host(Kh, row_in), n * row_in, cudaMemcpyHostToDevice, hp->in);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(dev(Vd, row_in), host(Vh, row_in), n * row_in, cudaMemcpyHostToDevice, hp->in);
        if (e == cudaSuccess) e = cudaEventRecord(hp->landed[c], hp->in);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s, hp->landed[c], 0);
        if (e != cudaSuccess) {
            st = fa_cuda_fail(e);
            break;
        }
        st = fwd_dense(dev(Qd, row_in), dev(Kd, row_in), dev(Vd, row_in), dev(Od, row_out),
                       reinterpret_cast<float *>(dev(Ld, row_l)), 1, (int)n, N, D, scale, causal, -1,
                       causal ? 0 : -1, dtype, stream);
        if (st != FA_OK) break;
        e = cudaEventRecord(hp->computed[c], s);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->out, hp->computed[c], 0);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(static_cast<char *>(Oh) + (size_t)u0 * row_out, dev(Od, row_out), n * row_out,
                                cudaMemcpyDeviceToHost, hp->out);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(reinterpret_cast<char *>(Lh) + (size_t)u0 * row_l, dev(Ld, row_l), n * row_l,
                                cudaMemcpyDeviceToHost, hp->out);
        if (e != cudaSuccess) st = fa_cuda_fail(e);
    }
    // `stream` completes after the last copy in either direction, also on a
    // failure, so no copy outlives the caller's view of the buffers
    cudaError_t e2 = cudaEventRecord(hp->end, hp->out);
    if (e2 == cudaSuccess) e2 = cudaStreamWaitEvent(s, hp->end, 0);
    if (e2 == cudaSuccess) e2 = cudaEventRecord(hp->start, hp->in);
    if (e2 == cudaSuccess) e2 = cudaStreamWaitEvent(s, hp->start, 0);
    if (e2 != cudaSuccess && st == FA_OK) st = fa_cuda_fail(e2);
    return st;
}

fa_status fa_fwd_window(const void *Q, const void *K, const void *V, void *O, float *L, int B,
                        int H, int N, int D, float scale, int window_left, int window_right,
                        fa_dtype dtype, fa_stream_t stream) {
    if (window_left < -1 || window_right < -1) return FA_ERR_INVALID_ARG;
    // (-1, 0) is the causal mask: the causal kernels skip the tiles above the diagonal
    const int causal = window_left < 0 && window_right == 0;
    return fwd_dense(Q, K, V, O, L, B, H, N, D, scale, causal, window_left, window_right, dtype, stream);
}

fa_status fa_fwd_varlen(const void *Q, const void *K, const void *V, void *O, float *L,
                        const int32_t *cu_seqlens, int num_seqs, int total_tokens,
                        int max_seqlen, int H, int D, float scale, int causal,
                        fa_dtype dtype, fa_stream_t stream) {
    if (num_seqs < 0 || total_tokens < 0 || max_seqlen < 0 || H < 0)
        return FA_ERR_INVALID_ARG;
    fa_status st = check_common(Q, K, V, O, L, H, total_tokens, D, scale, causal, dtype);
    if (st != FA_OK) return st;
    if (num_seqs == 0 || H == 0 || total_tokens == 0 || max_seqlen == 0) return FA_OK;
    if (!cu_seqlens || (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u))
        return FA_ERR_INVALID_ARG;
    if ((int64_t)num_seqs * H > INT32_MAX) return FA_ERR_UNSUPPORTED;
    FaProblem p{};
    p.q = Q;
    p.k = K;
    p.v = V;
    p.o = O;
    p.lse = L;
    p.cu_seqlens = cu_seqlens;
    p.varlen = 1;
    p.heads = H;
    p.units_bh = num_seqs * H;
    p.num_seqs = num_seqs;
    p.n = max_seqlen;
    p.total = total_tokens;
    p.D = D;
    p.scale = scale;
    p.causal = causal;
    p.wl = -1;
    p.wr = causal ? 0 : -1;
    p.dtype = dtype;
    p.stream = static_cast<cudaStream_t>(stream);
    return dispatch(p);
}

fa_status fa_fwd_splitkv(const void *Q, const void *K, const void *V, void *O, float *L, int B,
                         int H, int N, int D, float scale, int causal, fa_dtype dtype,
                         int num_splits, void *workspace, size_t workspace_bytes,
                         fa_stream_t stream) {
    if (B < 0 || H < 0 || N < 0 || num_splits < 0 || num_splits > 64) return FA_ERR_INVALID_ARG;
    const int64_t heads = (int64_t)B * H;
    fa_status st = check_common(Q, K, V, O, L, heads, N, D, scale, causal, dtype);
    if (st != FA_OK) return st;
    if (dtype == FA_F32) return FA_ERR_UNSUPPORTED;
    if (heads == 0 || N == 0) return FA_OK;
    int splits = 1;
    size_t need = 0;
    if (!fa_tc_split_plan((int)heads, N, D, num_splits, splits, need)) return FA_ERR_CUDA;
    if (splits > 1) {
        if (!workspace || !aligned16(workspace) || workspace_bytes < need) return FA_ERR_INVALID_ARG;
        const void *ins[3] = {Q, K, V};
        const size_t ni = (size_t)heads * N * D * in_bytes(dtype);
        for (const void *x : ins)
            if (overlaps(workspace, need, x, ni)) return FA_ERR_INVALID_ARG;
        if (overlaps(workspace, need, O, (size_t)heads * N * D * out_bytes(dtype)) ||
            overlaps(workspace, need, L, (size_t)heads * N * sizeof(float)))
            return FA_ERR_INVALID_ARG;
    }
    FaProblem p{};
    p.q = Q;
    p.k = K;
    p.v = V;
    p.o = O;
    p.lse = L;
    p.heads = H;
    p.units_bh = (int)heads;
    p.n = N;
    p.total = N;
    p.D = D;
    p.scale = scale;
    p.causal = causal;
    p.wl = -1;
    p.wr = causal ? 0 : -1;
    p.dtype = dtype;
    p.num_splits = splits;
    p.workspace = workspace;
    p.workspace_bytes = workspace_bytes;
    p.stream = static_cast<cudaStream_t>(stream);
    p.err = err_word();
    if (!p.err) return FA_ERR_CUDA;
    p.grid_ctas = g_opts.grid_ctas;
    p.wait_limit_ns = g_opts.wait_limit_ns ? g_opts.wait_limit_ns : kDefaultWaitLimitNs;
    return fa_launch_tc(p);
}

size_t fa_fwd_splitkv_workspace_size(int B, int H, int N, int D, int num_splits) {
    if (B <= 0 || H <= 0 || N <= 0 || (D != 64 && D != 128) || num_splits < 0 || num_splits > 64)
        return 0;
    if ((int64_t)B * H > INT32_MAX) return 0;
    int splits = 1;
    size_t need = 0;
    if (!fa_tc_split_plan(B * H, N, D, num_splits, splits, need)) return 0;
    return need;
}

size_t fa_bwd_workspace_size(int B, int H, int N) {
    if (B <= 0 || H <= 0 || N <= 0) return 0;
    const size_t rows = (size_t)B * (size_t)H * (size_t)N;
    return (rows * sizeof(float) + 255) / 256 * 256;
}

// Checks shared by the backward entry points; `rows` = heads * tokens.
static fa_status check_bwd(const void *Q, const void *K, const void *V, const void *O, const void *dO,
                           const float *L, void *dQ, void *dK, void *dV, int64_t rows, int D,
                           float scale, int causal, fa_dtype dtype, void *workspace,
                           size_t workspace_bytes) {
    if (D <= 0) return FA_ERR_INVALID_ARG;
    if (dtype != FA_F32 && dtype != FA_BF16 && dtype != FA_BF16_OUT_F32) return FA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    if (!isfinite(scale)) return FA_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
    if (rows == 0) return FA_OK;
    const void *ins[6] = {Q, K, V, O, dO, L};
    void *outs[3] = {dQ, dK, dV};
    for (const void *x : ins)
        if (!x || !aligned16(x)) return FA_ERR_INVALID_ARG;
    for (const void *x : outs)
        if (!x || !aligned16(x)) return FA_ERR_INVALID_ARG;
    const size_t nw = (size_t)rows * sizeof(float);
    if (!workspace || !aligned16(workspace) || workspace_bytes < nw) return FA_ERR_INVALID_ARG;
    const size_t ni = (size_t)rows * D * in_bytes(dtype), no = (size_t)rows * D * out_bytes(dtype);
    const size_t in_sizes[6] = {ni, ni, ni, ni, ni, nw};
    for (int a = 0; a < 3; ++a) {
        for (int b = 0; b < 6; ++b)
            if (overlaps(outs[a], no, ins[b], in_sizes[b])) return FA_ERR_INVALID_ARG;
        for (int b = a + 1; b < 3; ++b)
            if (overlaps(outs[a], no, outs[b], no)) return FA_ERR_INVALID_ARG;
        if (overlaps(outs[a], no, workspace, nw)) return FA_ERR_INVALID_ARG;
    }
    for (int b = 0; b < 6; ++b)
        if (overlaps(workspace, nw, ins[b], in_sizes[b])) return FA_ERR_INVALID_ARG;
    return FA_OK;
}

// Kernel choice as in dispatch: bf16 gradients come from the tensor-core
// kernels or the call returns the reason they cannot, before any launch.
static fa_status run_bwd(FaBwdProblem &p) {
    const bool bf16 = p.dtype != FA_F32;
    const bool simt = g_opts.kernel == FA_KERNEL_SIMT || (g_opts.kernel == FA_KERNEL_AUTO && !bf16);
    if (!simt) {
        if (!bf16) return FA_ERR_UNSUPPORTED;
        const fa_status st = fa_bwd_tc_supports(p);
        if (st != FA_OK) return st;
    }
    p.err = err_word();
    if (!p.err) return FA_ERR_CUDA;
    p.grid_ctas = g_opts.grid_ctas;
    p.wait_limit_ns = g_opts.wait_limit_ns ? g_opts.wait_limit_ns : kDefaultWaitLimitNs;
    fa_status st = fa_launch_bwd_delta(p);
    if (st != FA_OK) return st;
    return simt ? fa_launch_bwd_simt(p) : fa_launch_bwd_tc(p);
}

fa_status fa_bwd(const void *Q, const void *K, const void *V, const void *O, const void *dO,
                 const float *L, void *dQ, void *dK, void *dV, int B, int H, int N, int D,
                 float scale, int causal, fa_dtype dtype, void *workspace,
                 size_t workspace_bytes, fa_stream_t stream) {
    if (B < 0 || H < 0 || N < 0) return FA_ERR_INVALID_ARG;
    const int64_t units = (int64_t)B * H;
    if (units > INT32_MAX || (int64_t)N > INT32_MAX / 2) return FA_ERR_UNSUPPORTED;
    const int64_t rows = units * N;
    fa_status st = check_bwd(Q, K, V, O, dO, L, dQ, dK, dV, rows, D, scale, causal, dtype,
                             workspace, workspace_bytes);
    if (st != FA_OK || rows == 0) return st;
    if (workspace_bytes < fa_bwd_workspace_size(B, H, N)) return FA_ERR_INVALID_ARG;
    FaBwdProblem p{};
    p.q = Q;
    p.k = K;
    p.v = V;
    p.o = O;
    p.dout = dO;
    p.lse = L;
    p.dq = dQ;
    p.dk = dK;
    p.dv = dV;
    p.delta = static_cast<float *>(workspace);
    p.heads = H;
    p.units_bh = (int)units;
    p.n = N;
    p.total = N;
    p.D = D;
    p.scale = scale;
    p.causal = causal;
    p.wl = -1;
    p.wr = causal ? 0 : -1;
    p.dtype = dtype;
    p.stream = static_cast<cudaStream_t>(stream);
    return run_bwd(p);
}

fa_status fa_bwd_window(const void *Q, const void *K, const void *V, const void *O, const void *dO,
                        const float *L, void *dQ, void *dK, void *dV, int B, int H, int N, int D,
                        float scale, int window_left, int window_right, fa_dtype dtype,
                        void *workspace, size_t workspace_bytes, fa_stream_t stream) {
    if (window_left < -1 || window_right < -1) return FA_ERR_INVALID_ARG;
    if (B < 0 || H < 0 || N < 0) return FA_ERR_INVALID_ARG;
    const int64_t units = (int64_t)B * H;
    if (units > INT32_MAX || (int64_t)N > INT32_MAX / 2) return FA_ERR_UNSUPPORTED;
    const int64_t rows = units * N;
    // (-1, 0) is the causal mask, (-1, -1) none: both run the plain kernels
    const int causal = window_left < 0 && window_right == 0;
    fa_status st = check_bwd(Q, K, V, O, dO, L, dQ, dK, dV, rows, D, scale, causal, dtype, workspace,
                             workspace_bytes);
    if (st != FA_OK || rows == 0) return st;
    if (workspace_bytes < fa_bwd_workspace_size(B, H, N)) return FA_ERR_INVALID_ARG;
    FaBwdProblem p{};
    p.q = Q;
    p.k = K;
    p.v = V;
    p.o = O;
    p.dout = dO;
    p.lse = L;
    p.dq = dQ;
    p.dk = dK;
    p.dv = dV;
    p.delta = static_cast<float *>(workspace);
    p.heads = H;
    p.units_bh = (int)units;
    p.n = N;
    p.total = N;
    p.D = D;
    p.scale = scale;
    p.causal = causal;
    p.wl = window_left;
    p.wr = window_right;
    p.dtype = dtype;
    p.stream = static_cast<cudaStream_t>(stream);
    return run_bwd(p);
}

size_t fa_bwd_varlen_workspace_size(int total_tokens, int H) {
    if (total_tokens <= 0 || H <= 0) return 0;
    return ((size_t)total_tokens * (size_t)H * sizeof(float) + 255) / 256 * 256;
}

fa_status fa_bwd_varlen(const void *Q, const void *K, const void *V, const void *O, const void *dO,
                        const float *L, void *dQ, void *dK, void *dV, const int32_t *cu_seqlens,
                        int num_seqs, int total_tokens, int max_seqlen, int H, int D, float scale,
                        int causal, fa_dtype dtype, void *workspace, size_t workspace_bytes,
                        fa_stream_t stream) {
    if (num_seqs < 0 || total_tokens < 0 || max_seqlen < 0 || H < 0) return FA_ERR_INVALID_ARG;
    const int64_t rows = (int64_t)total_tokens * H;
    fa_status st = check_bwd(Q, K, V, O, dO, L, dQ, dK, dV, rows, D, scale, causal, dtype,
                             workspace, workspace_bytes);
    if (st != FA_OK) return st;
    if (num_seqs == 0 || rows == 0 || max_seqlen == 0) return FA_OK;
    if (!cu_seqlens || (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u)) return FA_ERR_INVALID_ARG;
    if ((int64_t)num_seqs * H > INT32_MAX || max_seqlen > INT32_MAX / 2) return FA_ERR_UNSUPPORTED;
    FaBwdProblem p{};
    p.q = Q;
    p.k = K;
    p.v = V;
    p.o = O;
    p.dout = dO;
    p.lse = L;
    p.dq = dQ;
    p.dk = dK;
    p.dv = dV;
    p.delta = static_cast<float *>(workspace);
    p.cu_seqlens = cu_seqlens;
    p.varlen = 1;
    p.heads = H;
    p.num_seqs = num_seqs;
    p.units_bh = num_seqs * H;
    p.n = max_seqlen;
    p.total = total_tokens;
    p.D = D;
    p.scale = scale;
    p.causal = causal;
    p.wl = -1;
    p.wr = causal ? 0 : -1;
    p.dtype = dtype;
    p.stream = static_cast<cudaStream_t>(stream);
    return run_bwd(p);
}

fa_status fa_check_device_error(fa_stream_t stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t *err = err_word();
    if (!err) return FA_ERR_CUDA;
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return fa_cuda_fail(e);
    uint32_t word = 0;
    if ((e = cudaMemcpyAsync(&word, err, sizeof(word), cudaMemcpyDeviceToHost, s)) != cudaSuccess ||
        (e = cudaMemsetAsync(err, 0, sizeof(uint32_t), s)) != cudaSuccess ||
        (e = cudaStreamSynchronize(s)) != cudaSuccess)
        return fa_cuda_fail(e);
    return static_cast<fa_status>(word >> 24);
}

const char *fa_last_cuda_error(void) { return cudaGetErrorString(t_last_cuda_error); }

const char *fa_status_string(fa_status status) {
    switch (status) {
        case FA_OK: return "FA_OK: success";
        case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG: invalid argument";
        case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED: unsupported size or head dimension";
        case FA_ERR_CUDA: return "FA_ERR_CUDA: a CUDA call failed";
        case FA_ERR_DEVICE_TIMEOUT: return "FA_ERR_DEVICE_TIMEOUT: a device-side wait ran past its limit";
        default: return "unknown fa_status";
    }
}

fa_status fa_set_options(const fa_options *opts) {
    if (!opts) return FA_ERR_INVALID_ARG;
    if (opts->kernel < FA_KERNEL_AUTO || opts->kernel > FA_KERNEL_TC || opts->grid_ctas < 0)
        return FA_ERR_INVALID_ARG;
    g_opts = *opts;
    return FA_OK;
}

fa_status fa_get_options(fa_options *opts) {
    if (!opts) return FA_ERR_INVALID_ARG;
    *opts = g_opts;
    return FA_OK;
}

fa_status fa_watchdog_selftest(uint64_t limit_ns, fa_stream_t stream) {
    if (limit_ns == 0 || limit_ns > 1000000000ull) return FA_ERR_INVALID_ARG;
    uint32_t *err = err_word();
    if (!err) return FA_ERR_CUDA;
    return fa_launch_watchdog_selftest(err, limit_ns, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
