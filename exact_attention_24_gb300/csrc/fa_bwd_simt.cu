// FFMA (CUDA-core) backward pass, and the row statistic both backward paths
// share.
//
// The gradients of "FlashAttention -- for programmers, not researchers.",
// STAGE 5: the probabilities are never stored; every (query, key) entry is
// recomputed from Q, K and the forward pass's L as p = exp(scale q.k - L).
// With delta_i = rowsum(dO_i * O_i) (computed once per row by
// bwd_delta_kernel), the five contractions of the "FlashAttention" docs
// page, section "Application in Backward Pass (5 MMAs)", become per entry:
//     dV_j += p dO_i,  dp = dO_i . V_j,  ds = p (dp - delta_i),
//     dK_j += scale ds Q_i,  dQ_i += scale ds K_j.
//
// Two passes keep every sum in a fixed order (no atomics): the dK/dV pass
// gives each warp four keys and walks the query rows that can see them; the
// dQ pass gives each warp four query rows and walks their keys.  Within a
// warp, lane t holds columns t, t + 32, ... of every row it touches, and the
// two dot products per entry are warp shuffles.
//
// Serves FA_F32 (float32 throughout, accurate expf) and is the reference GPU
// path the tests run beside the tensor-core backward for bf16.
#include <cuda_bf16.h>
#include <math.h>

#include "device_common.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kWarps = 8;
constexpr int kPerWarp = 4;                  // keys (dK/dV pass) or rows (dQ pass) per warp
constexpr int kBlock = kWarps * kPerWarp;    // 32 keys or rows per CTA
constexpr int kTile = 32;                    // rows staged in shared memory per step

struct BwdParams {
    const void *q, *k, *v, *o, *dout;
    const float *lse, *delta;
    void *dq, *dk, *dv;
    const int32_t *cu;
    int varlen, heads, num_seqs;
    int64_t total;
    int n, D;
    float scale;
    int causal, wl, wr;
    uint32_t *err;
};

// One attention problem of the batch: (batch, head) of a dense batch or
// (sequence, head) of a packed one.  Row i of its Q (K, V, ...) starts at
// element elem0 + i * rstride; its L and delta at stat0 + i.
struct Head {
    int64_t elem0, rstride, stat0;
    int len;
};

__device__ __forceinline__ Head head_of(const BwdParams &p, int unit, int D) {
    Head h;
    if (!p.varlen) {
        h.elem0 = (int64_t)unit * p.n * D;
        h.rstride = D;
        h.stat0 = (int64_t)unit * p.n;
        h.len = p.n;
    } else {
        const int s = unit / p.heads, hh = unit % p.heads;
        int64_t start;
        int len;
        seq_bounds(p.cu, s, p.total, p.n, p.err, start, len);  // invalid: len = 0
        h.elem0 = (start * p.heads + hh) * D;
        h.rstride = (int64_t)p.heads * D;
        h.stat0 = (int64_t)hh * p.total + start;
        h.len = len;
    }
    return h;
}

__device__ __forceinline__ float ldf(const float *p) { return *p; }
__device__ __forceinline__ float ldf(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
__device__ __forceinline__ void stf(float *p, float x) { *p = x; }
__device__ __forceinline__ void stf(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

__device__ __forceinline__ float wsum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

__device__ __forceinline__ bool visible(int i, int j, const BwdParams &p) {
    if (p.causal && j > i) return false;
    if (p.wl >= 0 && j < i - p.wl) return false;
    if (p.wr >= 0 && j > i + p.wr) return false;
    return true;
}

// delta = sum_c dO[row, c] * O[row, c]; one warp per row.  Rows are taken
// in memory order; a packed batch ([total, H, D]) stores row t*H + h's
// statistic at h*total + t, like L.
template <typename T>
__global__ void __launch_bounds__(256) bwd_delta_kernel(const T *o, const T *dout, float *delta,
                                                        int64_t rows, int D, int heads, int64_t total) {
    // launched with programmatic stream serialization: the next kernel may
    // start its setup now; this one waits for the previous before reading
    pdl_launch_dependents();
    pdl_wait();
    const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const T *a = o + row * D, *b = dout + row * D;
    float s = 0.f;
    for (int c = lane; c < D; c += 32) s = fmaf(ldf(a + c), ldf(b + c), s);
    s = wsum(s);
    if (lane == 0) delta[heads > 0 ? (row % heads) * total + row / heads : row] = s;
}

// Same, with 16-byte loads: V = D * sizeof(T) / 16 threads per row (8, 16
// or 32), each taking one 16-byte piece of O and of dO, then a sum over the
// row's V lanes.  Needs O and dO 16-byte aligned (D is 64 or 128).
__device__ __forceinline__ float dot16(const uint4 &a, const uint4 &b, float) {
    const float *x = reinterpret_cast<const float *>(&a), *y = reinterpret_cast<const float *>(&b);
    return fmaf(x[0], y[0], fmaf(x[1], y[1], fmaf(x[2], y[2], x[3] * y[3])));
}
__device__ __forceinline__ float dot16(const uint4 &a, const uint4 &b, __nv_bfloat16) {
    const __nv_bfloat162 *x = reinterpret_cast<const __nv_bfloat162 *>(&a);
    const __nv_bfloat162 *y = reinterpret_cast<const __nv_bfloat162 *>(&b);
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 u = __bfloat1622float2(x[i]), v = __bfloat1622float2(y[i]);
        s = fmaf(u.x, v.x, fmaf(u.y, v.y, s));
    }
    return s;
}
template <typename T, int V>
__global__ void __launch_bounds__(256) bwd_delta16_kernel(const T *o, const T *dout, float *delta,
                                                          int64_t rows, int heads, int64_t total) {
    // Launched with programmatic stream serialization.  The next kernel is
    // released only as the CTAs finish: released at the start, its CTAs
    // would take registers from this memory-bound kernel's later CTAs.
    pdl_wait();
    const int64_t row = ((int64_t)blockIdx.x * 256 + threadIdx.x) / V;
    const int part = threadIdx.x % V;
    const bool live = row < rows;
    float s = 0.f;
    if (live) {
        const uint4 a = reinterpret_cast<const uint4 *>(o)[row * V + part];
        const uint4 b = reinterpret_cast<const uint4 *>(dout)[row * V + part];
        s = dot16(a, b, T());
    }
#pragma unroll
    for (int off = V / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (live && part == 0) delta[heads > 0 ? (row % heads) * total + row / heads : row] = s;
    pdl_launch_dependents();
}

// Rows [r0, r0 + kTile) of a head (row stride rs elements) into shared
// memory as float32 (zero past n).
template <int D, typename T>
__device__ __forceinline__ void stage(float *dst, const T *src, int64_t rs, int r0, int n) {
    for (int x = threadIdx.x; x < kTile * D; x += blockDim.x) {
        const int r = x / D, c = x % D;
        dst[x] = r0 + r < n ? ldf(src + (int64_t)(r0 + r) * rs + c) : 0.f;
    }
}

// dK, dV for 32 keys of one (batch, head).  Grid: units_bh * key blocks,
// lowest key block first (under the causal mask it has the most rows).
template <int D, typename Tin, typename Tout>
__global__ void __launch_bounds__(kWarps * 32) bwd_dkdv_simt_kernel(BwdParams p, int nblk) {
    constexpr int C = D / 32;
    __shared__ float sq[kTile * D], sdo[kTile * D];
    __shared__ float sl[kTile], sd[kTile];
    const int bh = blockIdx.x / nblk, j0 = (blockIdx.x % nblk) * kBlock;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Head hd = head_of(p, bh, D);
    if (j0 >= hd.len) return;
    const int n = hd.len;
    const int64_t rs = hd.rstride;
    const Tin *Q = static_cast<const Tin *>(p.q) + hd.elem0;
    const Tin *K = static_cast<const Tin *>(p.k) + hd.elem0;
    const Tin *V = static_cast<const Tin *>(p.v) + hd.elem0;
    const Tin *dO = static_cast<const Tin *>(p.dout) + hd.elem0;
    const float *L = p.lse + hd.stat0, *Dl = p.delta + hd.stat0;

    float kr[kPerWarp][C], vr[kPerWarp][C], dk[kPerWarp][C], dv[kPerWarp][C];
    int jk[kPerWarp];
#pragma unroll
    for (int t = 0; t < kPerWarp; ++t) {
        const int j = j0 + warp * kPerWarp + t;
        jk[t] = j;
#pragma unroll
        for (int c = 0; c < C; ++c) {
            const int col = lane + 32 * c;
            kr[t][c] = j < n ? ldf(K + (int64_t)j * rs + col) : 0.f;
            vr[t][c] = j < n ? ldf(V + (int64_t)j * rs + col) : 0.f;
            dk[t][c] = dv[t][c] = 0.f;
        }
    }
    // rows that can see some key of this block
    const int jl = j0 + kBlock - 1;
    int i_lo = 0, i_hi = n;
    if (p.causal) i_lo = j0;
    if (p.wr >= 0) i_lo = max(i_lo, j0 - p.wr);
    if (p.wl >= 0) i_hi = min(i_hi, jl + p.wl + 1);
    for (int i0 = i_lo; i0 < i_hi; i0 += kTile) {
        __syncthreads();
        stage<D>(sq, Q, rs, i0, n);
        stage<D>(sdo, dO, rs, i0, n);
        if (threadIdx.x < kTile) {
            const int i = i0 + threadIdx.x;
            sl[threadIdx.x] = i < n ? L[i] : 0.f;
            sd[threadIdx.x] = i < n ? Dl[i] : 0.f;
        }
        __syncthreads();
        const int rows = min(kTile, i_hi - i0);
        for (int r = 0; r < rows; ++r) {
            const int i = i0 + r;
            float qv[C], dov[C];
#pragma unroll
            for (int c = 0; c < C; ++c) {
                qv[c] = sq[r * D + lane + 32 * c];
                dov[c] = sdo[r * D + lane + 32 * c];
            }
#pragma unroll
            for (int t = 0; t < kPerWarp; ++t) {
                if (jk[t] >= n || !visible(i, jk[t], p)) continue;
                float s = 0.f, dp = 0.f;
#pragma unroll
                for (int c = 0; c < C; ++c) {
                    s = fmaf(qv[c], kr[t][c], s);
                    dp = fmaf(dov[c], vr[t][c], dp);
                }
                s = wsum(s);
                dp = wsum(dp);
                const float pij = expf(p.scale * s - sl[r]);
                const float ds = pij * (dp - sd[r]);
#pragma unroll
                for (int c = 0; c < C; ++c) {
                    dv[t][c] = fmaf(pij, dov[c], dv[t][c]);
                    dk[t][c] = fmaf(ds, qv[c], dk[t][c]);
                }
            }
        }
    }
    Tout *dK = static_cast<Tout *>(p.dk) + hd.elem0;
    Tout *dV = static_cast<Tout *>(p.dv) + hd.elem0;
#pragma unroll
    for (int t = 0; t < kPerWarp; ++t) {
        if (jk[t] >= n) continue;
#pragma unroll
        for (int c = 0; c < C; ++c) {
            const int col = lane + 32 * c;
            stf(dK + (int64_t)jk[t] * rs + col, p.scale * dk[t][c]);
            stf(dV + (int64_t)jk[t] * rs + col, dv[t][c]);
        }
    }
}

// dQ for 32 query rows of one (batch, head).  Grid: units_bh * row blocks,
// highest row block first (under the causal mask it has the most keys).
template <int D, typename Tin, typename Tout>
__global__ void __launch_bounds__(kWarps * 32) bwd_dq_simt_kernel(BwdParams p, int nblk) {
    constexpr int C = D / 32;
    __shared__ float sk[kTile * D], sv[kTile * D];
    const int bh = blockIdx.x / nblk, i0 = (nblk - 1 - blockIdx.x % nblk) * kBlock;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Head hd = head_of(p, bh, D);
    if (i0 >= hd.len) return;
    const int n = hd.len;
    const int64_t rs = hd.rstride;
    const Tin *Q = static_cast<const Tin *>(p.q) + hd.elem0;
    const Tin *K = static_cast<const Tin *>(p.k) + hd.elem0;
    const Tin *V = static_cast<const Tin *>(p.v) + hd.elem0;
    const Tin *dO = static_cast<const Tin *>(p.dout) + hd.elem0;
    const float *L = p.lse + hd.stat0, *Dl = p.delta + hd.stat0;

    float qr[kPerWarp][C], dor[kPerWarp][C], dq[kPerWarp][C], li[kPerWarp], di[kPerWarp];
    int ir[kPerWarp];
#pragma unroll
    for (int t = 0; t < kPerWarp; ++t) {
        const int i = i0 + warp * kPerWarp + t;
        ir[t] = i;
        li[t] = i < n ? L[i] : 0.f;
        di[t] = i < n ? Dl[i] : 0.f;
#pragma unroll
        for (int c = 0; c < C; ++c) {
            const int col = lane + 32 * c;
            qr[t][c] = i < n ? ldf(Q + (int64_t)i * rs + col) : 0.f;
            dor[t][c] = i < n ? ldf(dO + (int64_t)i * rs + col) : 0.f;
            dq[t][c] = 0.f;
        }
    }
    const int il = min(n, i0 + kBlock) - 1;
    int j_lo = 0, j_hi = n;
    if (p.causal) j_hi = il + 1;
    if (p.wr >= 0) j_hi = min(j_hi, il + p.wr + 1);
    if (p.wl >= 0) j_lo = max(0, i0 - p.wl);
    for (int j0 = j_lo; j0 < j_hi; j0 += kTile) {
        __syncthreads();
        stage<D>(sk, K, rs, j0, n);
        stage<D>(sv, V, rs, j0, n);
        __syncthreads();
        const int keys = min(kTile, j_hi - j0);
        for (int x = 0; x < keys; ++x) {
            const int j = j0 + x;
            float kv[C], vv[C];
#pragma unroll
            for (int c = 0; c < C; ++c) {
                kv[c] = sk[x * D + lane + 32 * c];
                vv[c] = sv[x * D + lane + 32 * c];
            }
#pragma unroll
            for (int t = 0; t < kPerWarp; ++t) {
                if (ir[t] >= n || !visible(ir[t], j, p)) continue;
                float s = 0.f, dp = 0.f;
#pragma unroll
                for (int c = 0; c < C; ++c) {
                    s = fmaf(qr[t][c], kv[c], s);
                    dp = fmaf(dor[t][c], vv[c], dp);
                }
                s = wsum(s);
                dp = wsum(dp);
                const float pij = expf(p.scale * s - li[t]);
                const float ds = pij * (dp - di[t]);
#pragma unroll
                for (int c = 0; c < C; ++c) dq[t][c] = fmaf(ds, kv[c], dq[t][c]);
            }
        }
    }
    Tout *dQ = static_cast<Tout *>(p.dq) + hd.elem0;
#pragma unroll
    for (int t = 0; t < kPerWarp; ++t) {
        if (ir[t] >= n) continue;
#pragma unroll
        for (int c = 0; c < C; ++c) stf(dQ + (int64_t)ir[t] * rs + lane + 32 * c, p.scale * dq[t][c]);
    }
}

BwdParams make_params(const FaBwdProblem &p) {
    BwdParams k;
    k.q = p.q;
    k.k = p.k;
    k.v = p.v;
    k.o = p.o;
    k.dout = p.dout;
    k.lse = p.lse;
    k.delta = p.delta;
    k.dq = p.dq;
    k.dk = p.dk;
    k.dv = p.dv;
    k.cu = p.cu_seqlens;
    k.varlen = p.varlen;
    k.heads = p.heads;
    k.num_seqs = p.num_seqs;
    k.total = p.total;
    k.err = p.err;
    k.n = p.n;
    k.D = p.D;
    k.scale = p.scale;
    k.causal = p.causal;
    k.wl = p.wl;
    k.wr = p.wr;
    return k;
}

template <int D, typename Tin, typename Tout>
fa_status launch(const FaBwdProblem &p) {
    const BwdParams k = make_params(p);
    const int nblk = (p.n + kBlock - 1) / kBlock;
    const long long grid = (long long)nblk * p.units_bh;
    if (grid > INT32_MAX) return FA_ERR_UNSUPPORTED;
    bwd_dkdv_simt_kernel<D, Tin, Tout><<<(int)grid, kWarps * 32, 0, p.stream>>>(k, nblk);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fa_cuda_fail(e);
    bwd_dq_simt_kernel<D, Tin, Tout><<<(int)grid, kWarps * 32, 0, p.stream>>>(k, nblk);
    e = cudaGetLastError();
    return e == cudaSuccess ? FA_OK : fa_cuda_fail(e);
}

template <int D>
fa_status launch_d(const FaBwdProblem &p) {
    switch (p.dtype) {
        case FA_F32: return launch<D, float, float>(p);
        case FA_BF16: return launch<D, __nv_bfloat16, __nv_bfloat16>(p);
        case FA_BF16_OUT_F32: return launch<D, __nv_bfloat16, float>(p);
        default: return FA_ERR_INVALID_ARG;
    }
}

}  // namespace
}  // namespace fa

fa_status fa_launch_bwd_delta(const FaBwdProblem &p) {
    const int64_t rows = p.varlen ? p.total * p.heads : (int64_t)p.units_bh * p.n;
    const int heads = p.varlen ? p.heads : 0;
    if (rows == 0) return FA_OK;
    const int64_t grid = (rows + 7) / 8;
    if (grid > INT32_MAX) return FA_ERR_UNSUPPORTED;
    // 16-byte pieces per row: 8, 16 or 32 threads per row
    const int vec = p.D * (p.dtype == FA_F32 ? 4 : 2) / 16;
    const bool aligned = ((reinterpret_cast<uintptr_t>(p.o) | reinterpret_cast<uintptr_t>(p.dout)) & 15u) == 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(256);
    cfg.stream = p.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    if (aligned && (vec == 8 || vec == 16 || vec == 32)) {
        const int64_t g16 = (rows * vec + 255) / 256;
        if (g16 > INT32_MAX) return FA_ERR_UNSUPPORTED;
        cfg.gridDim = dim3((unsigned)g16);
        const float *of = static_cast<const float *>(p.o), *df = static_cast<const float *>(p.dout);
        const __nv_bfloat16 *ob = static_cast<const __nv_bfloat16 *>(p.o);
        const __nv_bfloat16 *db = static_cast<const __nv_bfloat16 *>(p.dout);
        const bool f32 = p.dtype == FA_F32;
        if (vec == 8)
            e = f32 ? cudaLaunchKernelEx(&cfg, fa::bwd_delta16_kernel<float, 8>, of, df, p.delta, rows, heads, p.total)
                    : cudaLaunchKernelEx(&cfg, fa::bwd_delta16_kernel<__nv_bfloat16, 8>, ob, db, p.delta, rows,
                                         heads, p.total);
        else if (vec == 16)
            e = f32 ? cudaLaunchKernelEx(&cfg, fa::bwd_delta16_kernel<float, 16>, of, df, p.delta, rows, heads, p.total)
                    : cudaLaunchKernelEx(&cfg, fa::bwd_delta16_kernel<__nv_bfloat16, 16>, ob, db, p.delta, rows,
                                         heads, p.total);
        else
            e = f32 ? cudaLaunchKernelEx(&cfg, fa::bwd_delta16_kernel<float, 32>, of, df, p.delta, rows, heads, p.total)
                    : cudaLaunchKernelEx(&cfg, fa::bwd_delta16_kernel<__nv_bfloat16, 32>, ob, db, p.delta, rows,
                                         heads, p.total);
    } else if (p.dtype == FA_F32)
        e = cudaLaunchKernelEx(&cfg, fa::bwd_delta_kernel<float>, static_cast<const float *>(p.o),
                               static_cast<const float *>(p.dout), p.delta, rows, p.D, heads, p.total);
    else
        e = cudaLaunchKernelEx(&cfg, fa::bwd_delta_kernel<__nv_bfloat16>,
                               static_cast<const __nv_bfloat16 *>(p.o),
                               static_cast<const __nv_bfloat16 *>(p.dout), p.delta, rows, p.D, heads,
                               p.total);
    if (e == cudaSuccess) e = cudaGetLastError();
    return e == cudaSuccess ? FA_OK : fa_cuda_fail(e);
}

fa_status fa_launch_bwd_simt(const FaBwdProblem &p) {
    if ((int64_t)p.units_bh * p.n == 0) return FA_OK;
    return p.D == 64 ? fa::launch_d<64>(p) : fa::launch_d<128>(p);
}
