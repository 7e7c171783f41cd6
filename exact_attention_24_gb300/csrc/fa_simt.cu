// FFMA (CUDA-core) FlashAttention-2 forward kernel.
//
// Serves FA_F32 (float32 in/out, full-precision expf/logf) and is the
// known-good fallback for the bf16 dtypes.  It follows the tiled loop of
// "FlashAttention -- for programmers, not researchers.", STAGE 4: one CTA
// owns a block of 64 query rows of one (batch, head) or (sequence, head) --
// "Kernel visualization: Flash Attention 2", section "Steps" (one block per
// Br rows of Q, grid over (Q tile, batch*head)) -- and streams 64-key K/V
// tiles through shared memory, carrying per row the running max m, running
// sum l and an unnormalised output accumulator that is rescaled by
// exp(m_old - m_new) whenever the max grows (STAGE 3/4, and the section
// "Iteration j = 1").  O is divided by l once at the end and L = m + ln l
// ("Write the data back to HBM").
//
// Mapping: 8 warps, each owning 8 query rows.  For one row, lane t scores
// keys t and t+32 (dot products out of padded shared memory), the row max
// and row sum are warp shuffles, and lane t accumulates output columns
// t, t+32, ... of the row.
#include <cuda_bf16.h>
#include <math.h>

#include "device_common.cuh"

namespace fa {
namespace {

constexpr int kBc = 64;      // keys per K/V tile
constexpr int kWarps = 8;    // a CTA's query rows: kWarps x rows per warp (8, or 1
                             // when the 64-row grid would leave SMs idle)

struct SimtParams {
    const void *q, *k, *v;
    void *o;
    float *lse;
    const int32_t *cu;
    int varlen, heads, n, D;
    int64_t total;
    float scale;
    int causal;
    int wl, wr;  // key j visible to row i iff i - wl <= j <= i + wr (< 0: unbounded)
    uint32_t *err;
};

__device__ __forceinline__ float ld_f32(const float *p) { return __ldg(p); }
__device__ __forceinline__ float ld_f32(const __nv_bfloat16 *p) {
    return __bfloat162float(*p);
}
__device__ __forceinline__ void st_out(float *p, float x) { *p = x; }
__device__ __forceinline__ void st_out(__nv_bfloat16 *p, float x) {
    *p = __float2bfloat16_rn(x);
}

// Copy ROWS rows of D elements (row stride `stride` elements) starting at
// row `r0` of a head into shared memory as fp32 with row pitch `pitch`;
// rows at or beyond `len` are zero-filled.  Each thread issues its global
// loads kBatch at a time into registers before storing them, so their
// latencies overlap (a load cannot pass a shared-memory store that might
// alias it).
template <int D, int ROWS, typename Tin>
__device__ __forceinline__ void load_tile(float *dst, int pitch, const Tin *src,
                                          int64_t stride, int r0, int len) {
    constexpr int kThreads = kWarps * 32;
    constexpr int kElems = ROWS * D;
    constexpr int kPer = (kElems + kThreads - 1) / kThreads;  // elements per thread
    constexpr int kBatch = kPer < 8 ? kPer : 8;
#pragma unroll
    for (int i0 = 0; i0 < kPer; i0 += kBatch) {
        float buf[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const int x = threadIdx.x + (i0 + i) * kThreads;
            const int row = r0 + x / D;
            buf[i] = (i0 + i < kPer && x < kElems && row < len)
                         ? ld_f32(src + (int64_t)row * stride + x % D) : 0.f;
        }
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const int x = threadIdx.x + (i0 + i) * kThreads;
            if (i0 + i < kPer && x < kElems) dst[(x / D) * pitch + x % D] = buf[i];
        }
    }
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

template <int D, int RPW, typename Tin, typename Tout>
__global__ void __launch_bounds__(kWarps * 32, 2)
    fa_simt_kernel(SimtParams p) {
    constexpr int kBr = RPW * kWarps;    // query rows per CTA
    extern __shared__ float smem[];
    float *sQ = smem;                    // [kBr][D]
    float *sK = sQ + kBr * D;            // [kBc][D + 1]  (padded: no bank conflicts)
    float *sV = sK + kBc * (D + 1);      // [kBc][D]

    const int unit = blockIdx.x;
    // Heaviest (latest) query tiles first under the causal mask.
    const int tile = p.causal ? (gridDim.y - 1 - blockIdx.y) : blockIdx.y;
    int64_t base, stride, lbase;
    int len;
    if (p.varlen) {
        const int s = unit / p.heads, h = unit % p.heads;
        int64_t start;
        if (!seq_bounds(p.cu, s, p.total, p.n, p.err, start, len)) return;
        base = (start * p.heads + h) * D;
        stride = (int64_t)p.heads * D;
        lbase = (int64_t)h * p.total + start;
    } else {
        len = p.n;
        base = (int64_t)unit * p.n * D;
        stride = D;
        lbase = (int64_t)unit * p.n;
    }
    const int q0 = tile * kBr;
    if (q0 >= len) return;

    const Tin *Q = static_cast<const Tin *>(p.q) + base;
    const Tin *K = static_cast<const Tin *>(p.k) + base;
    const Tin *V = static_cast<const Tin *>(p.v) + base;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int DC = D / 32;  // output columns per lane

    load_tile<D, kBr>(sQ, D, Q, stride, q0, len);

    float acc[RPW][DC];
    float m[RPW], l[RPW];
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
        m[r] = -INFINITY;
        l[r] = 0.f;
#pragma unroll
        for (int t = 0; t < DC; ++t) acc[r][t] = 0.f;
    }

    // Keys any row of this block can see: [kv_lo, kv_end).
    const int kv_end = p.wr >= 0 ? min(len, q0 + kBr - 1 + p.wr + 1) : len;
    const int kv_lo = p.wl >= 0 ? max(0, q0 - p.wl) / kBc * kBc : 0;
    for (int kv0 = kv_lo; kv0 < kv_end; kv0 += kBc) {
        __syncthreads();  // previous tile fully consumed (and sQ written)
        load_tile<D, kBc>(sK, D + 1, K, stride, kv0, len);
        load_tile<D, kBc>(sV, D, V, stride, kv0, len);
        __syncthreads();
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            const int row = warp * RPW + r;
            const int qi = q0 + row;
            if (qi >= len) continue;  // warp-uniform
            const float *qrow = sQ + row * D;
            const float *k0 = sK + lane * (D + 1);
            const float *k1 = sK + (lane + 32) * (D + 1);
            float s0 = 0.f, s1 = 0.f;
#pragma unroll 8
            for (int d = 0; d < D; ++d) {
                const float qd = qrow[d];
                s0 = fmaf(qd, k0[d], s0);
                s1 = fmaf(qd, k1[d], s1);
            }
            s0 *= p.scale;  // scale after the dot product
            s1 *= p.scale;
            const int key0 = kv0 + lane, key1 = kv0 + lane + 32;
            const int hi = p.wr >= 0 ? qi + p.wr : len - 1;   // last visible key
            const int lo = p.wl >= 0 ? qi - p.wl : 0;          // first visible key
            if (key0 >= len || key0 > hi || key0 < lo) s0 = -INFINITY;
            if (key1 >= len || key1 > hi || key1 < lo) s1 = -INFINITY;
            const float m_new = fmaxf(m[r], warp_max(fmaxf(s0, s1)));
            const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
            const float alpha = (m[r] == -INFINITY) ? 0.f : expf(m[r] - m_use);
            const float p0 = expf(s0 - m_use), p1 = expf(s1 - m_use);
            l[r] = alpha * l[r] + warp_sum(p0 + p1);
#pragma unroll
            for (int t = 0; t < DC; ++t) acc[r][t] *= alpha;
#pragma unroll 4
            for (int c = 0; c < 32; ++c) {
                const float pc = __shfl_sync(0xffffffffu, p0, c);
                const float *vr = sV + c * D + lane;
#pragma unroll
                for (int t = 0; t < DC; ++t) acc[r][t] = fmaf(pc, vr[32 * t], acc[r][t]);
            }
#pragma unroll 4
            for (int c = 0; c < 32; ++c) {
                const float pc = __shfl_sync(0xffffffffu, p1, c);
                const float *vr = sV + (c + 32) * D + lane;
#pragma unroll
                for (int t = 0; t < DC; ++t) acc[r][t] = fmaf(pc, vr[32 * t], acc[r][t]);
            }
            m[r] = m_new;
        }
    }

    Tout *O = static_cast<Tout *>(p.o) + base;
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
        const int qi = q0 + warp * RPW + r;
        if (qi >= len) continue;
        const bool live = l[r] > 0.f;
        const float inv = live ? 1.f / l[r] : 0.f;
#pragma unroll
        for (int t = 0; t < DC; ++t)
            st_out(O + (int64_t)qi * stride + lane + 32 * t, acc[r][t] * inv);
        if (lane == 0) p.lse[lbase + qi] = live ? m[r] + logf(l[r]) : -INFINITY;
    }
}

template <int D, int RPW, typename Tin, typename Tout>
fa_status launch(const FaProblem &pr) {
    constexpr int kBr = RPW * kWarps;
    SimtParams p;
    p.q = pr.q;
    p.k = pr.k;
    p.v = pr.v;
    p.o = pr.o;
    p.lse = pr.lse;
    p.cu = pr.cu_seqlens;
    p.varlen = pr.varlen;
    p.heads = pr.heads;
    p.n = pr.n;
    p.D = D;
    p.total = pr.total;
    p.scale = pr.scale;
    p.causal = pr.causal;
    p.wl = pr.wl;
    p.wr = pr.wr;
    p.err = pr.err;
    const size_t smem = sizeof(float) * (size_t)(kBr * D + kBc * (D + 1) + kBc * D);
    auto kern = fa_simt_kernel<D, RPW, Tin, Tout>;
    static FaCtxSet ready;  // contexts set up for this instantiation
    const fa_status su = fa_once_per_context(ready, [&]() -> fa_status {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        return e == cudaSuccess ? FA_OK : fa_cuda_fail(e);
    });
    if (su != FA_OK) return su;
    const int tiles = (pr.n + kBr - 1) / kBr;
    dim3 grid(pr.units_bh, tiles);
    kern<<<grid, kWarps * 32, smem, pr.stream>>>(p);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? FA_OK : fa_cuda_fail(e);
}

template <int D, int RPW>
fa_status launch_dt(const FaProblem &pr) {
    switch (pr.dtype) {
        case FA_F32: return launch<D, RPW, float, float>(pr);
        case FA_BF16: return launch<D, RPW, __nv_bfloat16, __nv_bfloat16>(pr);
        case FA_BF16_OUT_F32: return launch<D, RPW, __nv_bfloat16, float>(pr);
        default: return FA_ERR_INVALID_ARG;
    }
}


// 64-row CTAs (8 rows a warp) unless that grid leaves SMs idle; then 8-row
// CTAs (one row a warp), 8x the CTAs.  Each row's arithmetic is the same
// either way, so the results do not depend on the choice.
template <int D>
fa_status launch_d(const FaProblem &pr) {
    const int64_t blocks64 = (int64_t)pr.units_bh * ((pr.n + 8 * kWarps - 1) / (8 * kWarps));
    const bool small = blocks64 < fa_num_sms() && (pr.n + kWarps - 1) / kWarps <= 65535;
    return small ? launch_dt<D, 1>(pr) : launch_dt<D, 8>(pr);
}

}  // namespace
}  // namespace fa

fa_status fa_launch_simt(const FaProblem &pr) {
    if ((pr.n + 8 * fa::kWarps - 1) / (8 * fa::kWarps) > 65535) return FA_ERR_UNSUPPORTED;
    if (pr.D == 64) return fa::launch_d<64>(pr);
    if (pr.D == 128) return fa::launch_d<128>(pr);
    return FA_ERR_UNSUPPORTED;
}
