// Tensor-core (tcgen05) backward pass.
//
// The gradients of "FlashAttention -- for programmers, not researchers.",
// STAGE 5: the probabilities are recomputed tile by tile from Q, K and the
// forward pass's L, P = exp(scale Q K^T - L), never stored.  The five
// contractions of the "FlashAttention" docs page, section "Application in
// Backward Pass (5 MMAs)", run in two kernels so that every output has one
// owner and every sum a fixed order (no atomics):
//
//   dK/dV kernel, one 128-key block per CTA, K and V resident:
//     S^T = K Q_i^T, dP^T = V dO_i^T           (128 x 128, lanes = keys)
//     P^T = exp2(S^T c - L_i log2 e), dS^T = P^T (dP^T - delta_i)
//     dV += P^T dO_i, dK += dS^T Q_i           (A operand from TMEM)
//   dQ kernel, one 128-row query block per CTA, Q and dO resident:
//     S = Q K_j^T, dP = dO V_j^T               (lanes = query rows)
//     P, dS as above; dQ += dS K_j             (A operand from TMEM)
//
// Both are made of the forward pass's two MMA shapes (A B^T with both
// operands K-major in shared memory; A from TMEM times an MN-major shared
// operand).  The streamed operands (Q_i and dO_i, or K_j and V_j) flow
// through a TMA ring.  Two warpgroups turn S, dP into P, dS (one TMEM lane,
// i.e. one key or one query row, per thread), each on half of a tile's
// columns: warps 0-3 and 7-10 in the dK/dV kernel, 0-3 and 6-9 in the dQ
// kernel.  Warp 4 is the TMA producer, warp 5 allocates TMEM.  In the dK/dV
// kernel warps 5 and 6 issue the MMAs in turns, one per half-tile buffer; in
// the dQ kernel warp 5 issues them and warp 10 does the waits for its next
// issue block meanwhile.  Every wait is bounded (the device watchdog of the
// forward kernel).
#include <cuda.h>
#include <cuda_bf16.h>
#include <math.h>

#include "device_common.cuh"
#include "tc_common.cuh"

namespace fa {
namespace {

constexpr int kT = kTcRows;          // 128 rows / keys per tile
constexpr int kProdWarp = 4;
constexpr int kMmaWarp = 5;
// dQ kernel: two dS warpgroups, warps 0-3 for keys 0-63 of each tile and
// warps 6-9 for keys 64-127 (warp w reads TMEM lanes 32 (w % 4) ..)
constexpr int kDqThreads = 352;
constexpr int kDqEwB = 6;
// dQ kernel: warp 10 does the MMA warp's barrier waits for the next issue
// block while warp 5 issues the current one; they meet at named barrier 1
constexpr int kDqWaitWarp = 10;
constexpr uint32_t kDqGo = 1;
// dK/dV kernel: a second MMA issuer warp (see its MMA role) and a second
// elementwise warpgroup: warps 0-3 take query columns 0-31 of each half,
// warps 7-10 columns 32-63 (warp w reads TMEM lanes 32 (w % 4) ..)
constexpr int kDkThreads = 352;
constexpr int kDkMmaWarpA = 5;      // issuer of half-tile buffer 0; allocates TMEM
constexpr int kDkMmaWarpB = 6;      // issuer of half-tile buffer 1
constexpr int kDkEwB = 7;           // first warp of the second elementwise warpgroup
constexpr uint32_t kDkToken = 2;    // named barriers 2, 3 (1 and 4 are the elementwise warpgroups')
constexpr uint32_t kTmemCols = 512;

struct BwdTcParams {
    const float *lse, *delta;
    void *dq, *dk, *dv;
    const int32_t *cu;    // packed batch: sequence offsets (null for dense)
    int varlen, heads;
    int64_t total;
    int units;            // problems: B*H, or num_seqs*H
    int n, nblk;          // n: N, or the longest sequence of a packed batch
    float scale, scale_log2;
    int causal;
    int wl, wr;           // band: key j visible to row i iff i - wl <= j <= i + wr (< 0: unbounded)
    uint32_t *err;
    uint64_t wait_limit_ns;
    int num_seqs;         // packed batch: sequences
    int compact;          // packed batch: walk the compact order (bwd_decode_compact)
    int head_group;       // compact order: number of near-equal head groups
};

// Packed batches with at most kMaxBwdSchedSeqs sequences and
// kMaxBwdSchedLevels 128-row blocks per sequence walk a compact order: only
// blocks that hold rows, heads in groups whose streamed operands (Q and dO
// for dK/dV, K and V for dQ) stay in L2 while the group's items run.
constexpr int kMaxBwdSchedSeqs = 255;
constexpr int kMaxBwdSchedLevels = 128;
constexpr int kBwdSchedBytes = 416;  // ranked[256] + reach[128] (bytes) + the item count
#ifndef FA_BWD_GROUP_MB
#define FA_BWD_GROUP_MB 96
#endif
constexpr double kBwdL2GroupBytes = FA_BWD_GROUP_MB * 1024.0 * 1024;

// The compact order's table in shared memory: the sequences ranked by block
// count (longest first, ties by index) and, per block level L, how many
// sequences have more than L blocks.  Every CTA builds the same table.
struct BwdSched {
    const uint8_t *ranked;  // [num_seqs]
    const uint8_t *reach;   // [nblk]
    int per_head;           // blocks per head: the sum of reach over the levels
};

// Build the table at `tab` (all threads of the CTA; `scratch` holds an int
// per sequence and is generic-proxy memory the TMA overwrites afterwards).
__device__ __forceinline__ void build_bwd_sched(const BwdTcParams &p, uint8_t *tab, int *scratch) {
    for (int q = threadIdx.x; q < p.num_seqs; q += blockDim.x) {
        int64_t start;
        int len;
        seq_bounds(p.cu, q, p.total, p.n, p.err, start, len);  // invalid: len = 0
        scratch[q] = (len + kT - 1) / kT;
    }
    __syncthreads();
    uint8_t *ranked = tab, *reach = tab + 256;
    for (int q = threadIdx.x; q < p.num_seqs; q += blockDim.x) {
        const int nq = scratch[q];
        int rank = 0;
        for (int t = 0; t < p.num_seqs; ++t) rank += (scratch[t] > nq) || (scratch[t] == nq && t < q);
        ranked[rank] = (uint8_t)q;
    }
    for (int L = threadIdx.x; L < p.nblk; L += blockDim.x) {
        int r = 0;
        for (int t = 0; t < p.num_seqs; ++t) r += scratch[t] > L;
        reach[L] = (uint8_t)r;
    }
    if (threadIdx.x == 0) {
        int total = 0;
        for (int t = 0; t < p.num_seqs; ++t) total += scratch[t];
        *reinterpret_cast<int *>(tab + 400) = total;
    }
    // the scratch's generic-proxy use is over before TMA (async proxy) writes it
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ BwdSched bwd_sched(const BwdTcParams &p, const uint8_t *tab) {
    return BwdSched{tab, tab + 256, p.compact ? *reinterpret_cast<const int *>(tab + 400) : 0};
}

// Item `idx` of the compact order: heads in p.head_group near-equal groups;
// within a group block level L (from the first block up, or from the last
// block down), then the sequences that reach L (longest first), then the
// group's heads.
__device__ __forceinline__ bool bwd_decode_compact(const BwdTcParams &p, const BwdSched &sc, int idx,
                                                   bool from_top, int &unit, int &blk) {
    // p.head_group near-equal groups: group g holds heads [g H / n, (g + 1) H / n)
    const int ng = p.head_group;
    int grp = 0, h0 = 0, hn = 0;
    for (; grp < ng; ++grp) {
        h0 = grp * p.heads / ng;
        hn = (grp + 1) * p.heads / ng - h0;
        if (idx < sc.per_head * hn) break;
        idx -= sc.per_head * hn;
    }
    if (grp == ng) return false;
    int L = from_top ? p.nblk - 1 : 0;
    for (;;) {
        if (L < 0 || L >= p.nblk) return false;
        const int here = (int)sc.reach[L] * hn;
        if (idx < here) break;
        idx -= here;
        L += from_top ? -1 : 1;
    }
    unit = (int)sc.ranked[idx / hn] * p.heads + h0 + idx % hn;
    blk = L;
    return true;
}

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ void store_row(float *dst, const float *x, float mul) {
    float4 *d = reinterpret_cast<float4 *>(dst);
#pragma unroll
    for (int i = 0; i < 8; ++i)
        d[i] = make_float4(x[4 * i] * mul, x[4 * i + 1] * mul, x[4 * i + 2] * mul, x[4 * i + 3] * mul);
}
__device__ __forceinline__ void store_row(__nv_bfloat16 *dst, const float *x, float mul) {
    uint4 *d = reinterpret_cast<uint4 *>(dst);
#pragma unroll
    for (int i = 0; i < 4; ++i)
        d[i] = make_uint4(pack_bf16x2(x[8 * i] * mul, x[8 * i + 1] * mul),
                          pack_bf16x2(x[8 * i + 2] * mul, x[8 * i + 3] * mul),
                          pack_bf16x2(x[8 * i + 4] * mul, x[8 * i + 5] * mul),
                          pack_bf16x2(x[8 * i + 6] * mul, x[8 * i + 7] * mul));
}

// One attention problem of the batch -- (batch, head) of a dense [B, H, N, D]
// batch or (sequence, head) of a packed [total, H, D] one: row i of its
// tensors starts at element elem0 + i * rstride, its L / delta entry is at
// stat0 + i, and TMA addresses it as (unit, row) or (head, start + row).
struct Seq {
    int64_t elem0, rstride, stat0, start;
    int len, h, unit;
};

__device__ __forceinline__ Seq seq_of(const BwdTcParams &p, int unit, int D) {
    Seq q;
    q.unit = unit;
    if (!p.varlen) {
        q.start = 0;
        q.h = 0;
        q.len = p.n;
        q.elem0 = (int64_t)unit * p.n * D;
        q.rstride = D;
        q.stat0 = (int64_t)unit * p.n;
    } else {
        const int s = unit / p.heads;
        q.h = unit % p.heads;
        seq_bounds(p.cu, s, p.total, p.n, p.err, q.start, q.len);  // invalid: len = 0
        q.elem0 = (q.start * p.heads + q.h) * D;
        q.rstride = (int64_t)p.heads * D;
        q.stat0 = (int64_t)q.h * p.total + q.start;
    }
    return q;
}

// TMA: rows [row, row + box) (all D columns) of one problem's tensor; a box
// is 64 columns wide, `atom` bytes per 64-column group in shared memory.
template <int D>
__device__ __forceinline__ void load_rows(uint32_t dst, const CUtensorMap *tm, uint32_t bar, int row,
                                          const Seq &q, int varlen, int atom) {
#pragma unroll
    for (int hf = 0; hf < D / 64; ++hf) {
        if (varlen)
            tma_load_3d(dst + hf * atom, tm, bar, hf * 64, q.h, (int)(q.start + row));
        else
            tma_load_3d(dst + hf * atom, tm, bar, hf * 64, row, q.unit);
    }
}

// Query rows a dK/dV item walks: [i_first, i_first + 64 * halves) covers
// every row that sees some key of the block [j0, j0 + 128) (an even number
// of 64-row halves).  Causal / full attention, or a band (WIN).
template <bool WIN>
__device__ __forceinline__ void dk_rows(const BwdTcParams &p, int j0, int n, int &i_first, int &halves) {
    int lo = p.causal ? j0 : 0, hi = n;
    if (WIN) {
        lo = p.wr >= 0 ? max(0, j0 - p.wr) : 0;
        hi = p.wl >= 0 ? min(n, j0 + kT + p.wl) : n;
    }
    i_first = lo;
    halves = 2 * ((hi - lo + kT - 1) / kT);
}

// ------------------------------------------------------------ dK, dV --
// The streamed operands arrive as 64-row halves of a query tile (Q_x and
// dO_x of tile t, x = 0, 1) through a ring of kSlots half-tile slots, and
// each half has its own TMEM buffers S^T_x, dP^T_x (64 columns each).  While
// the softmax warps turn one half into P^T, dS^T, the MMA warp accumulates
// the other half and computes its next S^T, dP^T:
//   for half u = 2t + x:  wait P_x(u); dV += P^T_x dO_x; dK += dS^T_x Q_x;
//                         release slot u; S^T_x(u + 2) = K Q^T, dP^T_x(u + 2) = V dO^T
// (a buffer is overwritten only after the accumulating MMAs that read it:
// one issuing thread, executed in order).  The ring holds 2.5 tiles, so a
// half-tile's load is issued two halves before its first MMA.
template <int D>
struct DkCfg {
    static constexpr int kTileBytes = kT * D * 2;       // K or V (128 rows)
    static constexpr int kHalfBytes = 64 * D * 2;       // Q_x or dO_x (64 rows)
    static constexpr int kHalfAtom = 64 * 128;          // one 64-element-wide box of 64 rows
    static constexpr int kSlots = D == 128 ? 5 : 10;
    static constexpr int kSlotBytes = 2 * kHalfBytes;
    static constexpr int kRingOff = 2 * kTileBytes;
    static constexpr int kStatOff = kRingOff + kSlots * kSlotBytes;
    static constexpr int kStatBytes = 2 * 2 * 64 * 4;   // [half parity][L, delta][64]
    static constexpr int kBarOff = kStatOff + kStatBytes;
    static constexpr int kBarBytes = 256;
    static constexpr int kSchedOff = kBarOff + kBarBytes;   // packed-batch walk table
    static constexpr int kSmemBytes = kSchedOff + kBwdSchedBytes + 1024;
    static_assert(kSmemBytes <= 232448, "shared memory per CTA");
    static_assert(8 * (2 + 2 * kSlots + 7) + 16 <= kBarBytes, "barrier area");
};

// K/V loaded and free again, ring full/empty per slot, S^T/dP^T ready and
// P^T/dS^T ready per half-buffer, accumulators final and read, drain.
struct DkBars {
    uint32_t fix_full, kv_free, ring_full, ring_empty, s_full, p_full, o_final, acc_free, drain;
    __device__ DkBars(uint32_t b, int slots)
        : fix_full(b), kv_free(b + 8), ring_full(b + 16), ring_empty(b + 16 + 8 * slots),
          s_full(b + 16 + 16 * slots), p_full(b + 32 + 16 * slots), o_final(b + 48 + 16 * slots),
          acc_free(b + 56 + 16 * slots), drain(b + 64 + 16 * slots) {}
};

// The CTA's next dK/dV work item at or after walk position k: items are
// numbered key block first (lowest first: under the causal mask it has the
// most query rows), then problem; CTA c takes items c, 2G-1-c, 2G+c, ...
// Blocks past the end of their sequence are skipped.
__device__ __forceinline__ bool next_dk_item(const BwdTcParams &p, const BwdSched &sc, int &k, int cta, int G,
                                             int D, Seq &sq, int &j0) {
    if (p.compact) {  // key block from the first (most query rows under the causal mask) up
        const int items = sc.per_head * p.heads;
        for (; k * G < items; ++k) {
            const int idx = k * G + ((k & 1) ? (G - 1 - cta) : cta);
            int unit, blk;
            if (idx >= items || !bwd_decode_compact(p, sc, idx, false, unit, blk)) continue;
            sq = seq_of(p, unit, D);
            j0 = blk * kT;
            if (j0 < sq.len) {
                ++k;
                return true;
            }
        }
        return false;
    }
    const int items = p.nblk * p.units;
    for (; k * G < items; ++k) {
        const int idx = k * G + ((k & 1) ? (G - 1 - cta) : cta);
        if (idx >= items) continue;
        const int jb = idx / p.units, unit = idx % p.units;
        sq = seq_of(p, unit, D);
        j0 = jb * kT;
        if (j0 < sq.len) {
            ++k;
            return true;
        }
    }
    return false;
}

// S^T_x (TMEM, 128 keys x 64 queries fp32) = K (smem, 128 x D) * Q_x^T
// (smem, 64 x D): both K-major; K's 64-element boxes are 16 KB apart, a
// half-tile's 8 KB.
template <int D>
__device__ __forceinline__ void issue_st_half(uint32_t d_tmem, uint64_t da, uint64_t db) {
    constexpr uint32_t idesc = idesc_bf16(kTcRows, 64, 0);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t oa = (uint64_t)(((kk / 4) * kTcAtomBytes + (kk % 4) * 32) >> 4);
        const uint64_t ob = (uint64_t)(((kk / 4) * DkCfg<D>::kHalfAtom + (kk % 4) * 32) >> 4);
        mma_ss(d_tmem, da + oa, db + ob, idesc, kk > 0 ? 1u : 0u);
    }
}

// acc (TMEM, 128 x D fp32) (+)= A (TMEM, 128 x 64 bf16) * B_x with B_x a
// half-tile viewed MN-major (64 x D; boxes 8 KB apart): 4 MMAs of 16 rows.
// A's queries 32 c .. 32 c + 31 (bf16 pairs) sit at columns 32 c .. 32 c + 15,
// over the score columns that elementwise warpgroup c has read.
template <int D>
__device__ __forceinline__ void issue_acc_half(uint32_t d_tmem, uint32_t a_tmem, uint64_t db,
                                               uint32_t accumulate) {
    constexpr uint32_t idesc = idesc_bf16(kTcRows, D, 1);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
        mma_ts(d_tmem, a_tmem + (kk >> 1) * 32 + (kk & 1) * 8, db + (uint64_t)((kk * 2048) >> 4), idesc,
               (kk > 0 || accumulate) ? 1u : 0u);
}

template <int D, typename Tout, bool WIN>
__global__ void __launch_bounds__(kDkThreads, 1)
    bwd_dkdv_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       const BwdTcParams p) {
    // Persistent: each CTA walks its items in turn.  Across an item boundary
    // K and V are reloaded as soon as the item's last S^T, dP^T have been
    // issued, and the next item's first S^T, dP^T run while the softmax
    // warps store the previous dK, dV; its first accumulating MMA waits until
    // they have read them (acc_free).  Barrier phases and ring slots count
    // halves and items over the CTA's whole walk.
    using C = DkCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const DkBars b(base + C::kBarOff, C::kSlots);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + C::kBarOff + C::kBarBytes - 16);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(gbase + C::kBarOff + C::kBarBytes - 8);
    volatile int *exit_flag = reinterpret_cast<volatile int *>(gbase + C::kBarOff + C::kBarBytes - 12);
    float *stat = reinterpret_cast<float *>(gbase + C::kStatOff);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x, G = gridDim.x;

    if (warp == kProdWarp && lane == 0) {
        mbar_init(b.fix_full, 1);
        mbar_init(b.kv_free, 2);       // one commit per issuer
        for (int i = 0; i < C::kSlots; ++i) {
            mbar_init(b.ring_full + 8 * i, 1);
            mbar_init(b.ring_empty + 8 * i, 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(b.s_full + 8 * x, 1);
            mbar_init(b.p_full + 8 * x, 8);   // both elementwise warpgroups
        }
        mbar_init(b.o_final, 2);       // one commit per issuer
        mbar_init(b.acc_free, 8);
        mbar_init(b.drain, 2);
        fence_barrier_init();
        *abort_flag = 0;
        *exit_flag = 0;
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_do);
    }
    if (warp == kDkMmaWarpA) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    // the packed-batch walk table (scratch: the not yet used ring)
    uint8_t *sched_tab = gbase + C::kSchedOff;
    if (p.compact) build_bwd_sched(p, sched_tab, reinterpret_cast<int *>(gbase + C::kRingOff));
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const BwdSched sched = bwd_sched(p, sched_tab);
    const uint32_t tmem = *tmem_slot;
    const WaitCtx wc{p.err, abort_flag, p.wait_limit_ns};
    const uint32_t ring = base + C::kRingOff;

    if (warp == kProdWarp) {
        // ---------------------------------------------------- producer
        if (lane == 0) {
            int k = 0, it = 0, g = 0;  // walk position, items, halves loaded
            bool ok = true;
            Seq sq;
            int j0;
            while (ok && next_dk_item(p, sched, k, cta, G, D, sq, j0)) {
                int i_first, halves;
                dk_rows<WIN>(p, j0, sq.len, i_first, halves);
                if (it > 0 && !mbar_wait(b.kv_free, (it - 1) & 1, wc, 0x40)) break;
                mbar_arrive_expect_tx(b.fix_full, 2 * C::kTileBytes);
                load_rows<D>(base, &tm_k, b.fix_full, j0, sq, p.varlen, kTcAtomBytes);
                load_rows<D>(base + C::kTileBytes, &tm_v, b.fix_full, j0, sq, p.varlen, kTcAtomBytes);
                ++it;
                for (int u = 0; u < halves; ++u, ++g) {
                    const int slot = g % C::kSlots, round = g / C::kSlots;
                    if (round > 0 && !mbar_wait(b.ring_empty + 8 * slot, (round - 1) & 1, wc, 0x41)) {
                        ok = false;
                        break;
                    }
                    const uint32_t dst = ring + slot * C::kSlotBytes, fb = b.ring_full + 8 * slot;
                    mbar_arrive_expect_tx(fb, C::kSlotBytes);
                    load_rows<D>(dst, &tm_q, fb, i_first + 64 * u, sq, p.varlen, C::kHalfAtom);
                    load_rows<D>(dst + C::kHalfBytes, &tm_do, fb, i_first + 64 * u, sq, p.varlen, C::kHalfAtom);
                }
            }
            const uint64_t lim = p.wait_limit_ns;
            if (it > 0) mbar_drain(b.fix_full, (it - 1) & 1, lim);
            for (int v = g > C::kSlots ? g - C::kSlots : 0; v < g; ++v)
                mbar_drain(b.ring_full + 8 * (v % C::kSlots), (v / C::kSlots) & 1, lim);
        }
    } else if (warp == kDkMmaWarpA || warp == kDkMmaWarpB) {
        // --------------------------------------------------------- MMA
        // Two issuer warps, one per half-tile buffer x (the halves u with
        // u % 2 == x).  tcgen05.mma issue is effectively synchronous with
        // execution, so an issuer's barrier waits are tensor idle time unless
        // the other issuer is issuing meanwhile: the warps take turns through
        // a token (named barriers kDkToken + x), each doing its waits while
        // the other issues.  Per item the turns are the two prologue halves,
        // then one per half (an even number in all).  K, V and the
        // accumulators are shared: their release barriers count a commit per
        // issuer.  A warp that must stop raises the exit flag and still passes
        // the token.
        constexpr uint64_t kTileDesc = C::kTileBytes >> 4, kSlotDesc = C::kSlotBytes >> 4;
        constexpr uint64_t kHalfDesc = C::kHalfBytes >> 4;
        const int X = warp - kDkMmaWarpA;
        const uint64_t d_k = smem_desc(base, 16, 1024), d_v = d_k + kTileDesc;
        const uint64_t d_ring_k = smem_desc(ring, 16, 1024);                 // K-major view
        const uint64_t d_ring_mn = smem_desc(ring, C::kHalfAtom, 1024);      // MN-major view
        const uint32_t t_dv = tmem + 2 * kT, t_dk = t_dv + D;
        const uint32_t t_st = tmem + X * 2 * 64, t_dpt = t_st + 64;        // this issuer's buffer
        const uint32_t tok_me = kDkToken + X, tok_other = kDkToken + 1 - X;
        auto turn_begin = [&](bool waits_ok) -> bool {
            named_bar_sync(tok_me, 64);
            if (*exit_flag) return false;
            if (!waits_ok || *abort_flag) {
                *exit_flag = 1;
                __threadfence_block();
                __syncwarp();
                named_bar_arrive(tok_other, 64);
                return false;
            }
            tc_fence_after();
            return true;
        };
        auto turn_end = [&]() {
            __syncwarp();
            named_bar_arrive(tok_other, 64);
        };
        if (X == 1) named_bar_arrive(kDkToken, 64);   // buffer 0's issuer takes the first turn
        int k = 0, it = 0, g = 0;
        bool run = true;
        Seq sq;
        int j0;
        while (run && next_dk_item(p, sched, k, cta, G, D, sq, j0)) {
            int i_first, halves;
            dk_rows<WIN>(p, j0, sq.len, i_first, halves);   // halves is even
            // prologue turn: S^T_X, dP^T_X of the item's half X
            bool okw = warp_wait(b.fix_full, it & 1, wc, 0x50) &&
                       ring_wait(b.ring_full, g + X, C::kSlots, wc, 0x51);
            if (!turn_begin(okw)) break;
            if (elect_one()) {
                const uint64_t sl = ((g + X) % C::kSlots) * kSlotDesc;
                issue_st_half<D>(t_st, d_k, d_ring_k + sl);
                issue_st_half<D>(t_dpt, d_v, d_ring_k + sl + kHalfDesc);
                mma_commit(b.s_full + 8 * X);
                if (halves <= 2) mma_commit(b.kv_free);   // this issuer's last reader of K, V
            }
            turn_end();
            for (int u = 0; u < halves; ++u) {
                if ((u & 1) != X) continue;   // the other issuer's half (its turn)
                const int gu = g + u;
                const bool next = u + 2 < halves;
                okw = warp_wait(b.p_full + 8 * X, (gu >> 1) & 1, wc, 0x52);
                if (okw && next) okw = ring_wait(b.ring_full, gu + 2, C::kSlots, wc, 0x53);
                // the previous item's dK, dV have been read out of TMEM (the
                // first accumulating MMA of an item is half 0's)
                if (okw && u == 0 && it > 0) okw = warp_wait(b.acc_free, (it - 1) & 1, wc, 0x59);
                if (!turn_begin(okw)) {
                    run = false;
                    break;
                }
                if (elect_one()) {
                    const uint64_t sl = (gu % C::kSlots) * kSlotDesc;
                    const uint32_t acc = u > 0 ? 1u : 0u;
                    issue_acc_half<D>(t_dv, t_st, d_ring_mn + sl + kHalfDesc, acc);   // dV += P^T dO_x
                    issue_acc_half<D>(t_dk, t_dpt, d_ring_mn + sl, acc);              // dK += dS^T Q_x
                    mma_commit(b.ring_empty + 8 * (gu % C::kSlots));
                    if (next) {
                        const uint64_t sn = ((gu + 2) % C::kSlots) * kSlotDesc;
                        issue_st_half<D>(t_st, d_k, d_ring_k + sn);
                        issue_st_half<D>(t_dpt, d_v, d_ring_k + sn + kHalfDesc);
                        mma_commit(b.s_full + 8 * X);
                        if (u + 4 >= halves) mma_commit(b.kv_free);   // this issuer's last reader of K, V
                    } else {
                        mma_commit(b.o_final);   // this issuer's last accumulation of the item
                    }
                }
                turn_end();
            }
            g += halves;
            ++it;
        }
        if (elect_one()) mma_commit(b.drain);
        __syncwarp();
        mbar_drain(b.drain, 0, p.wait_limit_ns);
    } else {
        // ---------------------------------------------- P^T and dS^T
        // Two warpgroups: cw = 0 (warps 0-3) takes the queries 0-31 of each
        // half, cw = 1 (warps 7-10) the queries 32-63; both cover all keys.
        const int cw = warp < kDkEwB ? 0 : 1;
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;        // key within the block (TMEM lane)
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t t_s = tmem + lane_off;
        const uint32_t t_dv = t_s + 2 * kT, t_dk = t_dv + D;
        const float c = p.scale_log2;
        int k = 0, it = 0, g = 0;
        bool ok = true;
        // lanes 0..31 of the quarter-0 warp stage the row statistics of
        // query 32 cw + r of each half, loaded one half ahead (across items:
        // the next item's first half during the current item's last); the
        // loaded values are first used when they are staged, so the load's
        // latency does not hold up the warp (and with it its warpgroup's
        // barrier)
        Seq sq;
        int j0;
        bool have = next_dk_item(p, sched, k, cta, G, D, sq, j0);
        float rl = 0.f, rd = 0.f;
        if (have && r < 32) {
            int i_f, hv;
            dk_rows<WIN>(p, j0, sq.len, i_f, hv);
            const int iq0 = i_f + 32 * cw + r;
            if (iq0 < sq.len) {
                rl = p.lse[sq.stat0 + iq0];
                rd = p.delta[sq.stat0 + iq0];
            }
        }
        while (ok && have) {
            const int n = sq.len;
            int i_first, halves;
            dk_rows<WIN>(p, j0, n, i_first, halves);
            const float *L = p.lse + sq.stat0;
            const float *Dl = p.delta + sq.stat0;
            int iq = i_first + 32 * cw + r;
            // the next item, for its first half's statistics
            Seq sq2;
            int j02;
            const bool have2 = next_dk_item(p, sched, k, cta, G, D, sq2, j02);
            int iq2 = 0;
            if (have2) {
                int i_f2, hv2;
                dk_rows<WIN>(p, j02, sq2.len, i_f2, hv2);
                iq2 = i_f2 + 32 * cw + r;
            }
            for (int u = 0; u < halves; ++u) {
                const int gu = g + u, x = u & 1;
                float *sl = stat + x * 2 * 64, *sd = sl + 64;
                if (r < 32) {
                    sl[32 * cw + r] = iq < n ? rl * kLog2e : INFINITY;
                    sd[32 * cw + r] = iq < n ? rd : 0.f;
                    iq += 64;
                    if (u + 1 < halves) {
                        if (iq < n) {
                            rl = L[iq];
                            rd = Dl[iq];
                        }
                    } else if (have2 && iq2 < sq2.len) {
                        rl = p.lse[sq2.stat0 + iq2];
                        rd = p.delta[sq2.stat0 + iq2];
                    }
                }
                named_bar_sync(cw == 0 ? 1u : 4u, 128);   // this warpgroup's statistics staged
                const uint32_t t_st = t_s + x * 2 * 64, t_dpt = t_st + 64;
                if (!warp_wait(b.s_full + 8 * x, (gu >> 1) & 1, wc, 0x60)) { ok = false; break; }
                tc_fence_after();
                // queries qi of this half that key r sees: qmin <= qi <= qmax.
                // Causal: q >= r, which only the first tile can break; band:
                // key - wr <= q <= key + wl, checked where a half crosses an edge.
                int qmin, qmax;
                bool diag;
                if (WIN) {
                    const int qb = i_first + 64 * u, key = j0 + r;
                    qmin = p.wr >= 0 ? key - p.wr - qb : 0;
                    qmax = p.wl >= 0 ? key + p.wl - qb : 63;
                    diag = __any_sync(0xffffffffu, qmin > 0 || qmax < 63);
                } else {
                    diag = p.causal && u < 2;
                    qmin = r - x * 64;
                    qmax = 63;
                }
                {
                    const int cc = cw;
                    float sv[32], dpv[32];
                    tmem_ld32(t_st + cc * 32, sv);
                    tmem_ld32(t_dpt + cc * 32, dpv);
                    tmem_wait_ld();
                    uint32_t pk[16], dk[16];
                    const float2 c2 = make_float2(c, c);
#pragma unroll
                    for (int e = 0; e < 32; e += 4) {
                        const int qi = cc * 32 + e;              // query within the half
                        // the statistics of four queries: one 16-byte broadcast load each
                        const float4 l4 = *reinterpret_cast<const float4 *>(sl + qi);
                        const float4 d4 = *reinterpret_cast<const float4 *>(sd + qi);
                        const float2 a0 = __ffma2_rn(make_float2(sv[e], sv[e + 1]), c2, make_float2(-l4.x, -l4.y));
                        const float2 a1 = __ffma2_rn(make_float2(sv[e + 2], sv[e + 3]), c2, make_float2(-l4.z, -l4.w));
                        float2 p0 = make_float2(ex2_approx(a0.x), ex2_approx(a0.y));
                        float2 p1 = make_float2(ex2_approx(a1.x), ex2_approx(a1.y));
                        if (diag) {
                            if (qi < qmin || qi > qmax) p0.x = 0.f;
                            if (qi + 1 < qmin || qi + 1 > qmax) p0.y = 0.f;
                            if (qi + 2 < qmin || qi + 2 > qmax) p1.x = 0.f;
                            if (qi + 3 < qmin || qi + 3 > qmax) p1.y = 0.f;
                        }
                        const float2 g0 = __fmul2_rn(p0, __fadd2_rn(make_float2(dpv[e], dpv[e + 1]), make_float2(-d4.x, -d4.y)));
                        const float2 g1 = __fmul2_rn(p1, __fadd2_rn(make_float2(dpv[e + 2], dpv[e + 3]), make_float2(-d4.z, -d4.w)));
                        pk[e / 2] = pack_bf16x2(p0.x, p0.y);
                        pk[e / 2 + 1] = pack_bf16x2(p1.x, p1.y);
                        dk[e / 2] = pack_bf16x2(g0.x, g0.y);
                        dk[e / 2 + 1] = pack_bf16x2(g1.x, g1.y);
                    }
                    tmem_st16(t_st + cc * 32, pk);    // P^T over S^T columns this warpgroup has read
                    tmem_st16(t_dpt + cc * 32, dk);   // dS^T over dP^T columns this warpgroup has read
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(b.p_full + 8 * x);
            }
            if (!ok) break;
            if (!warp_wait(b.o_final, it & 1, wc, 0x61)) break;
            tc_fence_after();
            const int key = j0 + r;
            Tout *dV = static_cast<Tout *>(p.dv) + sq.elem0 + key * sq.rstride;
            Tout *dK = static_cast<Tout *>(p.dk) + sq.elem0 + key * sq.rstride;
            // warpgroup 0 stores dV, warpgroup 1 dK
            const uint32_t t_acc = cw == 0 ? t_dv : t_dk;
            Tout *const dst = cw == 0 ? dV : dK;
            const float mul = cw == 0 ? 1.f : p.scale;
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
                float xo[32];
                tmem_ld32(t_acc + cc * 32, xo);
                tmem_wait_ld();
                if (key < n) store_row(dst + cc * 32, xo, mul);
            }
            // dK, dV are out of TMEM: the next item may overwrite them
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(b.acc_free);
            g += halves;
            ++it;
            sq = sq2;
            j0 = j02;
            have = have2;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kDkMmaWarpA) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------- dQ --
// Q and dO stay in shared memory; K_j and V_j stream through a ring of
// kSlots single-tile slots (loads K_0, V_0, K_1, V_1, ...), V_j released
// after dP_j, K_j after dQ's use of it.  Two TMEM buffers hold S (the
// softmax warps write dS over it), one holds dP.  Per tile t the MMA warp
// issues, once dS_t is ready (D = 128, causal or full):
//   S_{t+1} = Q K_{t+1}^T     (into dS_{t-1}'s buffer, which dQ has read)
//   dP_{t+1} = dO V_{t+1}^T   (the dP buffer has been read)
//   dQ += dS_t K_t
// so the softmax warps' next inputs come first.  D = 64 and the band
// instantiation keep S two tiles ahead instead: dP_{t+1}, dQ_t, then
// S_{t+2} into dS_t's buffer (measured faster there).  Persistent like the dK/dV kernel: Q
// and dO are reloaded once the item's last dP is issued, the next item's
// first S, dP run during the previous epilogue, and its first dQ MMA waits
// for that epilogue to have read dQ.
template <int D>
struct DqCfg {
    static constexpr int kTileBytes = kT * D * 2;
    static constexpr int kSlots = D == 128 ? 5 : 10;
    // D = 128: K_t is loaded twice, for S_t and for dQ_t, rather than held
    // from one to the other (see the producer).  D = 64 has slots to spare.
    static constexpr bool kReloadK = D == 128;
    static constexpr int kRingOff = 2 * kTileBytes;
    static constexpr int kBarOff = kRingOff + kSlots * kTileBytes;
    static constexpr int kBarBytes = 256;
    static constexpr int kSchedOff = kBarOff + kBarBytes;   // packed-batch walk table
    static constexpr int kSmemBytes = kSchedOff + kBwdSchedBytes + 1024;
    static_assert(kSmemBytes <= 232448, "shared memory per CTA");
    static_assert(8 * (2 + 2 * kSlots + 7) + 16 <= kBarBytes, "barrier area");
    static_assert(3 * kT + D <= (int)kTmemCols, "TMEM columns");
};

// The CTA's next dQ work item: query block first (highest first: under the
// causal mask it has the most keys), then problem; snake over CTAs.
__device__ __forceinline__ bool next_dq_item(const BwdTcParams &p, const BwdSched &sc, int &k, int cta, int G,
                                             int D, Seq &sq, int &ib) {
    if (p.compact) {  // query block from the last (most keys under the causal mask) down
        const int items = sc.per_head * p.heads;
        for (; k * G < items; ++k) {
            const int idx = k * G + ((k & 1) ? (G - 1 - cta) : cta);
            int unit, blk;
            if (idx >= items || !bwd_decode_compact(p, sc, idx, true, unit, blk)) continue;
            sq = seq_of(p, unit, D);
            ib = blk;
            if (ib * kT < sq.len) {
                ++k;
                return true;
            }
        }
        return false;
    }
    const int items = p.nblk * p.units;
    for (; k * G < items; ++k) {
        const int idx = k * G + ((k & 1) ? (G - 1 - cta) : cta);
        if (idx >= items) continue;
        ib = p.nblk - 1 - idx / p.units;
        sq = seq_of(p, idx % p.units, D);
        if (ib * kT < sq.len) {
            ++k;
            return true;
        }
    }
    return false;
}

// Key tiles a dQ item walks: [t_lo, t_lo + tiles) covers every key that
// some row of the block [128 ib, 128 ib + 128) sees.
template <bool WIN>
__device__ __forceinline__ void dq_tiles(const BwdTcParams &p, int ib, int len, int &t_lo, int &tiles) {
    const int key_tiles = (len + kT - 1) / kT;
    t_lo = 0;
    tiles = p.causal ? min(ib + 1, key_tiles) : key_tiles;
    if (WIN) {
        const int i0 = ib * kT, il = min(len, i0 + kT) - 1;
        const int lo = p.wl >= 0 ? max(0, i0 - p.wl) : 0;
        const int hi = p.wr >= 0 ? min(len - 1, il + p.wr) : len - 1;
        t_lo = lo / kT;
        tiles = hi / kT + 1 - t_lo;
    }
}

// dQ (TMEM, 128 x D fp32) (+)= dS (TMEM, 128 x 128 bf16) * K (smem, 128 x D,
// MN-major): as issue_pv, but dS's keys 64 c .. 64 c + 63 (bf16 pairs) sit at
// columns 64 c .. 64 c + 31, over the score columns dS warpgroup c has read.
template <int D>
__device__ __forceinline__ void issue_dq(uint32_t d_tmem, uint32_t a_tmem, uint64_t dk, uint32_t accumulate) {
    constexpr uint32_t idesc = idesc_bf16(kTcRows, D, 1);
#pragma unroll
    for (int kk = 0; kk < kTcRows / 16; ++kk)
        mma_ts(d_tmem, a_tmem + (kk >> 2) * 64 + (kk & 3) * 8, dk + (uint64_t)((kk * 2048) >> 4), idesc,
               (kk > 0 || accumulate) ? 1u : 0u);
}

template <int D, typename Tout, bool WIN>
__global__ void __launch_bounds__(kDqThreads, 1)
    bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                     const BwdTcParams p) {
    using C = DqCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const uint32_t bars = base + C::kBarOff;
    const uint32_t fix_full = bars, qd_free = bars + 8, kv_full = bars + 16, kv_empty = kv_full + 8 * C::kSlots;
    // s_full[2]: S of tile g ready in TMEM buffer g & 1 (phase (g >> 1) & 1);
    // dp_full: dP of tile g ready (phase g & 1).  Separate barriers let the dS
    // step compute P from S while dP is still being computed.
    const uint32_t s_full = kv_empty + 8 * C::kSlots, dp_full = s_full + 16, ds_full = dp_full + 8;
    const uint32_t o_final = ds_full + 8;
    const uint32_t acc_free = o_final + 8, drain = acc_free + 8;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + C::kBarOff + C::kBarBytes - 16);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(gbase + C::kBarOff + C::kBarBytes - 8);
    volatile int *stop_flag = reinterpret_cast<volatile int *>(gbase + C::kBarOff + C::kBarBytes - 12);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x, G = gridDim.x;

    if (warp == kProdWarp && lane == 0) {
        *stop_flag = 0;
        mbar_init(fix_full, 1);
        mbar_init(qd_free, 1);
        for (int i = 0; i < C::kSlots; ++i) {
            mbar_init(kv_full + 8 * i, 1);
            mbar_init(kv_empty + 8 * i, 1);
        }
        mbar_init(s_full, 1);
        mbar_init(s_full + 8, 1);
        mbar_init(dp_full, 1);
        mbar_init(ds_full, 8);   // both dS warpgroups
        mbar_init(o_final, 1);
        mbar_init(acc_free, 8);
        mbar_init(drain, 1);
        fence_barrier_init();
        *abort_flag = 0;
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_do);
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    // the packed-batch walk table (scratch: the not yet used ring)
    uint8_t *sched_tab = gbase + C::kSchedOff;
    if (p.compact) build_bwd_sched(p, sched_tab, reinterpret_cast<int *>(gbase + C::kRingOff));
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const BwdSched sched = bwd_sched(p, sched_tab);
    const uint32_t tmem = *tmem_slot;
    const WaitCtx wc{p.err, abort_flag, p.wait_limit_ns};
    const uint32_t ring = base + C::kRingOff;

    if (warp == kProdWarp) {
        // ---------------------------------------------------- producer
        if (lane == 0) {
            int k = 0, it = 0, ib;
            uint32_t li = 0;          // ring loads issued
            bool ok = true;
            Seq sq;
            while (ok && next_dq_item(p, sched, k, cta, G, D, sq, ib)) {
                int t_lo, tiles;
                dq_tiles<WIN>(p, ib, sq.len, t_lo, tiles);
                if (it > 0 && !mbar_wait(qd_free, (it - 1) & 1, wc, 0x43)) break;
                mbar_arrive_expect_tx(fix_full, 2 * C::kTileBytes);
                load_rows<D>(base, &tm_q, fix_full, ib * kT, sq, p.varlen, kTcAtomBytes);
                load_rows<D>(base + C::kTileBytes, &tm_do, fix_full, ib * kT, sq, p.varlen, kTcAtomBytes);
                ++it;
                // kReloadK: one reader per ring load, in the order the MMA warp
                // reads them: K_0 (S_0), V_0 (dP_0), K_1 (S_1), then per tile t:
                // V_{t+1} (dP_{t+1}), K_t again (dQ_t), K_{t+2} (S_{t+2}).  Held
                // from S_t to dQ_t instead, three K tiles and a V tile fill four of
                // the five 32 KB slots at D = 128, and the next loads wait for
                // slots.  Otherwise K_j, V_j in turn, K_j read by S_j and dQ_j.
                auto load = [&](int kv, int j) -> bool {
                    const uint32_t slot = li % C::kSlots, round = li / C::kSlots;
                    if (round > 0 && !mbar_wait(kv_empty + 8 * slot, (round - 1) & 1, wc, 0x42)) return false;
                    mbar_arrive_expect_tx(kv_full + 8 * slot, C::kTileBytes);
                    load_rows<D>(ring + slot * C::kTileBytes, kv == 0 ? &tm_k : &tm_v, kv_full + 8 * slot,
                                 (t_lo + j) * kT, sq, p.varlen, kTcAtomBytes);
                    ++li;
                    return true;
                };
                if (C::kReloadK) {
                    ok = load(0, 0) && load(1, 0) && (tiles < 2 || load(0, 1));
                    for (int t = 0; ok && t < tiles; ++t)
                        ok = (t + 1 >= tiles || load(1, t + 1)) && load(0, t) && (t + 2 >= tiles || load(0, t + 2));
                } else {
                    for (int j = 0; ok && j < tiles; ++j) ok = load(0, j) && load(1, j);
                }
            }
            const uint64_t lim = p.wait_limit_ns;
            if (it > 0) mbar_drain(fix_full, (it - 1) & 1, lim);
            for (uint32_t u = li > (uint32_t)C::kSlots ? li - C::kSlots : 0; u < li; ++u)
                mbar_drain(kv_full + 8 * (u % C::kSlots), (u / C::kSlots) & 1, lim);
        }
    } else if (warp == kMmaWarp || warp == kDqWaitWarp) {
        // --------------------------------------------------------- MMA
        // Warp 5 issues; warp 10 runs the same walk but only waits: for each
        // issue step it waits for that step's barriers (ring loads, dS, the
        // previous item's dQ read) while warp 5 is still issuing the step
        // before, then both meet at named barrier kDqGo and warp 5 issues.
        // The waits (each costs the issuer a few hundred cycles when the dS
        // warps of its sub-partition are busy) thus overlap the MMAs.  A
        // wait that gives up raises the stop flag before the meeting.
        const bool issuer = warp == kMmaWarp;
        auto go = [&](bool waits_ok) -> bool {
            if (!waits_ok) *stop_flag = 1;
            __syncwarp();
            named_bar_sync(kDqGo, 64);
            if (*stop_flag) return false;
            if (issuer) tc_fence_after();
            return true;
        };
        constexpr uint64_t kTileDesc = C::kTileBytes >> 4;
        const uint64_t d_q = smem_desc(base, 16, 1024), d_do = d_q + kTileDesc;
        const uint64_t d_ring_k = smem_desc(ring, 16, 1024);
        const uint64_t d_ring_mn = smem_desc(ring, kTcAtomBytes, 1024);
        const uint32_t t_dp = tmem + 2 * kT, t_dq = tmem + 3 * kT;
        int k = 0, it = 0, ib;
        uint32_t lb = 0, gt = 0;      // ring loads and tiles of earlier items
        bool ok = true;
        Seq sq;
        while (ok && next_dq_item(p, sched, k, cta, G, D, sq, ib)) {
            int t_lo, tiles;
            dq_tiles<WIN>(p, ib, sq.len, t_lo, tiles);
            // Ring loads in the producer's order: K_0 = lb, V_0 = lb + 1;
            // then per tile t: K_{t+1}, V_{t+1}, K_t again (kReloadK, one
            // reader each; the same sequence as the producer's K_1 | V_1, K_0,
            // K_2 | ...), or K_j = lb + 2j, V_j = lb + 2j + 1.  Tile t uses S
            // buffer (gt + t) & 1.
            uint32_t cur = lb;
            const uint32_t ls0 = cur++, lv0 = cur++;
            if (!go(issuer || (warp_wait(fix_full, it & 1, wc, 0x54) && ring_wait(kv_full, ls0, C::kSlots, wc, 0x55) &&
                               ring_wait(kv_full, lv0, C::kSlots, wc, 0x55))))
                break;
            if (issuer && elect_one()) {
                issue_qk<D>(tmem + (gt & 1) * kT, d_q, d_ring_k + (ls0 % C::kSlots) * kTileDesc);  // S_0
                mma_commit(s_full + 8 * (gt & 1));
                if (C::kReloadK) mma_commit(kv_empty + 8 * (ls0 % C::kSlots));
                issue_qk<D>(t_dp, d_do, d_ring_k + (lv0 % C::kSlots) * kTileDesc);                 // dP_0
                mma_commit(dp_full);
                mma_commit(kv_empty + 8 * (lv0 % C::kSlots));                                    // V_0 read
                if (tiles == 1) mma_commit(qd_free);                                            // Q, dO read
            }
            __syncwarp();
            if constexpr (!C::kReloadK) {
                // D = 64: S computed two tiles ahead.  Per tile t, once dS_t is
                // in: dP_{t+1}, dQ_t, then S_{t+2} into dS_t's buffer (after dQ_t
                // has read it, in order).  (The order of the D = 128 branch
                // measured 8% slower here.)
                if (tiles > 1) {
                    const uint32_t ls1 = lb + 2;
                    if (!go(issuer || ring_wait(kv_full, ls1, C::kSlots, wc, 0x55))) break;
                    if (issuer && elect_one()) {
                        issue_qk<D>(tmem + ((gt + 1) & 1) * kT, d_q, d_ring_k + (ls1 % C::kSlots) * kTileDesc);
                        mma_commit(s_full + 8 * ((gt + 1) & 1));                                // S_1
                    }
                    __syncwarp();
                }
                for (int t = 0; t < tiles; ++t) {
                    const uint32_t g = gt + t;
                    const uint32_t t_buf = tmem + (g & 1) * kT;
                    const uint32_t lk = lb + 2 * t, lvn = lk + 3, lk2 = lk + 4;   // K_t, V_{t+1}, K_{t+2}
                    bool okw = true;
                    if (!issuer) {
                        okw = (t + 1 >= tiles || ring_wait(kv_full, lvn, C::kSlots, wc, 0x57)) &&
                              ring_wait(kv_full, lk, C::kSlots, wc, 0x57) &&
                              (t + 2 >= tiles || ring_wait(kv_full, lk2, C::kSlots, wc, 0x58)) &&
                              warp_wait(ds_full, g & 1, wc, 0x56) &&
                              // the previous item's dQ has been read out of TMEM
                              (t != 0 || it == 0 || warp_wait(acc_free, (it - 1) & 1, wc, 0x5a));
                    }
                    if (!go(okw)) { ok = false; break; }
                    if (issuer && elect_one() && t + 1 < tiles) {
                        issue_qk<D>(t_dp, d_do, d_ring_k + (lvn % C::kSlots) * kTileDesc);   // dP_{t+1}
                        mma_commit(dp_full);
                        mma_commit(kv_empty + 8 * (lvn % C::kSlots));
                        if (t + 2 == tiles) mma_commit(qd_free);                           // Q, dO read
                    }
                    __syncwarp();
                    if (issuer && elect_one()) {
                        issue_dq<D>(t_dq, t_buf, d_ring_mn + (lk % C::kSlots) * kTileDesc, t > 0 ? 1u : 0u);
                        mma_commit(kv_empty + 8 * (lk % C::kSlots));                           // K_t read
                    }
                    __syncwarp();
                    if (t + 2 < tiles) {
                        if (issuer && elect_one()) {
                            issue_qk<D>(t_buf, d_q, d_ring_k + (lk2 % C::kSlots) * kTileDesc);  // S_{t+2}
                            mma_commit(s_full + 8 * (g & 1));
                        }
                        __syncwarp();
                    }
                }
            } else if constexpr (WIN) {
                // D = 128, band: S computed two tiles ahead, each tile in two
                // issue steps (the order below measured 9% slower here).
                if (tiles > 1) {
                    const uint32_t ls1 = cur++;
                    if (!go(issuer || ring_wait(kv_full, ls1, C::kSlots, wc, 0x55))) break;
                    if (issuer && elect_one()) {
                        issue_qk<D>(tmem + ((gt + 1) & 1) * kT, d_q, d_ring_k + (ls1 % C::kSlots) * kTileDesc);
                        mma_commit(s_full + 8 * ((gt + 1) & 1));                                    // S_1
                        mma_commit(kv_empty + 8 * (ls1 % C::kSlots));
                    }
                    __syncwarp();
                }
                for (int t = 0; t < tiles; ++t) {
                    const uint32_t g = gt + t;
                    const uint32_t t_buf = tmem + (g & 1) * kT;
                    // V_{t+1}, K_t again (for dQ_t), K_{t+2}
                    const uint32_t lvn = t + 1 < tiles ? cur++ : 0u;
                    const uint32_t lk = cur++;
                    const uint32_t lk2 = t + 2 < tiles ? cur++ : 0u;
                    // Step 1: dP_{t+1} and dQ_t, once V_{t+1}, K_t and dS_t are in.
                    // Step 2: S_{t+2}, once K_{t+2} is in.  K_{t+2}'s load is the
                    // block's last, into the slot that the previous block's dP
                    // freed, so waiting for it only after step 1 lets dP_{t+1}
                    // start as soon as dS_t is in.
                    bool okw = true;
                    if (!issuer) {
                        okw = (t + 1 >= tiles || ring_wait(kv_full, lvn, C::kSlots, wc, 0x57)) &&
                              ring_wait(kv_full, lk, C::kSlots, wc, 0x57) &&
                              warp_wait(ds_full, g & 1, wc, 0x56) &&
                              // the previous item's dQ has been read out of TMEM
                              (t != 0 || it == 0 || warp_wait(acc_free, (it - 1) & 1, wc, 0x5a));
                    }
                    if (!go(okw)) { ok = false; break; }
                    if (issuer && elect_one() && t + 1 < tiles) {
                        issue_qk<D>(t_dp, d_do, d_ring_k + (lvn % C::kSlots) * kTileDesc);   // dP_{t+1}
                        mma_commit(dp_full);
                        mma_commit(kv_empty + 8 * (lvn % C::kSlots));
                        if (t + 2 == tiles) mma_commit(qd_free);                           // Q, dO read
                    }
                    __syncwarp();
                    if (issuer && elect_one()) {
                        issue_dq<D>(t_dq, t_buf, d_ring_mn + (lk % C::kSlots) * kTileDesc, t > 0 ? 1u : 0u);
                        mma_commit(kv_empty + 8 * (lk % C::kSlots));                           // K_t read
                    }
                    __syncwarp();
                    if (t + 2 < tiles) {
                        if (!go(issuer || ring_wait(kv_full, lk2, C::kSlots, wc, 0x58))) { ok = false; break; }
                        if (issuer && elect_one()) {
                            // S_{t+2} overwrites dS_t's buffer after dQ_t has read it (in order)
                            issue_qk<D>(t_buf, d_q, d_ring_k + (lk2 % C::kSlots) * kTileDesc);  // S_{t+2}
                            mma_commit(s_full + 8 * (g & 1));
                            mma_commit(kv_empty + 8 * (lk2 % C::kSlots));
                        }
                        __syncwarp();
                    }
                }
            } else {
                // D = 128, causal or full:
                for (int t = 0; t < tiles; ++t) {
                    const uint32_t g = gt + t;
                    const uint32_t t_buf = tmem + (g & 1) * kT;                 // dS_t
                    const uint32_t t_nxt = tmem + ((g + 1) & 1) * kT;           // S_{t+1}
                    // K_{t+1} (for S_{t+1}), V_{t+1}, K_t again (for dQ_t)
                    const uint32_t lkn = t + 1 < tiles ? cur++ : 0u;
                    const uint32_t lvn = t + 1 < tiles ? cur++ : 0u;
                    const uint32_t lk = cur++;
                    // One issue block per key tile: S_{t+1}, dP_{t+1}, dQ_t.
                    // S_{t+1} goes into the buffer that dQ_{t-1} has read (issued
                    // before it, in order), so it needs no more than its K; the
                    // block waits for dS_t (dP_{t+1} overwrites the dP that the dS
                    // step read, dQ_t reads dS_t).  The three loads are the block's
                    // share of the ring in load order, all issued a block earlier.
                    bool okw = true;
                    if (!issuer) {
                        okw = (t + 1 >= tiles || (ring_wait(kv_full, lkn, C::kSlots, wc, 0x57) &&
                                                  ring_wait(kv_full, lvn, C::kSlots, wc, 0x57))) &&
                              ring_wait(kv_full, lk, C::kSlots, wc, 0x58) &&
                              warp_wait(ds_full, g & 1, wc, 0x56) &&
                              // the previous item's dQ has been read out of TMEM
                              (t != 0 || it == 0 || warp_wait(acc_free, (it - 1) & 1, wc, 0x5a));
                    }
                    if (!go(okw)) { ok = false; break; }
                    if (issuer && elect_one() && t + 1 < tiles) {
                        issue_qk<D>(t_nxt, d_q, d_ring_k + (lkn % C::kSlots) * kTileDesc);   // S_{t+1}
                        mma_commit(s_full + 8 * ((g + 1) & 1));
                        mma_commit(kv_empty + 8 * (lkn % C::kSlots));
                        issue_qk<D>(t_dp, d_do, d_ring_k + (lvn % C::kSlots) * kTileDesc);   // dP_{t+1}
                        mma_commit(dp_full);
                        mma_commit(kv_empty + 8 * (lvn % C::kSlots));
                        if (t + 2 == tiles) mma_commit(qd_free);                           // Q, dO read
                    }
                    __syncwarp();
                    if (issuer && elect_one()) {
                        issue_dq<D>(t_dq, t_buf, d_ring_mn + (lk % C::kSlots) * kTileDesc, t > 0 ? 1u : 0u);
                        mma_commit(kv_empty + 8 * (lk % C::kSlots));                           // K_t read
                    }
                    __syncwarp();
                }
            }
            if (!ok) break;
            if (issuer && elect_one()) mma_commit(o_final);
            __syncwarp();
            lb = C::kReloadK ? cur : lb + 2 * tiles;
            gt += tiles;
            ++it;
        }
        if (issuer) {
            // Teardown: wait for every MMA issued so far before TMEM is freed.
            if (elect_one()) mma_commit(drain);
            __syncwarp();
            mbar_drain(drain, 0, p.wait_limit_ns);
        }
    } else {
        // ------------------------------------------------------- dS
        // Two warpgroups: cw = 0 (warps 0-3) takes keys 0-63 of each tile,
        // cw = 1 (warps 6-9) keys 64-127; both cover all query rows.
        const int cw = warp < kDqEwB ? 0 : 1;
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;        // query row within the block (TMEM lane)
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t t_s0 = tmem + lane_off, t_dp = t_s0 + 2 * kT, t_dq = t_s0 + 3 * kT;
        const float c = p.scale_log2;
        constexpr int kH = kT / 2;                // keys per warpgroup
        int k = 0, it = 0, ib;
        uint32_t gt = 0;
        bool ok = true;
        Seq sq;
        while (ok && next_dq_item(p, sched, k, cta, G, D, sq, ib)) {
            const int n = sq.len;
            int t_lo, tiles;
            dq_tiles<WIN>(p, ib, n, t_lo, tiles);
            const int row = ib * kT + r;
            const float lrow = row < n ? p.lse[sq.stat0 + row] * kLog2e : INFINITY;
            const float drow = row < n ? p.delta[sq.stat0 + row] : 0.f;
            // keys outside [lim_lo, lim): past the causal diagonal, outside the
            // band or past the end
            int lim = p.causal ? min(row + 1, n) : n, lim_lo = 0;
            if (WIN) {
                lim = p.wr >= 0 ? min(row + p.wr + 1, n) : n;
                lim_lo = p.wl >= 0 ? row - p.wl : 0;
            }
            for (int t = 0; t < tiles; ++t) {
                const uint32_t g = gt + t;
                const uint32_t t_s = t_s0 + (g & 1) * kT + cw * kH;   // this warpgroup's keys
                if (!warp_wait(s_full + 8 * (g & 1), (g >> 1) & 1, wc, 0x70)) { ok = false; break; }
                tc_fence_after();
                const int key0 = (t_lo + t) * kT + cw * kH;
                const bool need_mask = key0 + kH > lim || (WIN && key0 < lim_lo);
                // P = exp2(S c - L) for the warpgroup's keys while dP may still be computed
                float pv[kH];
#pragma unroll
                for (int cc = 0; cc < kH / 32; ++cc) tmem_ld32(t_s + cc * 32, pv + cc * 32);
                tmem_wait_ld();
                const float2 c2 = make_float2(c, c), nl2 = make_float2(-lrow, -lrow);
                const float2 nd2 = make_float2(-drow, -drow);
#pragma unroll
                for (int x = 0; x < kH; x += 2) {
                    const float2 a = __ffma2_rn(make_float2(pv[x], pv[x + 1]), c2, nl2);
                    float2 pp = make_float2(ex2_approx(a.x), ex2_approx(a.y));
                    if (need_mask) {
                        const int key = key0 + x;
                        if (key >= lim || (WIN && key < lim_lo)) pp.x = 0.f;
                        if (key + 1 >= lim || (WIN && key + 1 < lim_lo)) pp.y = 0.f;
                    }
                    pv[x] = pp.x;
                    pv[x + 1] = pp.y;
                }
                if (!warp_wait(dp_full, g & 1, wc, 0x72)) { ok = false; break; }
                tc_fence_after();
#pragma unroll
                for (int cc = 0; cc < kH / 32; ++cc) {
                    float dpv[32];
                    tmem_ld32(t_dp + cw * kH + cc * 32, dpv);
                    tmem_wait_ld();
                    uint32_t dk[16];
#pragma unroll
                    for (int x = 0; x < 32; x += 2) {
                        const float2 pp = make_float2(pv[cc * 32 + x], pv[cc * 32 + x + 1]);
                        const float2 gg = __fmul2_rn(pp, __fadd2_rn(make_float2(dpv[x], dpv[x + 1]), nd2));
                        dk[x / 2] = pack_bf16x2(gg.x, gg.y);
                    }
                    tmem_st16(t_s + cc * 16, dk);    // dS over S columns this warpgroup has read
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(ds_full);
            }
            if (!ok) break;
            if (!warp_wait(o_final, it & 1, wc, 0x71)) break;
            tc_fence_after();
            // each warpgroup stores half of the row's dQ columns
            Tout *dQ = static_cast<Tout *>(p.dq) + sq.elem0 + row * sq.rstride + cw * (D / 2);
#pragma unroll
            for (int cc = 0; cc < D / 64; ++cc) {
                float x[32];
                tmem_ld32(t_dq + cw * (D / 2) + cc * 32, x);
                tmem_wait_ld();
                if (row < n) store_row(dQ + cc * 32, x, p.scale);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_free);
            gt += tiles;
            ++it;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <typename K>
fa_status prepare(K kernel, int smem, int threads) {
    cudaFuncAttributes a;
    cudaError_t e = cudaFuncGetAttributes(&a, kernel);
    if (e != cudaSuccess) return fa_cuda_fail(e);
    if (a.maxThreadsPerBlock < threads) return fa_cuda_fail(cudaErrorLaunchOutOfResources);
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    return e == cudaSuccess ? FA_OK : fa_cuda_fail(e);
}

template <int D, typename Tout, bool WIN>
fa_status launch(const FaBwdProblem &p) {
    // dense: dims {D, N, B*H}, a box is {64, rows, 1}; packed: dims
    // {D, H, total}, a box is {64, 1, rows}
    CUtensorMap tq, tk, tv, tdo, tq64, tdo64;
    const uint64_t rb = (uint64_t)D * 2;
    const uint64_t d1 = p.varlen ? (uint64_t)p.heads : (uint64_t)p.n;
    const uint64_t d2 = p.varlen ? (uint64_t)p.total : (uint64_t)p.units_bh;
    const uint64_t s2 = d1 * rb;
    auto map = [&](CUtensorMap *m, const void *ptr, uint32_t rows) {
        return p.varlen ? make_map(m, ptr, D, d1, d2, rb, s2, 1, rows) : make_map(m, ptr, D, d1, d2, rb, s2, rows, 1);
    };
    if (!map(&tq, p.q, kT) || !map(&tk, p.k, kT) || !map(&tv, p.v, kT) || !map(&tdo, p.dout, kT) ||
        !map(&tq64, p.q, 64) || !map(&tdo64, p.dout, 64))
        return FA_ERR_CUDA;
    BwdTcParams k;
    k.lse = p.lse;
    k.delta = p.delta;
    k.dq = p.dq;
    k.dk = p.dk;
    k.dv = p.dv;
    k.cu = p.cu_seqlens;
    k.units = p.units_bh;
    k.varlen = p.varlen;
    k.heads = p.heads;
    k.total = p.total;
    k.n = p.n;
    k.nblk = (p.n + kT - 1) / kT;
    k.scale = p.scale;
    k.scale_log2 = p.scale * kLog2e;
    k.causal = p.causal;
    k.wl = p.wl;
    k.wr = p.wr;
    k.err = p.err;
    k.wait_limit_ns = p.wait_limit_ns;
    // Packed batches of few sequences walk the compact order, heads in groups
    // whose streamed operands (Q and dO, or K and V: the same size) fit
    // kBwdL2GroupBytes.
    k.num_seqs = p.varlen ? p.num_seqs : 0;
    k.compact = p.varlen && p.num_seqs <= kMaxBwdSchedSeqs && k.nblk <= kMaxBwdSchedLevels;
    {
        const double per_head = (double)p.total * D * 2 * 2;
        long long hg = per_head > 0 ? (long long)(kBwdL2GroupBytes / per_head) : p.heads;
        hg = hg < 1 ? 1 : (hg > p.heads ? p.heads : hg);
        k.head_group = (int)((p.heads + hg - 1) / hg);   // groups of at most hg heads, near-equal
    }
    const long long grid = (long long)k.nblk * p.units_bh;
    if (grid > INT32_MAX) return FA_ERR_UNSUPPORTED;
    static FaCtxSet ready;  // contexts set up for this instantiation
    const fa_status su = fa_once_per_context(ready, []() -> fa_status {
        const fa_status st = prepare(bwd_dkdv_tc_kernel<D, Tout, WIN>, DkCfg<D>::kSmemBytes, kDkThreads);
        return st == FA_OK ? prepare(bwd_dq_tc_kernel<D, Tout, WIN>, DqCfg<D>::kSmemBytes, kDqThreads) : st;
    });
    if (su != FA_OK) return su;
    int grid_dk = p.grid_ctas > 0 ? p.grid_ctas : num_sms();   // persistent: one CTA per SM
    if (grid_dk <= 0) return FA_ERR_CUDA;
    if (grid_dk > grid) grid_dk = (int)grid;
    bwd_dkdv_tc_kernel<D, Tout, WIN><<<grid_dk, kDkThreads, DkCfg<D>::kSmemBytes, p.stream>>>(tq64, tk, tv, tdo64,
                                                                                         k);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fa_cuda_fail(e);
    bwd_dq_tc_kernel<D, Tout, WIN><<<grid_dk, kDqThreads, DqCfg<D>::kSmemBytes, p.stream>>>(tq, tk, tv, tdo, k);
    e = cudaGetLastError();
    return e == cudaSuccess ? FA_OK : fa_cuda_fail(e);
}

}  // namespace
}  // namespace fa

fa_status fa_bwd_tc_supports(const FaBwdProblem &p) {
    if (p.dtype != FA_BF16 && p.dtype != FA_BF16_OUT_F32) return FA_ERR_UNSUPPORTED;
    if (p.D != 64 && p.D != 128) return FA_ERR_UNSUPPORTED;
    // one CTA-sized block per 128 keys (or rows) of every problem, counted in 32 bits
    if (p.n < 0 || p.units_bh < 0 || (int64_t)((p.n + fa::kT - 1) / fa::kT) * p.units_bh > INT32_MAX)
        return FA_ERR_UNSUPPORTED;
    return FA_OK;
}

fa_status fa_launch_bwd_tc(const FaBwdProblem &p) {
    const fa_status sup = fa_bwd_tc_supports(p);
    if (sup != FA_OK) return sup;
    if ((int64_t)p.units_bh * p.n == 0) return FA_OK;
    const bool f32 = p.dtype == FA_BF16_OUT_F32;
    // the band instantiation serves windows other than causal (-1, 0) and full (-1, -1)
    const bool win = p.wl >= 0 || p.wr > 0;
    if (p.D == 64) {
        if (win) return f32 ? fa::launch<64, float, true>(p) : fa::launch<64, __nv_bfloat16, true>(p);
        return f32 ? fa::launch<64, float, false>(p) : fa::launch<64, __nv_bfloat16, false>(p);
    }
    if (win) return f32 ? fa::launch<128, float, true>(p) : fa::launch<128, __nv_bfloat16, true>(p);
    return f32 ? fa::launch<128, float, false>(p) : fa::launch<128, __nv_bfloat16, false>(p);
}
