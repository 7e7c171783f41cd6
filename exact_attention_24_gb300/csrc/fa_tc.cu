// Tensor-core (tcgen05 + TMA + TMEM) FlashAttention-2 forward kernel for
// sm_103a, bf16 inputs, fp32 accumulation.
//
// What it computes is the tiled loop of "FlashAttention -- for programmers,
// not researchers.", STAGE 4 (Q row blocks outside, K/V column blocks
// inside, running max m / sum l / unnormalised output carried per row, l
// AND the output rescaled when m moves, one division by l at the end), with
// the scale applied after the dot product and L = m + ln l written next to O
// ("Kernel visualization: Flash Attention 2", sections "Iteration j = 0" and
// "Write the data back to HBM").  Work units are independent (the section
// "Same operations in another block"), so a persistent grid walks them.
//
// How it maps onto GB300 (one CTA per SM, 11 warps):
//   warps 0-3  softmax for query tile 0 (rows 0..127 of the CTA's block;
//              TMEM lanes 0..127, one row per thread)
//   warps 4-7  softmax for query tile 1 (rows 128..255)
//   warp 8     TMA producer: Q tiles once per block, then K_j, V_j tiles
//              through an NSLOT-deep ring of shared-memory slots guarded by
//              full/empty mbarriers
//   warps 9-10 MMA issuers, one per query tile s (one elected thread each;
//              warp 9 also allocates TMEM), taking turns through a token:
//                S_s = Q_s K_j^T          tcgen05.mma, A and B in smem
//                O_s (+)= P_s V_j         tcgen05.mma, A (=P, bf16) in TMEM
// TMEM (512 columns): S_0 [0,128), S_1 [128,256), O_0 [256,256+D),
// O_1 [256+D, 256+2D).  P_s (bf16, packed 2 per column) overwrites the first
// 64 columns of S_s after the softmax has read S_s into registers.
//
// The two query tiles ping-pong: while the softmax warps of one tile work
// on S, the tensor core runs the other tile's P V and next Q K^T.
//
// Online softmax details (all per row, in registers of the row's thread):
//   scores stay unscaled; exponentials are exp2(S*c - m*c), c = scale*log2 e
//   the running max m is only moved (and l, O rescaled) when the new max
//   exceeds it by more than 16 in log2 units; otherwise the stale m is kept,
//   which is exact (l and O share the same reference) and bounds P by 2^16.
//
// Every mbarrier wait is bounded (device_common.cuh): a stuck pipeline is
// reported as FA_ERR_DEVICE_TIMEOUT and the CTA drains its copies and MMAs,
// frees TMEM and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>
#include <math.h>

#include "device_common.cuh"
#include "tc_common.cuh"

namespace fa {
namespace {

constexpr int BM = 128;             // rows per query tile (MMA M)
constexpr int BN = 128;             // keys per K/V tile
constexpr int kThreads = 352;       // 11 warps
constexpr int kProducerWarp = 8;
constexpr int kMmaWarpA = 9;        // MMA issuer of query tile 0; allocates TMEM
constexpr int kMmaWarpB = 10;       // MMA issuer of query tile 1
constexpr uint32_t kTokenBar = 1;   // named barriers 1, 2: the issuers' turn tokens
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 16.0f;  // log2 units
// Epilogue destinations.
constexpr int kOutBf16 = 0;   // O bf16, L
constexpr int kOutF32 = 1;    // O fp32, L
constexpr int kOutPart = 2;   // split-key partial: O_g fp32 and L_g into the workspace

// Varlen batches with at most kMaxSchedSeqs sequences and kMaxSchedLevels
// 256-row blocks per sequence get a compact schedule (see decode_item).
constexpr int kMaxSchedSeqs = 384;
// K/V bytes of the heads that a varlen batch's compact order keeps in
// flight together (the L2 is 129 MB; Q, O and other traffic share it).
constexpr double kL2GroupBytes = 64.0 * 1024 * 1024;
constexpr int kMaxSchedLevels = 128;

template <int D>
struct Cfg {
    static constexpr int kHalves = D / 64;                    // 128-byte swizzle atoms per row
    static constexpr int kTileBytes = BN * D * 2;             // one K or V tile (== Q tile)
    static constexpr int kHalfBytes = BN * 64 * 2;            // 16 KB
    static constexpr int kSlots = (D == 128) ? 5 : 10;
    static constexpr int kQBytes = 2 * kTileBytes;
    static constexpr int kRingOff = kQBytes;
    static constexpr int kBarOff = kRingOff + kSlots * kTileBytes;
    // D=128 fills TMEM with S_0, S_1, O_0, O_1, so P_s overwrites S_s and the
    // next Q K^T must follow P V.  At D=64 P_s gets columns of its own: the
    // next S_s is computed as soon as the softmax has read S_s, so the
    // softmax warps never wait for S.
    static constexpr bool kPAlias = (D == 128);
    static constexpr int kBarBytes = kPAlias ? 256 : 512;
    static constexpr int kSchedOff = kBarOff + kBarBytes;         // varlen schedule table
    static constexpr int kSchedBytes = 2 * (kMaxSchedSeqs + kMaxSchedLevels) + 16;
    static constexpr int kSmemBytes = kSchedOff + kSchedBytes + 1024;  // + alignment slack
    static_assert(kSmemBytes <= 232448, "shared memory per CTA");
    // q full/empty, ring full/empty, s_full, p_full, o_final, s_free, pv_done
    // (two each), drain, then the TMEM address and the abort flag.
    static_assert(kBarBytes >= 8 * (2 + 2 * kSlots + 10 + 1) + 16, "barrier area");
};

struct TcParams {
    float *lse;
    void *o;
    const int32_t *cu;
    int varlen;
    int heads;
    int units_bh;     // dense: B*H; varlen: num_seqs*H
    int n;            // dense: N; varlen: max_seqlen
    int64_t total;    // varlen: total tokens
    int num_mblk;     // ceil(n / 256)
    int num_splits;   // key-range splits per block (1 = none)
    int num_seqs;     // varlen: sequences
    int compact;      // varlen: use the compact schedule table
    int num_items;    // num_mblk * num_splits * units_bh
    int head_group;   // varlen compact order: heads per group
    float *ws_o;      // split mode: partial O, fp32 [splits][units][n][D]
    float *ws_l;      // split mode: partial L, fp32 [splits][units][n]
    float scale;
    float scale_log2;  // scale * log2(e)
    int causal;
    int wl, wr;        // key j visible to row i iff i - wl <= j <= i + wr (< 0: unbounded)
    uint32_t *err;
    uint64_t wait_limit_ns;
    int o_v8;          // output base 32-byte aligned: the epilogue stores 32 B per instruction
};

// One work item = one 256-row block (two query tiles) of one (b, h) or
// (sequence, h).  Items are ordered heaviest block first; CTA c takes items
// c, 2G-1-c, 2G+c, 4G-1-c, ... (a snake over the ordered list), which pairs
// heavy and light causal blocks on the same CTA.
struct Item {
    int bh;          // dense: b*H + h
    int h;           // head (varlen coordinates)
    int64_t start;   // first token of the sequence (varlen), else 0
    int len;         // rows (= keys) of the sequence
    int mb;          // 256-row block index
    int g;           // key-range split of the block
    int t0;          // first K/V tile of the split
    int a0, a1;      // first K/V tile (relative to t0) of query tile 0 / 1
    int nk0, nk1;    // end (exclusive, relative to t0) of the tiles of query tile 0 / 1
    int nkv;         // max(nk0, nk1): tiles loaded for the item
};

// K/V tile range of split g of a block whose two query tiles need nk0_full and
// nk1_full tiles from tile 0: the block's nkv tiles are cut into num_splits
// contiguous, near-equal ranges.  Shared by the kernel and the merge.
__host__ __device__ __forceinline__ void split_range(int nk0_full, int nk1_full, int g, int S,
                                                     int &t0, int &nk0, int &nk1) {
    const int nkv = nk0_full > nk1_full ? nk0_full : nk1_full;
    const int ta = (int)(((long long)g * nkv) / S), tb = (int)(((long long)(g + 1) * nkv) / S);
    t0 = ta;
    const int e0 = (nk0_full < tb ? nk0_full : tb) - ta, e1 = (nk1_full < tb ? nk1_full : tb) - ta;
    nk0 = e0 > 0 ? e0 : 0;
    nk1 = e1 > 0 ? e1 : 0;
}

__device__ __forceinline__ int snake_item(int round, int cta, int G) {
    return round * G + ((round & 1) ? (G - 1 - cta) : cta);
}

// Tiles needed from tile 0 by the two query tiles of block mb (rows
// [256 mb, 256 mb + 256)) of a sequence of `len` rows, causal or full: the
// no-left-bound case of block_ranges, in closed form.
__host__ __device__ __forceinline__ void block_tiles(int len, int mb, int causal, int &nk0, int &nk1) {
    const int row0 = mb * 256;
    const int tiles = (len + 127) / 128;
    if (causal) {
        nk0 = tiles < 2 * mb + 1 ? tiles : 2 * mb + 1;
        nk1 = (row0 + 128 < len) ? (tiles < 2 * mb + 2 ? tiles : 2 * mb + 2) : 0;
    } else {
        nk0 = tiles;
        nk1 = (row0 + 128 < len) ? tiles : 0;
    }
}

// K/V tile ranges [lo_s, hi_s) needed by the two query tiles of block mb
// when key j is visible to row i iff i - wl <= j <= i + wr (a negative bound
// is unbounded; causal is (-1, 0), no mask (-1, -1)).  An empty query tile
// gets lo = hi = 0.  Because wl + wr >= 0, the two ranges touch: every tile in
// [lo_0, hi_1) is read by at least one query tile.
__host__ __device__ __forceinline__ void block_ranges(int len, int mb, int wl, int wr, int &lo0, int &hi0,
                                                      int &lo1, int &hi1) {
    int lo[2], hi[2];
    for (int s = 0; s < 2; ++s) {
        const int r0 = mb * 256 + s * 128;
        if (r0 >= len) {
            lo[s] = hi[s] = 0;
            continue;
        }
        const int r1 = (r0 + 127 < len - 1) ? r0 + 127 : len - 1;
        const int klo = wl < 0 ? 0 : (r0 - wl > 0 ? r0 - wl : 0);
        const int khi = wr < 0 ? len - 1 : (r1 + wr < len - 1 ? r1 + wr : len - 1);
        lo[s] = klo / 128;
        hi[s] = khi / 128 + 1;
    }
    lo0 = lo[0];
    hi0 = hi[0];
    lo1 = lo[1];
    hi1 = hi[1];
}

// Fill the tile ranges of an (unsplit) item.
template <bool WIN>
__device__ __forceinline__ void item_ranges(const TcParams &p, Item &it) {
    if (!WIN) {
        it.t0 = 0;
        it.a0 = it.a1 = 0;
        block_tiles(it.len, it.mb, p.causal, it.nk0, it.nk1);
        it.nkv = max(it.nk0, it.nk1);
        return;
    }
    int lo0, hi0, lo1, hi1;
    block_ranges(it.len, it.mb, p.wl, p.wr, lo0, hi0, lo1, hi1);
    it.t0 = lo0;
    it.a0 = 0;
    it.nk0 = hi0 - lo0;
    if (hi1 > lo1) {
        it.a1 = lo1 - lo0;
        it.nk1 = hi1 - lo0;
    } else {
        it.a1 = 0;
        it.nk1 = 0;
    }
    it.nkv = max(it.nk0, it.nk1);
}

// Decode item `idx`; returns false when the item holds no work.  Items are
// ordered block-from-the-end (heaviest causal blocks first), then split, then
// (batch, head) / (sequence, head).
// Shared-memory schedule of a varlen batch: the sequences ranked by their
// number of 256-row blocks (longest first, ties by index) and, per block
// level L, how many sequences reach it.  Built once per CTA; every role
// decodes from it, so all agree on the order.
struct Sched {
    const uint16_t *ranked;   // [num_seqs] sequence ids, longest first
    const uint16_t *reach;    // [num_mblk] #sequences with more than L blocks
    int per_head;             // items per head: the sum of reach over the levels
};

// Varlen compact order: heads in groups of p.head_group (a group's K and V
// sized to stay in L2 while its items run); within a group, level L from
// the top, then the sequences that reach L (longest first), then the
// group's heads -- only items that hold work, so the snake assignment
// spreads real work evenly instead of walking empty slots.
template <bool WIN>
__device__ __forceinline__ bool decode_varlen_compact(const TcParams &p, const Sched &sc, int idx,
                                                      Item &it) {
    const int grp = idx / (sc.per_head * p.head_group);
    idx -= grp * sc.per_head * p.head_group;
    const int h0 = grp * p.head_group;
    if (h0 >= p.heads) return false;
    const int hn = min(p.head_group, p.heads - h0);
    int L = p.num_mblk - 1;
    for (; L >= 0; --L) {
        const int here = (int)sc.reach[L] * hn;
        if (idx < here) break;
        idx -= here;
    }
    if (L < 0) return false;
    const int seq = sc.ranked[idx / hn];
    it.h = h0 + idx % hn;
    it.bh = 0;
    it.g = 0;
    it.mb = L;
    int64_t start;
    int len;
    if (!seq_bounds(p.cu, seq, p.total, p.n, p.err, start, len)) return false;
    it.start = start;
    it.len = len;
    if (it.mb * 2 * BM >= it.len) return false;
    item_ranges<WIN>(p, it);
    return it.nkv > 0;
}

template <bool SPLIT, bool WIN>
__device__ __forceinline__ bool decode_item(const TcParams &p, const Sched &sc, int idx, Item &it) {
    if (!SPLIT && p.compact) return decode_varlen_compact<WIN>(p, sc, idx, it);
    const int S = SPLIT ? p.num_splits : 1;
    const int per_blk = p.units_bh * S;
    const int blk_from_end = idx / per_blk;
    const int rem = idx % per_blk;
    it.g = rem / p.units_bh;
    const int u = rem % p.units_bh;
    it.mb = p.num_mblk - 1 - blk_from_end;
    if (p.varlen) {
        const int s = u / p.heads;
        it.h = u % p.heads;
        it.bh = 0;
        int len;
        int64_t start;
        if (!seq_bounds(p.cu, s, p.total, p.n, p.err, start, len)) return false;
        it.start = start;
        it.len = len;
    } else {
        it.bh = u;
        it.h = 0;
        it.start = 0;
        it.len = p.n;
    }
    if (it.mb * 2 * BM >= it.len) return false;
    if (SPLIT) {  // split mode has no window: every range starts at tile 0
        int nk0_full, nk1_full;
        block_tiles(it.len, it.mb, p.causal, nk0_full, nk1_full);
        split_range(nk0_full, nk1_full, it.g, S, it.t0, it.nk0, it.nk1);
        it.a0 = it.a1 = 0;
        it.nkv = max(it.nk0, it.nk1);
    } else {
        item_ranges<WIN>(p, it);
    }
    return it.nkv > 0;
}

// --------------------------------------------------------------- kernel --
template <int D, int OUT, bool WIN>
// 11 warps put 3 warps on three of the four SM sub-partitions, whose register
// files hold 16K registers each: at most 168 registers per thread.
__global__ void __launch_bounds__(kThreads, 1)
    fa_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const TcParams p) {
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);

    const uint32_t q_smem = base;                  // [2][halves][128 rows][128 B]
    const uint32_t ring = base + C::kRingOff;      // [slots][halves][128][128 B]
    const uint32_t bars = base + C::kBarOff;
    // barrier addresses
    const uint32_t bar_q_full = bars + 0;
    const uint32_t bar_q_empty = bars + 8;
    const uint32_t bar_kv_full = bars + 16;                    // [slots]
    const uint32_t bar_kv_empty = bar_kv_full + 8 * C::kSlots; // [slots]
    const uint32_t bar_s_full = bar_kv_empty + 8 * C::kSlots;  // [2]
    const uint32_t bar_p_full = bar_s_full + 16;               // [2]
    const uint32_t bar_o_final = bar_p_full + 16;              // [2]
    const uint32_t bar_s_free = bar_o_final + 16;              // [2] S_s read (D=64)
    const uint32_t bar_pv_done = bar_s_free + 16;              // [2] P_s V done (D=64)
    const uint32_t bar_drain = bar_pv_done + 16;
    uint8_t *gbars = gbase + C::kBarOff;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbars + C::kBarBytes - 16);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(gbars + C::kBarBytes - 8);
    volatile int *exit_flag = reinterpret_cast<volatile int *>(gbars + C::kBarBytes - 12);  // issuers stop

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Band masks with a left bound exist only in the WIN instantiation; the
    // plain causal / full kernels keep the simpler fixed-start schedule.
    const int win_l = WIN ? p.wl : -1;

    // The next launch may set up its CTAs while this grid's last ones run.
    pdl_launch_dependents();
    if (warp == kProducerWarp && lane == 0) {
        mbar_init(bar_q_full, 1);
        mbar_init(bar_q_empty, 2);    // one commit per issuer warp
        for (int i = 0; i < C::kSlots; ++i) {
            mbar_init(bar_kv_full + 8 * i, 1);
            mbar_init(bar_kv_empty + 8 * i, 2);   // one commit per issuer warp
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar_s_full + 8 * s, 1);
            mbar_init(bar_p_full + 8 * s, 4);
            mbar_init(bar_o_final + 8 * s, 1);
            mbar_init(bar_s_free + 8 * s, 4);
            mbar_init(bar_pv_done + 8 * s, 1);
        }
        mbar_init(bar_drain, 2);
        *abort_flag = 0;
        *exit_flag = 0;
        fence_barrier_init();
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
    }
    if (warp == kMmaWarpA) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    // Everything above touched only shared memory and TMEM: wait here for the
    // previous kernel in the stream before any global memory access.
    pdl_wait();
    // Varlen compact schedule: rank the sequences by block count and count
    // how many reach each block level.  The lengths are staged in the (not
    // yet used) K/V ring; TMA writes there only after the barrier below.
    uint16_t *sched_ranked = reinterpret_cast<uint16_t *>(gbase + C::kSchedOff);
    uint16_t *sched_reach = sched_ranked + kMaxSchedSeqs;
    if (p.compact) {
        int *nblk = reinterpret_cast<int *>(gbase + C::kRingOff);
        for (int q = threadIdx.x; q < p.num_seqs; q += blockDim.x) {
            int64_t start;
            int len;
            seq_bounds(p.cu, q, p.total, p.n, p.err, start, len);  // invalid: len = 0
            nblk[q] = (len + 2 * BM - 1) / (2 * BM);
        }
        __syncthreads();
        for (int q = threadIdx.x; q < p.num_seqs; q += blockDim.x) {
            const int nq = nblk[q];
            int rank = 0;
            for (int t = 0; t < p.num_seqs; ++t) {
                const int nt = nblk[t];
                rank += (nt > nq) || (nt == nq && t < q);
            }
            sched_ranked[rank] = (uint16_t)q;
        }
        for (int L = threadIdx.x; L < p.num_mblk; L += blockDim.x) {
            int reach = 0;
            for (int t = 0; t < p.num_seqs; ++t) reach += nblk[t] > L;
            sched_reach[L] = (uint16_t)reach;
        }
        if (threadIdx.x == 0) {
            int total = 0;
            for (int t = 0; t < p.num_seqs; ++t) total += nblk[t];
            *reinterpret_cast<int *>(sched_reach + kMaxSchedLevels) = total;
        }
        // generic-proxy use of the ring is over before TMA (async proxy) writes it
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const Sched sched{sched_ranked, sched_reach,
                      p.compact ? *reinterpret_cast<const int *>(sched_reach + kMaxSchedLevels) : 0};
    const uint32_t tmem = *tmem_slot;

    const WaitCtx wc{p.err, abort_flag, p.wait_limit_ns};
    const int G = gridDim.x;
    const int cta = blockIdx.x;

    if (warp == kProducerWarp) {
        // ------------------------------------------------------ producer
        if (lane == 0) {
            uint32_t lc = 0;          // K/V loads issued
            uint32_t items = 0;       // items loaded
            bool ok = true;
            for (int k = 0; ok && k * G < p.num_items; ++k) {
                const int idx = snake_item(k, cta, G);
                if (idx >= p.num_items) continue;
                Item it;
                if (!decode_item<OUT == kOutPart, WIN>(p, sched, idx, it)) continue;
                if (items > 0 && !mbar_wait(bar_q_empty, (items - 1) & 1, wc, 1)) { ok = false; break; }
                mbar_arrive_expect_tx(bar_q_full, 2 * C::kTileBytes);
                for (int s = 0; s < 2; ++s) {
                    const int row = it.mb * 2 * BM + s * BM;
                    for (int hf = 0; hf < C::kHalves; ++hf) {
                        const uint32_t dst = q_smem + s * C::kTileBytes + hf * C::kHalfBytes;
                        if (p.varlen)
                            tma_load_3d(dst, &tm_q, bar_q_full, hf * 64, it.h, (int)(it.start + row));
                        else
                            tma_load_3d(dst, &tm_q, bar_q_full, hf * 64, row, it.bh);
                    }
                }
                ++items;
                for (int j = 0; j < it.nkv && ok; ++j) {
                    for (int kv = 0; kv < 2; ++kv) {
                        const uint32_t slot = lc % C::kSlots, round = lc / C::kSlots;
                        if (round > 0 && !mbar_wait(bar_kv_empty + 8 * slot, (round - 1) & 1, wc, 2)) {
                            ok = false;
                            break;
                        }
                        const uint32_t fb = bar_kv_full + 8 * slot;
                        mbar_arrive_expect_tx(fb, C::kTileBytes);
                        const CUtensorMap *tm = kv == 0 ? &tm_k : &tm_v;
                        for (int hf = 0; hf < C::kHalves; ++hf) {
                            const uint32_t dst = ring + slot * C::kTileBytes + hf * C::kHalfBytes;
                            if (p.varlen)
                                tma_load_3d(dst, tm, fb, hf * 64, it.h, (int)(it.start + (it.t0 + j) * BN));
                            else
                                tma_load_3d(dst, tm, fb, hf * 64, (it.t0 + j) * BN, it.bh);
                        }
                        ++lc;
                    }
                }
            }
            // Teardown: let every copy already issued land before exit.
            const uint64_t lim = p.wait_limit_ns;
            const uint32_t first = lc > (uint32_t)C::kSlots ? lc - C::kSlots : 0;
            for (uint32_t i = first; i < lc; ++i)
                mbar_drain(bar_kv_full + 8 * (i % C::kSlots), (i / C::kSlots) & 1, lim);
            if (items > 0) mbar_drain(bar_q_full, (items - 1) & 1, lim);
        }
    } else if (warp == kMmaWarpA || warp == kMmaWarpB) {
        // ----------------------------------------------------------- MMA
        // Two issuer warps, one per query tile s.  tcgen05.mma issue is
        // effectively synchronous with execution, so every cycle an issuer
        // spends on barrier waits, commits and control is tensor idle time.
        // The warps therefore take turns: each does its waits while the other
        // is issuing, then takes the turn token (a named barrier the other
        // warp arrives on when its block is issued) and issues its own block
        // back to back.  The token keeps the two tiles' blocks from
        // interleaving, so each block completes as early as with one issuer.
        // Within a warp the whole warp runs the control flow and waits; one
        // elected lane issues every tcgen05.mma / commit (always the same
        // lane).  A ring slot is released by both warps (its empty barrier
        // counts two commits), each commit covering that warp's reads of it.
        const int s = warp - kMmaWarpA;    // query tile this warp issues for
        const uint64_t dq_s = smem_desc(q_smem + s * C::kTileBytes, 16, 1024);
        const uint64_t dk_ring = smem_desc(ring, 16, 1024);
        const uint64_t dv_ring = smem_desc(ring, C::kHalfBytes, 1024);
        constexpr uint64_t kSlotDesc = C::kTileBytes >> 4;  // one slot in descriptor units
        const uint32_t t_s = tmem + s * BN;
        const uint32_t t_o = tmem + 2 * BN + s * D;
        const uint32_t t_p = C::kPAlias ? t_s : tmem + 2 * BN + 2 * D + s * (BN / 2);
        const uint32_t bar_sf = bar_s_full + 8 * s, bar_pf = bar_p_full + 8 * s;
        const uint32_t tok_me = kTokenBar + s, tok_other = kTokenBar + 1 - s;
        // Turn protocol.  Every turn: this warp's (bounded) waits, then the
        // token; a warp that must stop (a wait gave up, or the CTA aborts)
        // raises the exit flag and still passes the token, so the other warp,
        // which reads the flag right after taking the token, never waits on
        // a token that will not come.
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
        if (s == 1) named_bar_arrive(kTokenBar, 64);  // tile 0's warp takes the first turn
        uint32_t lc = 0, items = 0, pc = 0, fc = 0;   // ring loads, items, P_full / S_free phases
        bool run = true;
        for (int k = 0; run && k * G < p.num_items; ++k) {
            const int idx = snake_item(k, cta, G);
            if (idx >= p.num_items) continue;
            Item it;
            if (!decode_item<OUT == kOutPart, WIN>(p, sched, idx, it)) continue;
            // this tile reads K/V tiles [a_s, nk_s) of the item
            const int a_s = s == 0 ? 0 : (WIN ? it.a1 : 0);
            const int nk_s = s == 0 ? it.nk0 : it.nk1;
            bool okw = warp_wait(bar_q_full, items & 1, wc, 3);
            ++items;
            // K_j and V_j are ring loads number l0 + 2j and l0 + 2j + 1.
            const uint32_t l0 = lc;
            lc += 2 * it.nkv;
            const uint32_t s_k0 = l0 % C::kSlots;
            // prologue: S_s = Q_s K_0^T when the tile starts at tile 0 (in
            // split mode tile 0's range can be empty)
            const bool first = nk_s > a_s && a_s == 0;
            if (okw && first) okw = warp_wait(bar_kv_full + 8 * s_k0, (l0 / C::kSlots) & 1, wc, 4);
            if (!turn_begin(okw)) {
                run = false;
                break;
            }
            if (elect_one()) {
                if (first) {
                    issue_qk<D>(t_s, dq_s, dk_ring + s_k0 * kSlotDesc);
                    mma_commit(bar_sf);
                }
                mma_commit(bar_kv_empty + 8 * s_k0);
                if (it.nkv == 1) mma_commit(bar_q_empty);
            }
            turn_end();
            for (int j = 0; j < it.nkv; ++j) {
                const uint32_t li_v = l0 + 2 * j + 1, li_kn = li_v + 1;
                const uint32_t s_v = li_v % C::kSlots, s_kn = li_kn % C::kSlots;
                const uint64_t dv = dv_ring + s_v * kSlotDesc;
                const uint64_t dkn = dk_ring + s_kn * kSlotDesc;
                const bool reads = j >= a_s && j < nk_s;                   // P_s V_j
                const bool next = j + 1 >= a_s && j + 1 < nk_s;            // Q_s K_{j+1}^T
                if (C::kPAlias) {
                    // D=128: one turn per tile: O_s (+)= P_s V_j, then
                    // S_s = Q_s K_{j+1}^T (P_s overwrites S_s, so the next
                    // Q K^T must follow P V); a tile whose range starts at
                    // j + 1 issues its first Q K^T here.
                    // The ring loads are normally in place long before the
                    // softmax hands over P_s: wait for them first, so that
                    // only the token stands between P_full and the issue.
                    okw = true;
                    if (reads) okw = ring_wait(bar_kv_full, li_v, C::kSlots, wc, 5);
                    if (okw && next) okw = ring_wait(bar_kv_full, li_kn, C::kSlots, wc, 8 + s);
                    if (reads) {
                        okw = okw && warp_wait(bar_pf, pc & 1, wc, 6 + s);
                        ++pc;
                    }
                    if (!turn_begin(okw)) {
                        run = false;
                        break;
                    }
                    if (elect_one()) {
                        if (reads) issue_pv<D>(t_o, t_p, dv, j > a_s ? 1u : 0u);
                        if (next) {
                            issue_qk<D>(t_s, dq_s, dkn);
                            mma_commit(bar_sf);
                        } else if (reads) {
                            mma_commit(bar_o_final + 8 * s);
                        }
                        // K_{j+1} and V_j: this warp's reads of them are issued
                        if (j + 1 < it.nkv) mma_commit(bar_kv_empty + 8 * s_kn);
                        if (j == it.nkv - 2) mma_commit(bar_q_empty);  // the item's last Q K^T
                        mma_commit(bar_kv_empty + 8 * s_v);
                    }
                    turn_end();
                } else {
                    // D=64: P_s has its own TMEM columns.  Turn 1: the next
                    // S_s as soon as the softmax has read S_s; turn 2: P_s V_j.
                    if (j + 1 < it.nkv) {
                        okw = true;
                        if (next) {
                            okw = ring_wait(bar_kv_full, li_kn, C::kSlots, wc, 8 + s);
                            // a tile that starts at j + 1 has no softmax of tile j to wait for
                            if (okw && j >= a_s) {
                                okw = warp_wait(bar_s_free + 8 * s, fc & 1, wc, 10 + s);
                                ++fc;
                            }
                        }
                        if (!turn_begin(okw)) {
                            run = false;
                            break;
                        }
                        if (elect_one()) {
                            if (next) {
                                issue_qk<D>(t_s, dq_s, dkn);
                                mma_commit(bar_sf);
                            }
                            mma_commit(bar_kv_empty + 8 * s_kn);  // K_{j+1} has had this warp's reader
                            if (j + 1 == it.nkv - 1) mma_commit(bar_q_empty);
                        }
                        turn_end();
                    }
                    okw = true;
                    if (reads) {
                        okw = ring_wait(bar_kv_full, li_v, C::kSlots, wc, 5) &&
                              warp_wait(bar_pf, pc & 1, wc, 6 + s);
                        ++pc;
                    }
                    if (!turn_begin(okw)) {
                        run = false;
                        break;
                    }
                    if (elect_one()) {
                        if (reads) {
                            issue_pv<D>(t_o, t_p, dv, j > a_s ? 1u : 0u);
                            mma_commit(bar_pv_done + 8 * s);
                        }
                        mma_commit(bar_kv_empty + 8 * s_v);
                    }
                    turn_end();
                }
            }
        }
        // Teardown: wait for every MMA issued so far before TMEM is freed.
        if (elect_one()) mma_commit(bar_drain);
        __syncwarp();
        mbar_drain(bar_drain, 0, p.wait_limit_ns);
    } else {
        // ------------------------------------------------------- softmax
        const int s = warp >> 2;          // query tile of this warpgroup
        const int quarter = warp & 3;     // TMEM lane quarter
        const int r = quarter * 32 + lane;  // row within the query tile
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t t_s = tmem + lane_off + s * BN;           // S_s
        const uint32_t t_o = tmem + lane_off + 2 * BN + s * D;   // O_s
        const uint32_t t_p = C::kPAlias ? t_s : tmem + lane_off + 2 * BN + 2 * D + s * (BN / 2);  // P_s
        const float c = p.scale_log2;
        uint32_t sc = 0, oc = 0, pvc = 0;  // S_full, O_final, PV_done phases consumed
        bool ok = true;
        for (int k = 0; ok && k * G < p.num_items; ++k) {
            const int idx = snake_item(k, cta, G);
            if (idx >= p.num_items) continue;
            Item it;
            if (!decode_item<OUT == kOutPart, WIN>(p, sched, idx, it)) continue;
            const int a_s = s == 0 ? 0 : (WIN ? it.a1 : 0);
            const int nks = (s == 0 ? it.nk0 : it.nk1) - a_s;  // tiles this query tile reads
            if (nks <= 0) continue;
            const int row = it.mb * 2 * BM + s * BM + r;   // row within the sequence
            const int len = it.len;
            const int key_base = (it.t0 + a_s) * BN;       // first key this query tile reads
            const bool store = row < len;
            int64_t orow, li;                              // where O and L of this row go
            if (OUT == kOutPart) {  // dense only: [split][b*h][row]
                li = ((int64_t)it.g * p.units_bh + it.bh) * p.n + row;
                orow = li * D;
            } else if (p.varlen) {
                orow = ((it.start + row) * p.heads + it.h) * (int64_t)D;
                li = (int64_t)it.h * p.total + it.start + row;
            } else {
                orow = ((int64_t)it.bh * p.n + row) * D;
                li = (int64_t)it.bh * p.n + row;
            }
            float m_use = -INFINITY, l = 0.f;
            for (int j = 0; j < nks; ++j) {
                if (!warp_wait(bar_s_full + 8 * s, sc & 1, wc, 16 + s)) { ok = false; break; }
                ++sc;
                tc_fence_after();
                const int key0 = key_base + j * BN;
                // Rows of this query tile are row - r .. row - r + 127; a tile needs
                // masking if it crosses the sequence end or a window edge.
                const bool need_mask = (key0 + BN > len) ||
                                       (p.wr >= 0 && key0 + BN - 1 > row - r + p.wr) ||
                                       (win_l >= 0 && key0 < row - r + 127 - win_l);
                float x[BN];
                float mx;
                if (!need_mask) {
                    // the row maximum comes with the load
                    tmem_ld128_max(t_s, x, mx);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int cc = 0; cc < BN / 32; ++cc)
                        tmem_ld32(t_s + cc * 32, x + cc * 32);
                    tmem_wait_ld();
                }
                if (!C::kPAlias && j + 1 < nks) {
                    // S_s is in registers: the MMA warp may compute the next S_s.
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar_s_free + 8 * s);
                }
                if (need_mask) {
                    // keys in [lo_lim, hi_lim) are live for this row
                    const int hi_lim = p.wr >= 0 ? min(row + p.wr + 1, len) : len;
                    const int lo_lim = win_l >= 0 ? row - win_l : 0;
#pragma unroll
                    for (int i = 0; i < BN; ++i)
                        if (key0 + i >= hi_lim || key0 + i < lo_lim) x[i] = -INFINITY;
                    // Row max of the masked scores: 8 independent chains of
                    // 3-input max, then a tree.
                    float mx8[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) mx8[k] = fmaxf(x[k], x[8 + k]);
#pragma unroll
                    for (int t = 2; t < 16; t += 2)
#pragma unroll
                        for (int k = 0; k < 8; ++k) mx8[k] = max3f(mx8[k], x[8 * t + k], x[8 * t + 8 + k]);
                    mx = fmaxf(max3f(mx8[0], mx8[1], mx8[2]),
                               max3f(max3f(mx8[3], mx8[4], mx8[5]), mx8[6], mx8[7]));
                }
                const float m_new = fmaxf(m_use, mx);
                const bool move = (m_new - m_use) * c > kRescaleThreshold;
                float alpha = 1.f;
                if (move) {
                    alpha = (m_use == -INFINITY) ? 0.f : ex2_approx((m_use - m_new) * c);
                    m_use = m_new;
                }
                // p = exp2(S*c - m*c): packed FFMA2 for the arguments, SFU ex2,
                // 8 independent partial row sums, bf16x2 packing into TMEM.
                if (!C::kPAlias && j > 0) {
                    // P_s(j-1) V is complete: P_s may be overwritten and O_s is
                    // stable.  (With P aliasing S this is implied by S_full:
                    // the next Q K^T was issued after that P V.)
                    if (!warp_wait(bar_pv_done + 8 * s, pvc & 1, wc, 20 + s)) { ok = false; break; }
                    ++pvc;
                    tc_fence_after();
                }
                const float mc = (m_use == -INFINITY) ? 0.f : m_use * c;
                const float2 c2 = make_float2(c, c), nmc2 = make_float2(-mc, -mc);
                float2 rs4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                 make_float2(0.f, 0.f)};
#pragma unroll
                for (int cc = 0; cc < BN / 32; ++cc) {
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float2 a = __ffma2_rn(make_float2(x[cc * 32 + 2 * i], x[cc * 32 + 2 * i + 1]),
                                                    c2, nmc2);
                        const float2 e = make_float2(ex2_approx(a.x), ex2_approx(a.y));
                        rs4[i & 3] = __fadd2_rn(rs4[i & 3], e);
                        pk[i] = pack_bf16x2(e.x, e.y);
                    }
                    tmem_st16(t_p + cc * 16, pk);
                }
                const float rs = ((rs4[0].x + rs4[0].y) + (rs4[1].x + rs4[1].y)) +
                                 ((rs4[2].x + rs4[2].y) + (rs4[3].x + rs4[3].y));
                if (j > 0 && __any_sync(0xffffffffu, move)) {
                    // O_s *= alpha (rows that keep their max use alpha = 1).
                    // PV of the previous tile is complete: S_full of this
                    // tile was committed after it.
#pragma unroll
                    for (int cc = 0; cc < D / 32; ++cc) {
                        float o[32];
                        tmem_ld32(t_o + cc * 32, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] *= alpha;
                        tmem_st32(t_o + cc * 32, o);
                    }
                }
                l = alpha * l + rs;
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_p_full + 8 * s);
            }
            if (!ok) break;
            // ------------------------------------------------- epilogue
            if (C::kPAlias) {
                if (!warp_wait(bar_o_final + 8 * s, oc & 1, wc, 18 + s)) { ok = false; break; }
                ++oc;
            } else {  // the last P V of the item
                if (!warp_wait(bar_pv_done + 8 * s, pvc & 1, wc, 20 + s)) { ok = false; break; }
                ++pvc;
            }
            tc_fence_after();
            const bool live = l > 0.f;
            const float inv = live ? 1.f / l : 0.f;
            float *const o32 = OUT == kOutPart ? p.ws_o : static_cast<float *>(p.o);
            float *const lout = OUT == kOutPart ? p.ws_l : p.lse;
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
                float o[32];
                tmem_ld32(t_o + cc * 32, o);
                tmem_wait_ld();
                if (!WIN && store && p.o_v8) {
                    // 32-byte stores: every sector a thread touches is written whole
                    // (measured faster for causal / full attention, slower for the
                    // short items of a narrow band)
                    if (OUT != kOutBf16) {
                        float *dst = o32 + orow + cc * 32;
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            uint32_t w[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) w[e] = __float_as_uint(o[8 * i + e] * inv);
                            st_global_v8(dst + 8 * i, w);
                        }
                    } else {
                        __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(p.o) + orow + cc * 32;
#pragma unroll
                        for (int i = 0; i < 2; ++i) {
                            uint32_t w[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                w[e] = pack_bf16x2(o[16 * i + 2 * e] * inv, o[16 * i + 2 * e + 1] * inv);
                            st_global_v8(dst + 16 * i, w);
                        }
                    }
                } else if (store) {
                    if (OUT != kOutBf16) {
                        float4 *dst = reinterpret_cast<float4 *>(o32 + orow + cc * 32);
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            dst[i] = make_float4(o[4 * i] * inv, o[4 * i + 1] * inv, o[4 * i + 2] * inv,
                                                 o[4 * i + 3] * inv);
                    } else {
                        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.o) + orow +
                                                               cc * 32);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            dst[i] = make_uint4(pack_bf16x2(o[8 * i] * inv, o[8 * i + 1] * inv),
                                                pack_bf16x2(o[8 * i + 2] * inv, o[8 * i + 3] * inv),
                                                pack_bf16x2(o[8 * i + 4] * inv, o[8 * i + 5] * inv),
                                                pack_bf16x2(o[8 * i + 6] * inv, o[8 * i + 7] * inv));
                    }
                }
            }
            tc_fence_before();
            if (store) lout[li] = live ? m_use * p.scale + logf(l) : -INFINITY;
        }
    }

    __syncthreads();
    if (warp == kMmaWarpA) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------------ host side --
// Workspace layout of split-key mode: partial O (fp32) then partial L.
constexpr size_t kWsAlign = 256;
inline size_t ws_o_bytes(int S, int units, int n, int D) {
    return ((size_t)S * units * n * D * sizeof(float) + kWsAlign - 1) / kWsAlign * kWsAlign;
}
inline size_t ws_l_bytes(int S, int units, int n) {
    return ((size_t)S * units * n * sizeof(float) + kWsAlign - 1) / kWsAlign * kWsAlign;
}

// Merge of split-key partials: for each row, L = ln sum_g exp(L_g) and
// O = sum_g exp(L_g - L) O_g over the splits whose key range holds keys of
// the row -- the online-softmax rescale of "FlashAttention -- for
// programmers, not researchers.", STAGE 3, applied across splits.  D/4
// threads per row, one float4 of O each; HBM-bound.
template <int D, bool OUT_F32>
__global__ void __launch_bounds__(256)
    fa_merge_kernel(const float *__restrict__ ws_o, const float *__restrict__ ws_l, void *o, float *lse,
                    int units, int n, int S, int causal) {
    constexpr int TPR = D / 4;
    constexpr int RPB = 256 / TPR;
    const int c4 = threadIdx.x % TPR;
    const int64_t rows = (int64_t)units * n;
    for (int64_t r = (int64_t)blockIdx.x * RPB + threadIdx.x / TPR; r < rows; r += (int64_t)gridDim.x * RPB) {
        const int u = (int)(r / n), i = (int)(r % n);
        const int mb = i / 256, st = (i % 256) / 128;
        int nk0f, nk1f;
        block_tiles(n, mb, causal, nk0f, nk1f);
        float m = -INFINITY;
        for (int g = 0; g < S; ++g) {
            int t0, a0, a1;
            split_range(nk0f, nk1f, g, S, t0, a0, a1);
            if ((st ? a1 : a0) > 0) m = fmaxf(m, ws_l[((int64_t)g * units + u) * n + i]);
        }
        float sum = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (m != -INFINITY) {
            for (int g = 0; g < S; ++g) {
                int t0, a0, a1;
                split_range(nk0f, nk1f, g, S, t0, a0, a1);
                if ((st ? a1 : a0) == 0) continue;
                const int64_t row = ((int64_t)g * units + u) * n + i;
                const float w = expf(ws_l[row] - m);
                const float4 og = reinterpret_cast<const float4 *>(ws_o + row * D)[c4];
                sum += w;
                acc.x = fmaf(w, og.x, acc.x);
                acc.y = fmaf(w, og.y, acc.y);
                acc.z = fmaf(w, og.z, acc.z);
                acc.w = fmaf(w, og.w, acc.w);
            }
        }
        const float inv = sum > 0.f ? 1.f / sum : 0.f;
        const int64_t orow = ((int64_t)u * n + i) * D;
        if (OUT_F32) {
            reinterpret_cast<float4 *>(static_cast<float *>(o) + orow)[c4] =
                make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        } else {
            reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(o) + orow)[c4] =
                make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
        }
        if (c4 == 0) lse[(int64_t)u * n + i] = sum > 0.f ? m + logf(sum) : -INFINITY;
    }
}

template <int D, int OUT, bool WIN>
fa_status launch(const FaProblem &pr, int splits) {
    using C = Cfg<D>;
    CUtensorMap mq, mk, mv;
    const uint64_t es = 2;
    bool ok;
    if (pr.varlen) {
        const uint64_t d1 = pr.heads, d2 = pr.total;
        const uint64_t s1 = D * es, s2 = (uint64_t)pr.heads * D * es;
        ok = make_map(&mq, pr.q, D, d1, d2, s1, s2, 1, BN) && make_map(&mk, pr.k, D, d1, d2, s1, s2, 1, BN) &&
             make_map(&mv, pr.v, D, d1, d2, s1, s2, 1, BN);
    } else {
        const uint64_t d1 = pr.n, d2 = pr.units_bh;
        const uint64_t s1 = D * es, s2 = (uint64_t)pr.n * D * es;
        ok = make_map(&mq, pr.q, D, d1, d2, s1, s2, BN, 1) && make_map(&mk, pr.k, D, d1, d2, s1, s2, BN, 1) &&
             make_map(&mv, pr.v, D, d1, d2, s1, s2, BN, 1);
    }
    if (!ok) return FA_ERR_CUDA;  // reason recorded by make_map
    TcParams p;
    p.lse = pr.lse;
    p.o = pr.o;
    p.cu = pr.cu_seqlens;
    p.varlen = pr.varlen;
    p.heads = pr.heads;
    p.units_bh = pr.units_bh;
    p.n = pr.n;
    p.total = pr.total;
    p.num_mblk = (pr.n + 2 * BM - 1) / (2 * BM);
    p.num_splits = splits;
    p.num_seqs = pr.num_seqs;
    p.compact = pr.varlen && pr.num_seqs <= kMaxSchedSeqs && p.num_mblk <= kMaxSchedLevels;
    // Heads per group in the compact order: as many as keep the group's K
    // and V within kL2GroupBytes.
    {
        const double kv_per_head = (double)pr.total * D * 2 * 2;
        long long hg = kv_per_head > 0 ? (long long)(kL2GroupBytes / kv_per_head) : pr.heads;
        p.head_group = (int)(hg < 1 ? 1 : (hg > pr.heads ? pr.heads : hg));
    }
    const int64_t items = (int64_t)p.num_mblk * splits * pr.units_bh;
    if (items > INT32_MAX / 2) return FA_ERR_UNSUPPORTED;
    p.num_items = (int)items;
    p.ws_o = nullptr;
    p.ws_l = nullptr;
    if (OUT == kOutPart) {
        uint8_t *ws = static_cast<uint8_t *>(pr.workspace);
        p.ws_o = reinterpret_cast<float *>(ws);
        p.ws_l = reinterpret_cast<float *>(ws + ws_o_bytes(splits, pr.units_bh, pr.n, D));
    }
    p.scale = pr.scale;
    p.scale_log2 = pr.scale * 1.4426950408889634f;
    p.causal = pr.causal;
    p.wl = pr.wl;
    p.wr = pr.wr;
    p.err = pr.err;
    p.wait_limit_ns = pr.wait_limit_ns;
    p.o_v8 = (reinterpret_cast<uintptr_t>(OUT == kOutPart ? static_cast<void *>(p.ws_o) : p.o) & 31u) == 0;
    int grid = pr.grid_ctas > 0 ? pr.grid_ctas : num_sms();
    if (grid <= 0) return FA_ERR_CUDA;  // device query failed (recorded)
    if (grid > p.num_items) grid = p.num_items;
    auto kern = fa_tc_kernel<D, OUT, WIN>;
    static FaCtxSet ready;  // contexts set up for this instantiation
    const fa_status su = fa_once_per_context(ready, [&]() -> fa_status {
        cudaFuncAttributes fattr;
        cudaError_t e = cudaFuncGetAttributes(&fattr, kern);
        if (e != cudaSuccess) return fa_cuda_fail(e);
        if (fattr.maxThreadsPerBlock < kThreads) return fa_cuda_fail(cudaErrorLaunchOutOfResources);
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        return e == cudaSuccess ? FA_OK : fa_cuda_fail(e);
    });
    if (su != FA_OK) return su;
    // Programmatic stream serialization: the CTAs of this launch may start
    // (barrier and TMEM setup) while the previous kernel's last CTAs run;
    // the kernel waits for it (griddepcontrol.wait) before reading memory.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = pr.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, p);
    if (e == cudaSuccess) e = cudaGetLastError();
    return e == cudaSuccess ? FA_OK : fa_cuda_fail(e);
}

template <int D, bool OUT_F32>
fa_status launch_merge(const FaProblem &pr, int splits) {
    const uint8_t *ws = static_cast<const uint8_t *>(pr.workspace);
    const float *wo = reinterpret_cast<const float *>(ws);
    const float *wl = reinterpret_cast<const float *>(ws + ws_o_bytes(splits, pr.units_bh, pr.n, D));
    constexpr int RPB = 256 / (D / 4);
    const int64_t rows = (int64_t)pr.units_bh * pr.n;
    int64_t blocks = (rows + RPB - 1) / RPB;
    const int cap = (num_sms() > 0 ? num_sms() : 1) * 16;
    if (blocks > cap) blocks = cap;
    fa_merge_kernel<D, OUT_F32><<<(int)blocks, 256, 0, pr.stream>>>(wo, wl, pr.o, pr.lse, pr.units_bh, pr.n,
                                                                     splits, pr.causal);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? FA_OK : fa_cuda_fail(e);
}

template <int D>
fa_status launch_d(const FaProblem &pr) {
    const bool f32 = pr.dtype == FA_BF16_OUT_F32;
    // Causal (-1, 0) and full (-1, -1) use the plain kernels; any other band
    // the WIN instantiation.
    const bool win = pr.wl >= 0 || pr.wr > 0;
    if (pr.num_splits <= 1) {
        if (win) return f32 ? launch<D, kOutF32, true>(pr, 1) : launch<D, kOutBf16, true>(pr, 1);
        return f32 ? launch<D, kOutF32, false>(pr, 1) : launch<D, kOutBf16, false>(pr, 1);
    }
    const fa_status st = launch<D, kOutPart, false>(pr, pr.num_splits);
    if (st != FA_OK) return st;
    return f32 ? launch_merge<D, true>(pr, pr.num_splits) : launch_merge<D, false>(pr, pr.num_splits);
}

}  // namespace
}  // namespace fa

bool fa_tc_split_plan(int units_bh, int n, int D, int requested, int &splits, size_t &bytes) {
    const int num_mblk = (n + 2 * fa::BM - 1) / (2 * fa::BM);
    const int tiles = (n + fa::BN - 1) / fa::BN;
    int S = requested;
    if (S <= 0) {
        const int sms = fa::num_sms();
        if (sms <= 0) return false;
        const int64_t items = (int64_t)num_mblk * units_bh;
        S = items >= sms ? 1 : (int)((sms + items - 1) / items);
    }
    if (S > tiles) S = tiles;
    if (S > 64) S = 64;
    if (S < 1) S = 1;
    splits = S;
    bytes = S > 1 ? fa::ws_o_bytes(S, units_bh, n, D) + fa::ws_l_bytes(S, units_bh, n) : 0;
    return true;
}

fa_status fa_tc_supports(const FaProblem &pr) {
    if (pr.dtype != FA_BF16 && pr.dtype != FA_BF16_OUT_F32) return FA_ERR_UNSUPPORTED;
    if (pr.num_splits > 1 && (pr.varlen || pr.wl >= 0 || pr.wr > 0)) return FA_ERR_UNSUPPORTED;
    if (pr.D != 64 && pr.D != 128) return FA_ERR_UNSUPPORTED;
    // work items are numbered in 32-bit arithmetic with headroom
    const int64_t items = (int64_t)((pr.n + 2 * fa::BM - 1) / (2 * fa::BM)) *
                          (pr.num_splits > 1 ? pr.num_splits : 1) * pr.units_bh;
    if (pr.n < 0 || pr.units_bh < 0 || items > INT32_MAX / 2) return FA_ERR_UNSUPPORTED;
    return FA_OK;
}

fa_status fa_launch_tc(const FaProblem &pr) {
    const fa_status sup = fa_tc_supports(pr);
    if (sup != FA_OK) return sup;
    if (pr.D == 64) return fa::launch_d<64>(pr);
    if (pr.D == 128) return fa::launch_d<128>(pr);
    return FA_ERR_UNSUPPORTED;
}
