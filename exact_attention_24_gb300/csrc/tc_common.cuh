// Shared pieces of the tensor-core kernels (forward and backward): the
// warp-uniform bounded waits, tcgen05 shared-memory / instruction
// descriptors, the two MMA shapes every kernel here is built from, and the
// host-side TMA map encoder.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "device_common.cuh"
#include "fa_internal.h"

namespace fa {

constexpr int kTcRows = 128;             // MMA M, and the 128-row / 128-key tile
constexpr int kTcAtomBytes = 128 * 64 * 2;  // one 64-element-wide 128-byte-swizzle box of 128 rows

// Bounded wait by every lane of a warp, with a warp-uniform result (a lane
// that gave up makes the whole warp give up, so control flow never diverges
// around elect.sync / __syncwarp).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const WaitCtx &w,
                                          uint32_t site) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, w, site));
}

// Wait (whole warp) until ring load number `li` has landed in its slot.
__device__ __forceinline__ bool ring_wait(uint32_t bar_full, uint32_t li, uint32_t slots, const WaitCtx &w,
                                          uint32_t site) {
    return warp_wait(bar_full + 8 * (li % slots), (li / slots) & 1, w, site);
}

// ------------------------------------------------ UMMA descriptor helpers --
// Shared-memory matrix descriptor (tcgen05): start address, leading- and
// stride-dimension byte offsets (>> 4), fixed version bits 46-47 = 1,
// swizzle mode 2 (128-byte swizzle) in bits 61-63.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)(lbo >> 4) << 16) |
           ((uint64_t)(sbo >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor, kind::f16: D f32 (bits 4-5 = 1), A and B bf16
// (bits 7-9, 10-12 = 1), B transposed flag (bit 16: 1 = MN-major), N >> 3 in
// bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)b_mn_major << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// S (TMEM, 128 x 128 fp32) = Q (smem, 128 x D) * K^T (smem, 128 x D): both
// (and any A B^T of that shape, e.g. K Q^T or dO V^T in the backward pass)
// operands K-major with 128-byte swizzle; D/16 MMAs of K = 16.  Within a
// 64-element swizzle atom the K offset is a plain byte offset (32 B per
// step); the second half of D=128 is the next 16 KB box.  `dq`, `dk` are the
// descriptors of the tiles' first byte; the address field sits in the low
// bits, so an offset is added to the descriptor directly (in 16-byte units,
// never carrying out of the 14-bit field: shared memory is below 256 KB).
// The issue sequence is straight-line: the single issuing thread is the
// tensor core's only feeder, so every cycle spent here is tensor idle time.
template <int D>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint64_t dq, uint64_t dk) {
    constexpr uint32_t idesc = idesc_bf16(kTcRows, kTcRows, 0);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t off = (uint64_t)(((kk / 4) * kTcAtomBytes + (kk % 4) * 32) >> 4);
        mma_ss(d_tmem, dq + off, dk + off, idesc, kk > 0 ? 1u : 0u);
    }
}

// O (TMEM, 128 x D fp32) (+)= P (TMEM, 128 x 128 bf16) * V (smem, 128 x D)
// (and any A B of that shape with A in TMEM, e.g. dS K or P^T dO):
// V is MN-major (D contiguous) with 128-byte swizzle: 8-key groups are
// 1024 B apart (SBO), the two 64-column halves of D=128 are 16 KB apart
// (LBO).  Each MMA consumes 16 keys: 8 TMEM columns of P, 2048 B of V.
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t a_tmem, uint64_t dv,
                                         uint32_t accumulate) {
    constexpr uint32_t idesc = idesc_bf16(kTcRows, D, 1);
    mma_ts(d_tmem, a_tmem, dv, idesc, accumulate);
#pragma unroll
    for (int kk = 1; kk < kTcRows / 16; ++kk)
        mma_ts(d_tmem, a_tmem + kk * 8, dv + (uint64_t)((kk * 2048) >> 4), idesc, 1u);
}

// ------------------------------------------------------------ host side --
// The driver's tensor-map encoder, looked up once (thread-safe static
// initialisation); null, with the failure recorded, if the driver lacks it.
inline PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        const cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                                               cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess) {
            fa_cuda_fail(e != cudaSuccess ? e : cudaErrorSymbolNotFound);
            return nullptr;
        }
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }();
    if (!fn) fa_cuda_fail(cudaErrorSymbolNotFound);
    return fn;
}

// 3-D map over a bf16 tensor: dims {D, d1, d2} with byte strides {s1, s2};
// box {64, b1, b2}; 128-byte swizzle; out-of-range elements read as zero.
inline bool make_map(CUtensorMap *m, const void *ptr, int D, uint64_t d1, uint64_t d2, uint64_t s1,
              uint64_t s2, uint32_t b1, uint32_t b2) {
    auto enc = get_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, d1, d2};
    cuuint64_t strides[2] = {s1, s2};
    cuuint32_t box[3] = {64, b1, b2};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        fa_cuda_fail(cudaErrorInvalidValue);
        return false;
    }
    return true;
}

inline int num_sms() { return fa_num_sms(); }

}  // namespace fa
