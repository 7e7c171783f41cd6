/*
 * fa.h -- C ABI of the GB300 (sm_103a) FlashAttention-2 library: the
 * forward pass (fa_fwd and its variants) and its gradients (fa_bwd).
 *
 * The operation (for every batch b and head h, or every packed sequence s
 * and head h):
 *
 *     S = scale * Q K^T                    (scale applied after the dot
 *                                           product: "Kernel visualization:
 *                                           Flash Attention 2", section
 *                                           "Iteration j = 0")
 *     S[i][j] = -inf  for j > i            (causal only; i, j local to the
 *                                           sequence)
 *     O = softmax_rows(S) V                ("FlashAttention -- for
 *                                           programmers, not researchers.",
 *                                           STAGE 1 and STAGE 2)
 *     L[i] = m_i + ln(l_i) = ln sum_j exp(S[i][j])
 *                                          ("Kernel visualization: Flash
 *                                           Attention 2", section "Write the
 *                                           data back to HBM": O and L are
 *                                           written once; L is what the
 *                                           backward pass needs)
 *
 * computed by streaming K/V tiles through on-chip memory with an online
 * softmax (same script, STAGE 3 and STAGE 4), never forming the N x N
 * score matrix in memory.
 *
 * Conventions shared by every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller.  The
 *    library never allocates, frees or synchronises inside fa_fwd /
 *    fa_fwd_varlen; they only enqueue work on `stream` and return.
 *  - Tensors are contiguous, row-major, and 16-byte aligned.
 *  - Q, K, V may alias one another.  O and L must not overlap any input or
 *    each other.
 *  - D (head dimension) must be 64 or 128.
 *  - L is always float32, natural-log units.
 *  - A row whose keys are all masked (impossible for self-attention with
 *    the causal mask, since the diagonal is never masked) gets O = 0 and
 *    L = -inf.
 *  - Errors are returned as fa_status; nothing is thrown across the ABI.
 *    Checks that need device data (cu_seqlens contents) and the device
 *    watchdog report through fa_check_device_error().
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FA_API __attribute__((visibility("default")))
#else
#define FA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fa_status {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,    /* null / misaligned / overlapping pointer,
                                  negative size, bad dtype, non-finite
                                  scale, or (device side) cu_seqlens that is
                                  not non-decreasing within [0, total]     */
    FA_ERR_UNSUPPORTED = 2,    /* D not in {64, 128}; sizes beyond the
                                  int32 token / TMA coordinate range      */
    FA_ERR_CUDA = 3,           /* a CUDA runtime or driver call failed
                                  (launch, tensor-map encoding, sync); the
                                  runtime's last error is cleared         */
    FA_ERR_DEVICE_TIMEOUT = 4  /* a device-side wait ran past its limit;
                                  the kernel gave up and returned cleanly */
} fa_status;

typedef enum fa_dtype {
    FA_F32 = 0,          /* Q, K, V, O float32; arithmetic in fp32 FFMA    */
    FA_BF16 = 1,         /* Q, K, V, O bfloat16; tensor-core contractions
                            with fp32 accumulation, O rounded to nearest   */
    FA_BF16_OUT_F32 = 2  /* Q, K, V bfloat16, O float32 (same arithmetic
                            as FA_BF16 without the final rounding of O)    */
} fa_dtype;

/* A cudaStream_t.  NULL is the legacy default stream. */
typedef void *fa_stream_t;

/*
 * fa_fwd -- dense batch.
 *
 *   Q, K, V, O : [B, H, N, D] contiguous (element type per `dtype`)
 *   L          : [B, H, N] float32
 *   B, H, N    : >= 0 (any zero makes the call a no-op returning FA_OK)
 *   D          : 64 or 128
 *   scale      : finite; multiplies Q K^T (typically 1/sqrt(D))
 *   causal     : 0 or 1; when 1, key j is masked for query i if j > i
 *
 * The work is the set of independent (b, h, query-tile) units of the
 * "Same operations in another block" section of "Kernel visualization:
 * Flash Attention 2": no unit needs anything from another.
 *
 * Returns FA_OK once the work is enqueued on `stream`.
 */
FA_API fa_status fa_fwd(const void *Q, const void *K, const void *V, void *O,
                 float *L, int B, int H, int N, int D, float scale,
                 int causal, fa_dtype dtype, fa_stream_t stream);

/*
 * fa_fwd_window -- dense batch restricted to a local band of keys: key j is
 * visible to query i iff i - window_left <= j <= i + window_right, where -1
 * leaves that side unbounded.  (-1, 0) is the causal mask, (-1, -1) no mask,
 * and (64, 64) the local window that "FlashAttention -- for programmers, not
 * researchers.", DEMO 6, contrasts with exact attention (|i - j| <= 64).
 * Tiles wholly outside the band are never loaded.  Other arguments as fa_fwd.
 *
 *   window_left, window_right : >= -1 (FA_ERR_INVALID_ARG otherwise)
 */
FA_API fa_status fa_fwd_window(const void *Q, const void *K, const void *V, void *O,
                               float *L, int B, int H, int N, int D, float scale,
                               int window_left, int window_right, fa_dtype dtype,
                               fa_stream_t stream);

/*
 * fa_fwd_varlen -- packed batch of variable-length sequences (self
 * attention: queries and keys share cu_seqlens).
 *
 *   Q, K, V, O   : [total_tokens, H, D] contiguous (token-major packing)
 *   L            : [H, total_tokens] float32
 *   cu_seqlens   : DEVICE int32[num_seqs + 1]; cu_seqlens[0] = 0,
 *                  non-decreasing, cu_seqlens[num_seqs] = total_tokens.
 *                  Sequence s owns tokens cu_seqlens[s] .. cu_seqlens[s+1]-1
 *                  and attends only within itself (causal: local indices).
 *   max_seqlen   : >= the longest sequence (sizes the launch)
 *
 * Zero-length sequences are allowed and produce nothing.  The contents of
 * cu_seqlens are checked on the device; a violation skips the offending
 * sequence and is reported by fa_check_device_error() as
 * FA_ERR_INVALID_ARG.
 */
FA_API fa_status fa_fwd_varlen(const void *Q, const void *K, const void *V, void *O,
                        float *L, const int32_t *cu_seqlens, int num_seqs,
                        int total_tokens, int max_seqlen, int H, int D,
                        float scale, int causal, fa_dtype dtype,
                        fa_stream_t stream);

/*
 * fa_fwd_splitkv -- dense batch with each 256-row query block's keys cut into
 * `num_splits` contiguous ranges processed by separate work items, for
 * problems with too few (batch, head, query-block) units to fill the GPU
 * (small B*H, long N).  Each range produces a partial result normalised over
 * its own keys (O_g in fp32, L_g) in `workspace`; a merge kernel then
 * computes L = ln sum_g exp(L_g) and O = sum_g exp(L_g - L) O_g, which is the
 * online-softmax rescale of "FlashAttention -- for programmers, not
 * researchers.", STAGE 3, applied across ranges.  Same result as fa_fwd up
 * to rounding.
 *
 *   Q, K, V, O, L, B, H, N, D, scale, causal : as fa_fwd
 *   dtype           : FA_BF16 or FA_BF16_OUT_F32 (FA_F32: FA_ERR_UNSUPPORTED)
 *   num_splits      : 1..64, or 0 to choose automatically (enough work items
 *                     to cover the SMs); capped at ceil(N / 128)
 *   workspace       : caller-owned DEVICE memory, 16-byte aligned, at least
 *                     fa_fwd_splitkv_workspace_size(...) bytes; its contents
 *                     on entry do not matter and are garbage on exit.  May be
 *                     NULL when that size is 0 (a single split).
 *   workspace_bytes : its size
 *
 * Two kernels are enqueued on `stream`; calls that share a workspace must be
 * ordered on the GPU.
 */
FA_API fa_status fa_fwd_splitkv(const void *Q, const void *K, const void *V, void *O,
                                float *L, int B, int H, int N, int D, float scale,
                                int causal, fa_dtype dtype, int num_splits,
                                void *workspace, size_t workspace_bytes,
                                fa_stream_t stream);

/*
 * Workspace bytes fa_fwd_splitkv needs for these sizes and `num_splits`
 * (0 = the automatic choice, made for the current device).  Returns 0 when a
 * single split is used (or on an invalid size or a failed device query).
 */
FA_API size_t fa_fwd_splitkv_workspace_size(int B, int H, int N, int D,
                                            int num_splits);

/*
 * fa_fwd_splitkv_noalloc -- fa_fwd_splitkv for callers that cannot allocate
 * device memory: a plugin inside a host program that owns the device-memory
 * budget, a latency-critical caller that must not call cudaMalloc/cudaFree
 * (they can synchronise the device), or C code handed only its inputs and
 * outputs.  The pages have no counterpart of this entry point: it changes
 * where the split-key partials live, not what is computed.
 *
 * Arguments and results are those of fa_fwd_splitkv, without the workspace.
 * The partials go to one scratch array of FA_NOALLOC_SCRATCH_BYTES bytes in
 * the library, which every GPU that loads the library holds until the
 * process exits.  It calls no cudaMalloc, cudaFree or other allocating
 * routine.
 *
 *  - Sizes whose split workspace (fa_fwd_splitkv_workspace_size) exceeds
 *    FA_NOALLOC_SCRATCH_BYTES are rejected with FA_ERR_UNSUPPORTED before
 *    anything is enqueued.
 *  - The first call in a CUDA context looks up the array's device address
 *    there (a runtime query, no allocation); make that first call before any
 *    stream capture in the context.  The address belongs to the context: a
 *    new context (after cudaDeviceReset, or a host program's own driver-API
 *    context made current) gets its own lookup on its first call.
 *  - All calls share the array: calls that overlap on the GPU (other
 *    streams, other host threads) race on it.  Order them on one stream.
 */
#define FA_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)

FA_API fa_status fa_fwd_splitkv_noalloc(const void *Q, const void *K, const void *V,
                                        void *O, float *L, int B, int H, int N, int D,
                                        float scale, int causal, fa_dtype dtype,
                                        int num_splits, fa_stream_t stream);

/*
 * fa_fwd_host -- fa_fwd for inputs and outputs in HOST memory, with the
 * transfers overlapped with the computation.  The dense batch is cut into
 * `chunks` runs of consecutive (batch, head) problems.  Each run's Q, K, V go
 * host -> device on a copy stream, its forward pass runs on `stream` once
 * they have landed, and its O, L go device -> host on a second copy stream,
 * so both copy directions overlap the kernels of the neighbouring runs.  The
 * pages have no counterpart: this changes where the data lives, not what is
 * computed (the results are bitwise those of fa_fwd on the same data).
 *
 *   Qh, Kh, Vh : HOST [B, H, N, D] inputs.  Pinned memory (cudaHostAlloc or
 *                cudaHostRegister) gives the overlap; pageable memory works
 *                without it.
 *   Oh, Lh     : HOST outputs, [B, H, N, D] and [B, H, N] fp32
 *   Qd, Kd, Vd, Od, Ld : caller-owned DEVICE buffers of the full sizes (the
 *                staging area; same layout, alignment and overlap rules as
 *                fa_fwd's arguments).  Their contents on exit are the
 *                inputs and outputs of the pass.
 *   B, H, N, D, scale, causal, dtype : as fa_fwd
 *   chunks     : 1..64 runs (fewer if B*H is smaller).  Run boundaries fall
 *                on multiples of 4 / gcd(N, 4) problems, keeping every
 *                run's L slice 16-byte aligned.
 *   stream     : when the work on `stream` completes, Oh and Lh hold the
 *                results; the call itself returns after enqueueing.  Host
 *                buffers must stay valid until then.
 *
 * The two copy streams and the events that order the runs are created on a
 * device's first call and kept until the process exits.  Calls on one device
 * are enqueued under a lock and share them: concurrent calls are correct but
 * their runs serialise on the copy streams.
 *
 * Errors: FA_ERR_INVALID_ARG for a null host pointer, chunks outside 1..64
 * or any fa_fwd argument error, before anything is enqueued;
 * FA_ERR_UNSUPPORTED as fa_fwd; FA_ERR_CUDA if a copy, event or launch fails
 * (the stream still waits for every copy already enqueued).
 */
FA_API fa_status fa_fwd_host(const void *Qh, const void *Kh, const void *Vh, void *Oh,
                             float *Lh, void *Qd, void *Kd, void *Vd, void *Od, float *Ld,
                             int B, int H, int N, int D, float scale, int causal,
                             fa_dtype dtype, int chunks, fa_stream_t stream);

/*
 * fa_bwd -- gradients of the dense forward pass.  Given dO (the gradient of
 * a loss with respect to O), the forward inputs Q, K, V and the forward
 * outputs O and L, compute
 *
 *     P  = exp(scale * Q K^T - L)   (masked entries 0), recomputed tile by
 *                                    tile, never stored ("FlashAttention --
 *                                    for programmers, not researchers.",
 *                                    STAGE 5: keep only the per-row
 *                                    statistics, recompute the scores)
 *     dV = P^T dO,  dP = dO V^T,  dS = P * (dP - rowsum(dO * O)),
 *     dK = scale dS^T Q,  dQ = scale dS K
 *                                   (the five contractions of the
 *                                    "FlashAttention" docs page, section
 *                                    "Application in Backward Pass
 *                                    (5 MMAs)"; dS is the row-softmax
 *                                    derivative)
 *
 *   Q, K, V, O, dO : [B, H, N, D] contiguous; bf16 for FA_BF16 and
 *                    FA_BF16_OUT_F32, float32 for FA_F32.  O and L must be
 *                    the forward pass's outputs for the same Q, K, V,
 *                    scale and mask (O may be bf16-rounded).
 *   L              : [B, H, N] float32
 *   dQ, dK, dV     : [B, H, N, D] outputs: bf16 for FA_BF16, float32 for
 *                    FA_BF16_OUT_F32 and FA_F32.  They must not overlap any
 *                    input, each other or the workspace.
 *   workspace      : DEVICE memory of at least fa_bwd_workspace_size(B, H,
 *                    N) bytes, 16-byte aligned, owned by the caller; it
 *                    holds rowsum(dO * O) per row.  Contents on entry are
 *                    ignored.
 *
 * Deterministic: no atomics; dK/dV and dQ come from separate passes (dK and
 * dV owned by key blocks, dQ by query blocks), each summing in a fixed order.
 * Errors as fa_fwd, plus FA_ERR_INVALID_ARG for a short or null workspace.
 */
FA_API fa_status fa_bwd(const void *Q, const void *K, const void *V, const void *O,
                        const void *dO, const float *L, void *dQ, void *dK, void *dV, int B,
                        int H, int N, int D, float scale, int causal, fa_dtype dtype,
                        void *workspace, size_t workspace_bytes, fa_stream_t stream);

/* Workspace bytes fa_bwd needs: 4 * B * H * N rounded up to 256 (0 for an
 * empty problem or negative sizes). */
FA_API size_t fa_bwd_workspace_size(int B, int H, int N);

/*
 * fa_bwd_window -- gradients of the band forward pass (fa_fwd_window): the
 * operation of fa_bwd with key j visible to query i iff
 * i - window_left <= j <= i + window_right (-1: that side unbounded).
 * O and L must come from fa_fwd_window with the same window.  Arguments,
 * layouts, workspace and errors as fa_bwd; window bounds >= -1
 * (FA_ERR_INVALID_ARG otherwise).
 */
FA_API fa_status fa_bwd_window(const void *Q, const void *K, const void *V, const void *O,
                               const void *dO, const float *L, void *dQ, void *dK, void *dV, int B,
                               int H, int N, int D, float scale, int window_left, int window_right,
                               fa_dtype dtype, void *workspace, size_t workspace_bytes,
                               fa_stream_t stream);

/*
 * fa_bwd_varlen -- gradients of the packed-batch forward pass
 * (fa_fwd_varlen): the same operation as fa_bwd for every sequence and
 * head, with fa_fwd_varlen's layout.
 *
 *   Q, K, V, O, dO, dQ, dK, dV : [total_tokens, H, D] contiguous
 *   L                          : [H, total_tokens] float32
 *   cu_seqlens, num_seqs, max_seqlen : as fa_fwd_varlen (DEVICE int32
 *                  offsets, checked on the device; a violation skips the
 *                  sequence and is reported by fa_check_device_error())
 *   workspace      : at least fa_bwd_varlen_workspace_size(total_tokens, H)
 *                    bytes of DEVICE memory, 16-byte aligned (rowsum(dO * O),
 *                    laid out like L)
 *
 * Each sequence's rows and keys are its own: nothing crosses a sequence
 * boundary, so no buffer needs gaps between sequences.  Other arguments,
 * types and errors as fa_bwd.
 */
FA_API fa_status fa_bwd_varlen(const void *Q, const void *K, const void *V, const void *O,
                               const void *dO, const float *L, void *dQ, void *dK, void *dV,
                               const int32_t *cu_seqlens, int num_seqs, int total_tokens,
                               int max_seqlen, int H, int D, float scale, int causal,
                               fa_dtype dtype, void *workspace, size_t workspace_bytes,
                               fa_stream_t stream);

/* Workspace bytes fa_bwd_varlen needs: 4 * total_tokens * H rounded up to
 * 256 (0 for an empty problem or negative sizes). */
FA_API size_t fa_bwd_varlen_workspace_size(int total_tokens, int H);

/*
 * fa_check_device_error -- synchronise `stream`, then return (and clear)
 * the status recorded by kernels of this library on the current device:
 * FA_ERR_DEVICE_TIMEOUT if a device wait ran out, FA_ERR_INVALID_ARG if a
 * cu_seqlens check failed, FA_ERR_CUDA if the synchronisation itself
 * failed, else FA_OK.  This is the only entry point that blocks.
 */
FA_API fa_status fa_check_device_error(fa_stream_t stream);

/* Static, NUL-terminated description of a status code. */
FA_API const char *fa_status_string(fa_status status);

/*
 * fa_last_cuda_error -- after a call returned FA_ERR_CUDA, the CUDA runtime's
 * description of the failure (for example "too many resources requested for
 * launch"), recorded per calling thread; "no error" if none was recorded.
 * The string is static storage of the CUDA runtime.
 */
FA_API const char *fa_last_cuda_error(void);

/*
 * Process-wide knobs for tests and measurement (not thread-safe against
 * concurrent fa_fwd calls).
 *
 *   kernel        : FA_KERNEL_AUTO picks the tensor-core kernel for the
 *                   bf16 dtypes and the FFMA kernel for FA_F32; a bf16
 *                   problem the tensor-core kernel cannot take returns
 *                   FA_ERR_UNSUPPORTED (decided before any CUDA call) and
 *                   is never run on the FFMA kernel instead;
 *                   FA_KERNEL_SIMT forces the FFMA kernel for every dtype;
 *                   FA_KERNEL_TC forces the tensor-core kernel (bf16 only,
 *                   FA_ERR_UNSUPPORTED otherwise).
 *   grid_ctas     : persistent grid size of the tensor-core kernel; 0 means
 *                   one CTA per SM.  Results must not depend on it beyond
 *                   rounding (they are bitwise equal in practice: each
 *                   output row is computed by exactly one CTA in a fixed
 *                   order).
 *   wait_limit_ns : limit of every device-side wait; 0 means 2 s.
 */
typedef enum fa_kernel {
    FA_KERNEL_AUTO = 0,
    FA_KERNEL_SIMT = 1,
    FA_KERNEL_TC = 2
} fa_kernel;

typedef struct fa_options {
    int32_t kernel;
    int32_t grid_ctas;
    uint64_t wait_limit_ns;
} fa_options;

FA_API fa_status fa_set_options(const fa_options *opts);
FA_API fa_status fa_get_options(fa_options *opts);

/*
 * fa_watchdog_selftest -- enqueue one tiny kernel that waits, through the
 * same bounded-wait routine the attention kernels use, on an mbarrier that
 * nothing ever arrives on, with a limit of `limit_ns` nanoseconds (must be
 * in (0, 1e9]).  The wait runs out, the kernel records
 * FA_ERR_DEVICE_TIMEOUT and returns; the next fa_check_device_error()
 * reports it and the context stays usable.  Exists so the watchdog can be
 * tested without faulting or hanging a GPU.
 */
FA_API fa_status fa_watchdog_selftest(uint64_t limit_ns, fa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
