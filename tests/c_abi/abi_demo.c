/*
 * A plain C caller of the library: no Python, no torch.  It reads Q, K, V
 * and dO (float32, [B, H, N, D] contiguous) from a binary file, runs the
 * forward pass (fa_fwd) and the backward pass (fa_bwd) in float32 through
 * the C ABI on device memory it allocates itself, and writes O, L, dQ, dK,
 * dV to a second binary file.  Usage:
 *
 *     abi_demo <in.bin> <out.bin> B H N D causal scale
 */
#include <cuda_runtime.h>
#include <stdio.h>
#include <stdlib.h>

#include "fa.h"

#define CHECK_CUDA(x)                                                              \
    do {                                                                           \
        cudaError_t e_ = (x);                                                      \
        if (e_ != cudaSuccess) {                                                   \
            fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));               \
            return 2;                                                              \
        }                                                                          \
    } while (0)
#define CHECK_FA(x)                                                                \
    do {                                                                           \
        fa_status s_ = (x);                                                        \
        if (s_ != FA_OK) {                                                         \
            fprintf(stderr, "%s: %s\n", #x, fa_status_string(s_));                 \
            return 3;                                                              \
        }                                                                          \
    } while (0)

int main(int argc, char **argv) {
    if (argc != 9) {
        fprintf(stderr, "usage: abi_demo in.bin out.bin B H N D causal scale\n");
        return 1;
    }
    const int B = atoi(argv[3]), H = atoi(argv[4]), N = atoi(argv[5]), D = atoi(argv[6]);
    const int causal = atoi(argv[7]);
    const float scale = (float)atof(argv[8]);
    const size_t elems = (size_t)B * H * N * D, rows = (size_t)B * H * N;
    const size_t tb = elems * sizeof(float), lb = rows * sizeof(float);

    float *host = (float *)malloc(4 * tb);
    FILE *f = fopen(argv[1], "rb");
    if (!host || !f || fread(host, 1, 4 * tb, f) != 4 * tb) {
        fprintf(stderr, "cannot read %s\n", argv[1]);
        return 1;
    }
    fclose(f);

    float *q, *k, *v, *dout, *o, *l, *dq, *dk, *dv;
    void *ws;
    const size_t wsb = fa_bwd_workspace_size(B, H, N);
    CHECK_CUDA(cudaMalloc((void **)&q, tb));
    CHECK_CUDA(cudaMalloc((void **)&k, tb));
    CHECK_CUDA(cudaMalloc((void **)&v, tb));
    CHECK_CUDA(cudaMalloc((void **)&dout, tb));
    CHECK_CUDA(cudaMalloc((void **)&o, tb));
    CHECK_CUDA(cudaMalloc((void **)&l, lb));
    CHECK_CUDA(cudaMalloc((void **)&dq, tb));
    CHECK_CUDA(cudaMalloc((void **)&dk, tb));
    CHECK_CUDA(cudaMalloc((void **)&dv, tb));
    CHECK_CUDA(cudaMalloc(&ws, wsb));
    CHECK_CUDA(cudaMemcpy(q, host, tb, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(k, host + elems, tb, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(v, host + 2 * elems, tb, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dout, host + 3 * elems, tb, cudaMemcpyHostToDevice));

    /* the default stream: a null fa_stream_t */
    CHECK_FA(fa_fwd(q, k, v, o, l, B, H, N, D, scale, causal, FA_F32, NULL));
    CHECK_FA(fa_bwd(q, k, v, o, dout, l, dq, dk, dv, B, H, N, D, scale, causal, FA_F32, ws, wsb, NULL));
    CHECK_FA(fa_check_device_error(NULL));

    float *out = (float *)malloc(4 * tb + lb);
    CHECK_CUDA(cudaMemcpy(out, o, tb, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(out + elems, l, lb, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(out + elems + rows, dq, tb, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(out + 2 * elems + rows, dk, tb, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(out + 3 * elems + rows, dv, tb, cudaMemcpyDeviceToHost));
    f = fopen(argv[2], "wb");
    if (!f || fwrite(out, 1, 4 * tb + lb, f) != 4 * tb + lb) {
        fprintf(stderr, "cannot write %s\n", argv[2]);
        return 1;
    }
    fclose(f);
    printf("ok\n");
    return 0;
}
