/*
 * A plain C caller of the library: no Python, no torch.  It reads Q, K, V
 * and dO (float32, [B, H, N, D] contiguous) from a binary file and calls
 * the C ABI on device memory it allocates itself.
 *
 *   float32 mode (default): the forward pass (fa_fwd) and the backward pass
 *   (fa_bwd) in float32 on the FFMA kernels; writes O, L, dQ, dK, dV.
 *
 *   bf16 mode (ninth argument "bf16"): Q, K, V rounded to bf16 here, then
 *   the forward pass on the tensor-core kernel (selected explicitly with
 *   FA_KERNEL_TC, so that a call it could not take fails instead of running
 *   elsewhere), once with fp32 O (FA_BF16_OUT_F32) and once with bf16 O
 *   (FA_BF16); writes O (fp32), L, O (bf16, widened to float32), L.
 *
 * Usage:
 *
 *     abi_demo <in.bin> <out.bin> B H N D causal scale [bf16]
 */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

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

/* float32 -> bf16 bits, round to nearest even (finite inputs) */
static uint16_t to_bf16(float x) {
    uint32_t u;
    memcpy(&u, &x, 4);
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static float from_bf16(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float x;
    memcpy(&x, &u, 4);
    return x;
}

static int write_file(const char *path, const void *p, size_t n) {
    FILE *f = fopen(path, "wb");
    if (!f || fwrite(p, 1, n, f) != n) {
        fprintf(stderr, "cannot write %s\n", path);
        return 1;
    }
    fclose(f);
    return 0;
}

static int run_bf16(const float *host, const char *out_path, int B, int H, int N, int D, int causal,
                    float scale) {
    const size_t elems = (size_t)B * H * N * D, rows = (size_t)B * H * N;
    const size_t hb = elems * sizeof(uint16_t), fb = elems * sizeof(float), lb = rows * sizeof(float);
    uint16_t *h16 = (uint16_t *)malloc(3 * hb);
    float *out = (float *)malloc(2 * fb + 2 * lb);
    uint16_t *o16h = (uint16_t *)malloc(hb);
    if (!h16 || !out || !o16h) return 1;
    for (size_t i = 0; i < 3 * elems; ++i) h16[i] = to_bf16(host[i]);

    void *q, *k, *v, *o16;
    float *o32, *l1, *l2;
    CHECK_CUDA(cudaMalloc(&q, hb));
    CHECK_CUDA(cudaMalloc(&k, hb));
    CHECK_CUDA(cudaMalloc(&v, hb));
    CHECK_CUDA(cudaMalloc(&o16, hb));
    CHECK_CUDA(cudaMalloc((void **)&o32, fb));
    CHECK_CUDA(cudaMalloc((void **)&l1, lb));
    CHECK_CUDA(cudaMalloc((void **)&l2, lb));
    CHECK_CUDA(cudaMemcpy(q, h16, hb, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(k, h16 + elems, hb, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(v, h16 + 2 * elems, hb, cudaMemcpyHostToDevice));

    fa_options opts;
    CHECK_FA(fa_get_options(&opts));
    opts.kernel = FA_KERNEL_TC;
    CHECK_FA(fa_set_options(&opts));
    CHECK_FA(fa_fwd(q, k, v, o32, l1, B, H, N, D, scale, causal, FA_BF16_OUT_F32, NULL));
    CHECK_FA(fa_fwd(q, k, v, o16, l2, B, H, N, D, scale, causal, FA_BF16, NULL));
    CHECK_FA(fa_check_device_error(NULL));

    CHECK_CUDA(cudaMemcpy(out, o32, fb, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(out + elems, l1, lb, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(o16h, o16, hb, cudaMemcpyDeviceToHost));
    for (size_t i = 0; i < elems; ++i) out[elems + rows + i] = from_bf16(o16h[i]);
    CHECK_CUDA(cudaMemcpy(out + 2 * elems + rows, l2, lb, cudaMemcpyDeviceToHost));
    return write_file(out_path, out, 2 * fb + 2 * lb);
}

int main(int argc, char **argv) {
    if (argc != 9 && argc != 10) {
        fprintf(stderr, "usage: abi_demo in.bin out.bin B H N D causal scale [bf16]\n");
        return 1;
    }
    const int B = atoi(argv[3]), H = atoi(argv[4]), N = atoi(argv[5]), D = atoi(argv[6]);
    const int causal = atoi(argv[7]);
    const float scale = (float)atof(argv[8]);
    const int bf16 = argc == 10 && strcmp(argv[9], "bf16") == 0;
    if (argc == 10 && !bf16) {
        fprintf(stderr, "unknown mode %s\n", argv[9]);
        return 1;
    }
    const size_t elems = (size_t)B * H * N * D, rows = (size_t)B * H * N;
    const size_t tb = elems * sizeof(float), lb = rows * sizeof(float);

    float *host = (float *)malloc(4 * tb);
    FILE *f = fopen(argv[1], "rb");
    if (!host || !f || fread(host, 1, 4 * tb, f) != 4 * tb) {
        fprintf(stderr, "cannot read %s\n", argv[1]);
        return 1;
    }
    fclose(f);
    if (bf16) {
        const int r = run_bf16(host, argv[2], B, H, N, D, causal, scale);
        if (r == 0) printf("ok\n");
        return r;
    }

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
    if (write_file(argv[2], out, 4 * tb + lb)) return 1;
    printf("ok\n");
    return 0;
}
