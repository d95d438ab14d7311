/*
 * A C caller of librlq.so: allocates device buffers with the CUDA runtime,
 * quantizes a bf16 activation (1x128 + fused 128x1) and a weight (128x128 with
 * transposed codes), runs FProp and DGrad, checks for device-side errors and
 * writes inputs and outputs to files for comparison with the Python binding.
 *
 * usage: example <out_dir>
 */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "rlq.h"

enum { M = 200, N = 384, K = 512, LDM = 208 /* M rounded up to 16 */ };

static uint32_t lcg(uint32_t *st)
{
    *st = *st * 1664525u + 1013904223u;
    return *st;
}

/* bf16 bits of a value drawn uniformly from about [-amp, amp] */
static uint16_t rnd_bf16(uint32_t *st, float amp)
{
    const float u = (float)(lcg(st) >> 8) * (1.0f / 16777216.0f);
    const float v = (2.0f * u - 1.0f) * amp;
    uint32_t b;
    memcpy(&b, &v, 4);
    return (uint16_t)((b + 0x7FFFu + ((b >> 16) & 1u)) >> 16);
}

static int save(const char *dir, const char *name, const void *dev, size_t bytes)
{
    char path[1024];
    snprintf(path, sizeof path, "%s/%s.bin", dir, name);
    void *h = malloc(bytes);
    if (!h || cudaMemcpy(h, dev, bytes, cudaMemcpyDeviceToHost) != cudaSuccess)
        return 1;
    FILE *f = fopen(path, "wb");
    if (!f)
        return 1;
    fwrite(h, 1, bytes, f);
    fclose(f);
    free(h);
    return 0;
}

#define CHECK(call)                                                                         \
    do {                                                                                    \
        const rlq_status st_ = (call);                                                      \
        if (st_ != RLQ_OK) {                                                                \
            fprintf(stderr, "%s: %s (%s)\n", #call, rlq_status_string(st_), rlq_last_error()); \
            return 1;                                                                       \
        }                                                                                   \
    } while (0)

int main(int argc, char **argv)
{
    if (argc != 2) {
        fprintf(stderr, "usage: %s <out_dir>\n", argv[0]);
        return 2;
    }
    const char *dir = argv[1];
    uint16_t *hx = malloc(sizeof(uint16_t) * M * K), *hw = malloc(sizeof(uint16_t) * N * K),
             *hdy = malloc(sizeof(uint16_t) * M * N);
    uint32_t st = 12345u;
    for (int i = 0; i < M * K; ++i)
        hx[i] = rnd_bf16(&st, 3.0f);
    for (int i = 0; i < N * K; ++i)
        hw[i] = rnd_bf16(&st, 0.05f);
    for (int i = 0; i < M * N; ++i)
        hdy[i] = rnd_bf16(&st, 0.002f);

    uint16_t *x, *w, *dy, *y, *dx;
    uint8_t *qx, *qxT, *qw, *qwT, *qdy;
    float *sx, *sxc, *sw, *sdy;
    cudaMalloc((void **)&x, sizeof(uint16_t) * M * K);
    cudaMalloc((void **)&w, sizeof(uint16_t) * N * K);
    cudaMalloc((void **)&dy, sizeof(uint16_t) * M * N);
    cudaMalloc((void **)&y, sizeof(uint16_t) * M * N);
    cudaMalloc((void **)&dx, sizeof(uint16_t) * M * K);
    cudaMalloc((void **)&qx, (size_t)M * K);
    cudaMalloc((void **)&qxT, (size_t)K * LDM);
    cudaMalloc((void **)&qw, (size_t)N * K);
    cudaMalloc((void **)&qwT, (size_t)K * N);
    cudaMalloc((void **)&qdy, (size_t)M * N);
    cudaMalloc((void **)&sx, sizeof(float) * (K / 128) * M);
    cudaMalloc((void **)&sxc, sizeof(float) * ((M + 127) / 128) * K);
    cudaMalloc((void **)&sw, sizeof(float) * (N / 128) * (K / 128));
    cudaMalloc((void **)&sdy, sizeof(float) * (N / 128) * M);
    cudaMemset(qxT, 0, (size_t)K * LDM);
    cudaMemcpy(x, hx, sizeof(uint16_t) * M * K, cudaMemcpyHostToDevice);
    cudaMemcpy(w, hw, sizeof(uint16_t) * N * K, cudaMemcpyHostToDevice);
    cudaMemcpy(dy, hdy, sizeof(uint16_t) * M * N, cudaMemcpyHostToDevice);

    cudaStream_t s;
    cudaStreamCreate(&s);
    rlq_stream_t rs = (rlq_stream_t)s;
    CHECK(rlq_quant_act_1x128(x, M, K, K, qx, K, sx, M, qxT, LDM, sxc, K, rs));
    CHECK(rlq_quant_weight_128x128(w, N, K, K, qw, K, sw, K / 128, qwT, N, rs));
    CHECK(rlq_quant_act_1x128(dy, M, N, N, qdy, N, sdy, M, NULL, 0, NULL, 0, rs));
    CHECK(rlq_gemm_fprop(qx, K, sx, M, qw, K, sw, K / 128, y, N, M, N, K, rs));
    CHECK(rlq_gemm_dgrad(qdy, N, sdy, M, qwT, N, 1, sw, K / 128, dx, K, M, N, K, rs));
    CHECK(rlq_check(rs));

    int bad = 0;
    bad |= save(dir, "x", x, sizeof(uint16_t) * M * K);
    bad |= save(dir, "w", w, sizeof(uint16_t) * N * K);
    bad |= save(dir, "dy", dy, sizeof(uint16_t) * M * N);
    bad |= save(dir, "qx", qx, (size_t)M * K);
    bad |= save(dir, "sx", sx, sizeof(float) * (K / 128) * M);
    bad |= save(dir, "qxT", qxT, (size_t)K * LDM);
    bad |= save(dir, "sxc", sxc, sizeof(float) * ((M + 127) / 128) * K);
    bad |= save(dir, "qw", qw, (size_t)N * K);
    bad |= save(dir, "sw", sw, sizeof(float) * (N / 128) * (K / 128));
    bad |= save(dir, "y", y, sizeof(uint16_t) * M * N);
    bad |= save(dir, "dx", dx, sizeof(uint16_t) * M * K);
    printf("librlq %s: ok\n", rlq_version());
    return bad;
}
