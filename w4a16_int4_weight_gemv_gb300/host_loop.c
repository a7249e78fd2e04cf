/*
 * A plain C caller of the library: decode-step GEMVs whose activations and
 * results live in page-locked host memory.  Each step copies x to the
 * device (cudaMemcpyAsync), runs w4a16_gemv on resident weights, copies y
 * back and waits for the stream -- what a host-side serving loop does per
 * token.  The benchmark builds it against libw4a16.so and reports its time
 * per step as the end-to-end figure of the C interface.
 *
 *   host_loop M N K g steps warmup
 *
 * (Capturing a step's three operations in a CUDA graph, one launch per
 * step, measured slower on one GB300: 25.7 against 24.5 us per step for
 * the 4096 x 4096 GEMV of one token.)
 *
 * Weights, scales and zero points are synthetic (a fixed xorshift stream:
 * uniform codes, scales from a small table of bf16 values near 0.01, zero
 * point 8); eight activation vectors rotate.  After the timed steps one
 * more step is checked bit for bit against the same GEMV run on device
 * buffers only.  Prints one JSON line; exits non-zero on any error.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include <time.h>

#include <cuda_runtime.h>

#include "w4a16.h"

static uint64_t rng_state = 0x9E3779B97F4A7C15ull;
static uint32_t next_u32(void) {
    rng_state ^= rng_state << 13;
    rng_state ^= rng_state >> 7;
    rng_state ^= rng_state << 17;
    return (uint32_t)(rng_state >> 32);
}

static double now_s(void) {
    struct timespec ts;
    clock_gettime(CLOCK_MONOTONIC, &ts);
    return (double)ts.tv_sec + 1e-9 * (double)ts.tv_nsec;
}

#define CK(call)                                                                  \
    do {                                                                          \
        cudaError_t e_ = (call);                                                  \
        if (e_ != cudaSuccess) {                                                  \
            fprintf(stderr, "%s: %s\n", #call, cudaGetErrorString(e_));           \
            return 1;                                                             \
        }                                                                         \
    } while (0)
#define CKW(call)                                                                 \
    do {                                                                          \
        w4a16_status s_ = (call);                                                 \
        if (s_ != W4A16_OK) {                                                     \
            fprintf(stderr, "%s: %s\n", #call, w4a16_status_string(s_));          \
            return 1;                                                             \
        }                                                                         \
    } while (0)

int main(int argc, char** argv) {
    if (argc != 7) {
        fprintf(stderr, "usage: %s M N K g steps warmup\n", argv[0]);
        return 2;
    }
    const int M = atoi(argv[1]);
    const int64_t N = atoll(argv[2]), K = atoll(argv[3]), g = atoll(argv[4]);
    const int steps = atoi(argv[5]), warmup = atoi(argv[6]);
    if (M < 1 || N < 1 || K < 1 || g < 1 || K % g != 0 || K % 8 != 0 || steps < 1 || warmup < 0)
        return 2;
    const size_t nwq = (size_t)N * (size_t)(K / 8), ng = (size_t)N * (size_t)(K / g);
    const size_t xb = (size_t)M * (size_t)K * 2, yb = (size_t)M * (size_t)N * 2;
    enum { NX = 8 };

    /* weights on the device, written once */
    uint32_t* h_wq = (uint32_t*)malloc(nwq * 4);
    uint16_t* h_s = (uint16_t*)malloc(ng * 2);
    uint8_t* h_z = (uint8_t*)malloc(ng);
    if (!h_wq || !h_s || !h_z) return 1;
    static const uint16_t scale_bits[4] = {0x3C24, 0x3C1F, 0x3C2A, 0x3C19}; /* ~0.009..0.0104 */
    for (size_t i = 0; i < nwq; ++i) h_wq[i] = next_u32();
    for (size_t i = 0; i < ng; ++i) {
        h_s[i] = scale_bits[next_u32() & 3];
        h_z[i] = 8;
    }
    uint32_t* d_wq;
    uint16_t *d_s, *d_x, *d_y, *d_yref;
    uint8_t* d_z;
    CK(cudaMalloc((void**)&d_wq, nwq * 4));
    CK(cudaMalloc((void**)&d_s, ng * 2));
    CK(cudaMalloc((void**)&d_z, ng));
    CK(cudaMalloc((void**)&d_x, xb));
    CK(cudaMalloc((void**)&d_y, yb));
    CK(cudaMalloc((void**)&d_yref, yb));
    CK(cudaMemcpy(d_wq, h_wq, nwq * 4, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(d_s, h_s, ng * 2, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(d_z, h_z, ng, cudaMemcpyHostToDevice));

    /* page-locked activations (bf16 of uniform values in [-1, 1)) and result */
    uint16_t* h_x[NX];
    uint16_t *h_y, *h_yref;
    for (int i = 0; i < NX; ++i) {
        CK(cudaHostAlloc((void**)&h_x[i], xb, cudaHostAllocDefault));
        for (size_t j = 0; j < xb / 2; ++j) {
            const float v = (float)((int32_t)(next_u32() >> 8) - (1 << 23)) / (float)(1 << 23);
            uint32_t bits;
            memcpy(&bits, &v, 4);
            h_x[i][j] = (uint16_t)(bits >> 16);
        }
    }
    CK(cudaHostAlloc((void**)&h_y, yb, cudaHostAllocDefault));
    CK(cudaHostAlloc((void**)&h_yref, yb, cudaHostAllocDefault));
    cudaStream_t st;
    CK(cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking));

    /* one step on activation buffer b */
#define STEP(b)                                                                            \
    do {                                                                                   \
        CK(cudaMemcpyAsync(d_x, h_x[(b)], xb, cudaMemcpyHostToDevice, st));                \
        CKW(w4a16_gemv(d_x, d_wq, d_s, d_z, d_y, W4A16_OUT_BF16, M, N, K, g, NULL, 0, st));    \
        CK(cudaMemcpyAsync(h_y, d_y, yb, cudaMemcpyDeviceToHost, st));                     \
        CK(cudaStreamSynchronize(st));                                                     \
    } while (0)
    for (int i = 0; i < warmup; ++i) STEP(i % NX);
    const double t0 = now_s();
    for (int i = 0; i < steps; ++i) STEP(i % NX);
    const double dt = (now_s() - t0) / (double)steps;

    /* the last step's result against the same GEMV on device buffers */
    CK(cudaMemcpy(d_x, h_x[(steps - 1) % NX], xb, cudaMemcpyHostToDevice));
    CKW(w4a16_gemv(d_x, d_wq, d_s, d_z, d_yref, W4A16_OUT_BF16, M, N, K, g, NULL, 0, st));
    CK(cudaStreamSynchronize(st));
    CK(cudaMemcpy(h_yref, d_yref, yb, cudaMemcpyDeviceToHost));
    const int same = memcmp(h_y, h_yref, yb) == 0;
    uint32_t err_bits = 0;
    CKW(w4a16_device_error(&err_bits, 1, st));

    printf("{\"us_per_step\": %.4f, \"steps\": %d, \"warmup\": %d, \"h2d_bytes_per_step\": %zu, "
           "\"d2h_bytes_per_step\": %zu, \"check\": \"%s\", \"device_error\": %u}\n",
           dt * 1e6, steps, warmup, xb, yb, same ? "bit-equal" : "MISMATCH", err_bits);
    return (same && err_bits == 0) ? 0 : 1;
}
