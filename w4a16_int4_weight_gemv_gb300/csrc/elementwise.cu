// Elementwise kernels around the W4A16 GEMV (sm_103a): packing 4-bit codes,
// expanding packed weights, and the SwiGLU activation of the expert chain.
//
// Packing order (problem statement accompanying the local-kimi README's
// technical-detail section): eight codes per 32-bit word, the first code
// along K in the lowest nibble.  Dequantisation: W = (code - zero) * scale.
//
// ~3-bit expert weights (the README's hardware-requirements paragraph asks
// for expert weights near three bits and gives no format; this library's
// INT3 format): every 32 consecutive codes of a row (a chunk) take three
// 32-bit words.  Codes 0..29 are 3-bit fields, ten per word, five in each
// 16-bit half at bits 0, 3, 6, 9, 12 (code i of the chunk in word i / 10,
// half (i % 10) / 5, field i % 5); codes 30 and 31 spread their bits over
// the spare bits 15 and 31 of the three words (bit j in word j).
#include "common.cuh"
#include "launch.h"

namespace w4a16 {
namespace {

// Four code bytes (one per byte lane, low nibble significant) -> 16 bits,
// code of byte i at bits 4i.
__device__ __forceinline__ uint32_t pack4(uint32_t b) {
    b &= 0x0F0F0F0Fu;
    b = (b | (b >> 4)) & 0x00FF00FFu;
    b = (b | (b >> 8)) & 0x0000FFFFu;
    return b;
}

__global__ void k_pack(const uint2* __restrict__ codes, uint32_t* __restrict__ wq, int64_t words) {
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < words;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const uint2 v = codes[i];
        wq[i] = pack4(v.x) | (pack4(v.y) << 16);
    }
}

// One thread per packed word: 8 consecutive weights of one row.
__global__ void k_dequant(const uint32_t* __restrict__ wq, const uint16_t* __restrict__ scale,
                          const uint8_t* __restrict__ zero, void* __restrict__ w, int out_f32,
                          int64_t N, int64_t K, int64_t g) {
    const int64_t words = N * (K / 8);
    const int64_t wpr = K / 8;
    const int64_t G = K / g;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < words;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t n = i / wpr;
        const int64_t k0 = (i - n * wpr) * 8;
        const int64_t gi = n * G + k0 / g;
        const float s = bf16_to_f32(scale[gi]);
        const int z = zero[gi];
        const uint32_t v = wq[i];
        float out[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int q = static_cast<int>((v >> (4 * j)) & 0xFu);
            out[j] = static_cast<float>(q - z) * s;  // exact: <= 5 x 8 significant bits
        }
        if (out_f32) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(w) + n * K + k0);
            dst[0] = make_float4(out[0], out[1], out[2], out[3]);
            dst[1] = make_float4(out[4], out[5], out[6], out[7]);
        } else {
            uint4 o;
            o.x = f32_to_bf16_rn(out[0]) | (static_cast<uint32_t>(f32_to_bf16_rn(out[1])) << 16);
            o.y = f32_to_bf16_rn(out[2]) | (static_cast<uint32_t>(f32_to_bf16_rn(out[3])) << 16);
            o.z = f32_to_bf16_rn(out[4]) | (static_cast<uint32_t>(f32_to_bf16_rn(out[5])) << 16);
            o.w = f32_to_bf16_rn(out[6]) | (static_cast<uint32_t>(f32_to_bf16_rn(out[7])) << 16);
            *reinterpret_cast<uint4*>(static_cast<uint16_t*>(w) + n * K + k0) = o;
        }
    }
}

// One thread per INT3 chunk: 32 code bytes -> 3 words.
__global__ void k_pack3(const uint4* __restrict__ codes, uint32_t* __restrict__ wq3, int64_t chunks) {
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < chunks;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const uint4 v0 = codes[2 * i], v1 = codes[2 * i + 1];
        const uint32_t b[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        uint32_t w[3] = {0u, 0u, 0u};
#pragma unroll
        for (int c = 0; c < 30; ++c) {
            const uint32_t q = (b[c >> 2] >> (8 * (c & 3))) & 7u;
            const int f = c % 10;
            w[c / 10] |= q << ((f >= 5 ? 16 : 0) + 3 * (f % 5));
        }
        const uint32_t q30 = (b[7] >> 16) & 7u, q31 = (b[7] >> 24) & 7u;
#pragma unroll
        for (int j = 0; j < 3; ++j) w[j] |= (((q30 >> j) & 1u) << 15) | (((q31 >> j) & 1u) << 31);
        wq3[3 * i] = w[0];
        wq3[3 * i + 1] = w[1];
        wq3[3 * i + 2] = w[2];
    }
}

// One thread per INT3 chunk: 32 consecutive weights of one row (a chunk
// never straddles a group: g % 32 == 0).
__global__ void k_dequant3(const uint32_t* __restrict__ wq3, const uint16_t* __restrict__ scale,
                           const uint8_t* __restrict__ zero, void* __restrict__ w, int out_f32,
                           int64_t N, int64_t K, int64_t g) {
    const int64_t cpr = K / 32;  // chunks per row
    const int64_t chunks = N * cpr;
    const int64_t G = K / g;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < chunks;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t n = i / cpr;
        const int64_t k0 = (i - n * cpr) * 32;
        const int64_t gi = n * G + k0 / g;
        const float s = bf16_to_f32(scale[gi]);
        const int z = zero[gi];
        const uint32_t w0 = wq3[3 * i], w1 = wq3[3 * i + 1], w2 = wq3[3 * i + 2];
        const uint32_t ws[3] = {w0, w1, w2};
        float out[32];
#pragma unroll
        for (int c = 0; c < 30; ++c) {
            const int f = c % 10;
            const int q = static_cast<int>((ws[c / 10] >> ((f >= 5 ? 16 : 0) + 3 * (f % 5))) & 7u);
            out[c] = static_cast<float>(q - z) * s;  // exact: <= 4 x 8 significant bits
        }
        const int q30 = static_cast<int>(((w0 >> 15) & 1u) | (((w1 >> 15) & 1u) << 1) | (((w2 >> 15) & 1u) << 2));
        const int q31 = static_cast<int>((w0 >> 31) | ((w1 >> 31) << 1) | ((w2 >> 31) << 2));
        out[30] = static_cast<float>(q30 - z) * s;
        out[31] = static_cast<float>(q31 - z) * s;
        if (out_f32) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(w) + n * K + k0);
#pragma unroll
            for (int j = 0; j < 8; ++j) dst[j] = make_float4(out[4 * j], out[4 * j + 1], out[4 * j + 2], out[4 * j + 3]);
        } else {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(w) + n * K + k0);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t o[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    o[e] = f32_to_bf16_rn(out[8 * j + 2 * e]) |
                           (static_cast<uint32_t>(f32_to_bf16_rn(out[8 * j + 2 * e + 1])) << 16);
                dst[j] = make_uint4(o[0], o[1], o[2], o[3]);
            }
        }
    }
}

// Two adjacent outputs per thread (N even, rows 4-byte aligned).
__global__ void k_swiglu(const uint16_t* __restrict__ gate, const uint16_t* __restrict__ up,
                         int64_t ld_in, uint16_t* __restrict__ h, int64_t ld_out, int64_t rows,
                         int64_t N) {
    const int64_t half = N / 2;
    const int64_t total = rows * half;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / half;
        const int64_t n = (i - r * half) * 2;
        const uint32_t gv = *reinterpret_cast<const uint32_t*>(gate + r * ld_in + n);
        const uint32_t uv = *reinterpret_cast<const uint32_t*>(up + r * ld_in + n);
        const float o0 = silu_mul(bf16_to_f32(gv & 0xFFFFu), bf16_to_f32(uv & 0xFFFFu));
        const float o1 = silu_mul(bf16_to_f32(gv >> 16), bf16_to_f32(uv >> 16));
        *reinterpret_cast<uint32_t*>(h + r * ld_out + n) =
            f32_to_bf16_rn(o0) | (static_cast<uint32_t>(f32_to_bf16_rn(o1)) << 16);
    }
}

// One warp waits, bounded, on an mbarrier that one arrival completes; with
// arrive == 0 nothing arrives and the wait expires after max_iters tries,
// which raises W4A16_DEVERR_TIMEOUT exactly as an expired wait in the GEMV
// and expert kernels does.
__global__ void k_wait_selftest(uint32_t max_iters, int arrive, uint32_t* err) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) mbar_init(&bar, 1);
    __syncwarp();
    if (arrive && threadIdx.x == 0) mbar_arrive(&bar);
    const bool ok = mbar_wait_bounded(&bar, 0, max_iters);
    if (!ok && threadIdx.x == 0) raise_device_error(err, W4A16_DEVERR_TIMEOUT);
}

int grid_for(int64_t items, int threads, int sms) {
    int64_t b = (items + threads - 1) / threads;
    const int64_t cap = static_cast<int64_t>(sms) * 8;
    if (b > cap) b = cap;
    if (b < 1) b = 1;
    return static_cast<int>(b);
}

}  // namespace

cudaError_t launch_pack(const uint8_t* codes, uint32_t* wq, int64_t N, int64_t K, int sms,
                        cudaStream_t s) {
    const int64_t words = N * (K / 8);
    if (words == 0) return cudaSuccess;
    k_pack<<<grid_for(words, 256, sms), 256, 0, s>>>(reinterpret_cast<const uint2*>(codes), wq,
                                                      words);
    return cudaGetLastError();
}

cudaError_t launch_dequant(const uint32_t* wq, const uint16_t* scale, const uint8_t* zero,
                           void* w, int out_f32, int64_t N, int64_t K, int64_t g, int sms,
                           cudaStream_t s) {
    const int64_t words = N * (K / 8);
    if (words == 0) return cudaSuccess;
    k_dequant<<<grid_for(words, 256, sms), 256, 0, s>>>(wq, scale, zero, w, out_f32, N, K, g);
    return cudaGetLastError();
}

cudaError_t launch_pack3(const uint8_t* codes, uint32_t* wq3, int64_t N, int64_t K, int sms,
                         cudaStream_t s) {
    const int64_t chunks = N * (K / 32);
    if (chunks == 0) return cudaSuccess;
    k_pack3<<<grid_for(chunks, 256, sms), 256, 0, s>>>(reinterpret_cast<const uint4*>(codes), wq3,
                                                        chunks);
    return cudaGetLastError();
}

cudaError_t launch_dequant3(const uint32_t* wq3, const uint16_t* scale, const uint8_t* zero,
                            void* w, int out_f32, int64_t N, int64_t K, int64_t g, int sms,
                            cudaStream_t s) {
    const int64_t chunks = N * (K / 32);
    if (chunks == 0) return cudaSuccess;
    k_dequant3<<<grid_for(chunks, 256, sms), 256, 0, s>>>(wq3, scale, zero, w, out_f32, N, K, g);
    return cudaGetLastError();
}

cudaError_t launch_wait_selftest(uint32_t max_iters, int arrive, uint32_t* err, cudaStream_t s) {
    k_wait_selftest<<<1, 32, 0, s>>>(max_iters, arrive, err);
    return cudaGetLastError();
}

cudaError_t launch_swiglu(const uint16_t* gate, const uint16_t* up, int64_t ld_in, uint16_t* h,
                          int64_t ld_out, int64_t rows, int64_t N, int sms, cudaStream_t s) {
    const int64_t total = rows * (N / 2);
    if (total == 0) return cudaSuccess;
    k_swiglu<<<grid_for(total, 256, sms), 256, 0, s>>>(gate, up, ld_in, h, ld_out, rows, N);
    return cudaGetLastError();
}

}  // namespace w4a16
