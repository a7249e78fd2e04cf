// Warp-MMA building blocks of the W4A16 kernels with 1 <= M <= 16 tokens
// (dense GEMV and expert-indexed GEMV).  Internal to the library.
//
// Dequantisation in registers.  For a 32-bit word of eight codes, the LOP3
// (w >> 4i) & 0x000F000F | 0x43004300 yields two bf16 values 128 + code for
// nibbles i and i + 4 (0x4300 is 128.0 and its 7-bit mantissa holds the code
// exactly).  The MMA thus accumulates sum_k (128 + code_k) x_k over a block
// of 128 k; since g % 128 == 0 the block lies in one quantisation group, and
//     sum_k (code_k - z) s x_k = s * (C - (128 + z) * sum_k x_k),
// applied once per block with the block's activation sums precomputed.
//
// K order.  The k order inside the MMA is free (a dot product does not depend
// on it), so the activations are staged in shared memory to match the words
// each lane holds.  Within a 32-bit word of codes k..k+7 the LOP3 above
// produces the pairs (k0,k4), (k1,k5), (k2,k6), (k3,k7), so every 16-byte
// piece of eight activations is stored as those four pairs.  The weights
// reach the lanes by ldmatrix from shared memory: lane (r, c) holds word c of
// each 16-byte chunk j of the block, k = 32 j + 8 c + e, so apart from the
// pairing the pieces keep their natural order (pair_x_in_place).
//
#pragma once

#include "common.cuh"

namespace w4a16 {

// Bytes between tokens in the permuted activation layout for nb 128-k blocks
// (== 64 mod 128, so the two tokens a quarter-warp reads hit different banks).
__host__ __device__ inline int mma_token_stride(int nb) { return nb * 256 + 64; }

// In-place form for the dense GEMV: m token rows of nb 128-k blocks were
// copied verbatim to xs (token stride tok_stride bytes); pair the values
// inside every 16-byte piece and write the per-block sums xsum[b][Mpad]
// (tokens >= m get 0).  When the (block, token) items fit four to a thread
// slot in one round, four lanes share an item (four pieces each, block sum
// by two shuffles); otherwise one thread takes a whole item, its 16 pieces
// loaded together and summed in four independent chains, so the pass is not
// a chain of dependent latencies.  Either way the piece order is rotated by
// lane so that the eight lanes of a load phase hit eight bank groups.
template <int NT>
__device__ __forceinline__ void pair_x_in_place(int m, int nb, unsigned char* xs, float* xsum,
                                                int tok_stride) {
    constexpr int Mpad = 8 * NT;
    const int items = m * nb;
    if (items * 4 <= static_cast<int>(blockDim.x)) {
        const int i = threadIdx.x >> 2;  // item; lanes 4i..4i+3 of the CTA share it
        const int qtr = threadIdx.x & 3;
        const bool ok = i < items;
        const int b = ok ? i / m : 0;
        const int n = ok ? i - b * m : 0;
        uint4* p = reinterpret_cast<uint4*>(xs + n * tok_stride + b * 256 + qtr * 64);
        const int rot = (threadIdx.x >> 1) & 3;  // differs between quarters 0/1 and 2/3 too
        uint4 v[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) v[q] = ok ? p[(q + rot) & 3] : make_uint4(0u, 0u, 0u, 0u);
        float s[2] = {0.f, 0.f};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint32_t w[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
                s[e & 1] += bf16_to_f32(w[e] & 0xFFFFu) + bf16_to_f32(w[e] >> 16);
        }
        float sum = s[0] + s[1];
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        if (ok) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint4 o4;
                o4.x = __byte_perm(v[q].x, v[q].z, 0x5410);  // (x0, x4)
                o4.y = __byte_perm(v[q].x, v[q].z, 0x7632);  // (x1, x5)
                o4.z = __byte_perm(v[q].y, v[q].w, 0x5410);  // (x2, x6)
                o4.w = __byte_perm(v[q].y, v[q].w, 0x7632);  // (x3, x7)
                p[(q + rot) & 3] = o4;
            }
            if (qtr == 0) xsum[b * Mpad + n] = sum;
        }
    } else {
    const int rot = threadIdx.x & 15;
    for (int i = threadIdx.x; i < items; i += blockDim.x) {
        const int b = i / m;
        const int n = i - b * m;
        uint4* p = reinterpret_cast<uint4*>(xs + n * tok_stride + b * 256);
        uint4 v[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) v[q] = p[(q + rot) & 15];
        float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            const uint32_t w[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
                s[e] += bf16_to_f32(w[e] & 0xFFFFu) + bf16_to_f32(w[e] >> 16);
            uint4 o4;
            o4.x = __byte_perm(v[q].x, v[q].z, 0x5410);  // (x0, x4)
            o4.y = __byte_perm(v[q].x, v[q].z, 0x7632);  // (x1, x5)
            o4.z = __byte_perm(v[q].y, v[q].w, 0x5410);  // (x2, x6)
            o4.w = __byte_perm(v[q].y, v[q].w, 0x7632);  // (x3, x7)
            p[(q + rot) & 15] = o4;
        }
        xsum[b * Mpad + n] = (s[0] + s[1]) + (s[2] + s[3]);
    }
    }
    for (int i = threadIdx.x; i < nb * (Mpad - m); i += blockDim.x) {
        const int b = i / (Mpad - m);
        xsum[b * Mpad + m + (i - b * (Mpad - m))] = 0.f;
    }
}

// Packed codes, scale and zero of one thread for one 128-k block of a 16-row
// tile: rows r and r + 8 (r = lane / 4).
struct MmaBlockLoad {
    uint4 w0, w1;
    uint32_t sz0, sz1;  // scale bits | zero << 16
};

// One 128-k block of a 16-row tile: accumulate into acc[NT][4] (C-fragment
// layout: rows r, r + 8; tokens 2c, 2c + 1 of each 8-token tile).
//   xb: permuted x of this block for token 0; tokens >= m read as zero
//   xsb: activation sums of this block, [Mpad]
template <int NT>
__device__ __forceinline__ void mma_block(float (&acc)[NT][4], const MmaBlockLoad& L,
                                          const unsigned char* xb, const float* xsb,
                                          int tok_stride, int m, int lane) {
    const int c = lane & 3;
    const int n = lane >> 2;
    const uint32_t r0[4] = {L.w0.x, L.w0.y, L.w0.z, L.w0.w};
    const uint32_t r1[4] = {L.w1.x, L.w1.y, L.w1.z, L.w1.w};
    // two independent accumulation chains (h = 0, 1), added at the end
    float cacc[2][NT][4];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int i = 0; i < 4; ++i) cacc[h][t][i] = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t bq[NT][4];
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (t * 8 + n < m)
                v = *reinterpret_cast<const uint4*>(xb + (t * 8 + n) * tok_stride + j * 64 +
                                                    c * 16);
            bq[t][0] = v.x;
            bq[t][1] = v.y;
            bq[t][2] = v.z;
            bq[t][3] = v.w;
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t a_lo0 = ((r0[j] >> (8 * h)) & 0x000F000Fu) | 0x43004300u;
            const uint32_t a_hi0 = ((r0[j] >> (8 * h + 4)) & 0x000F000Fu) | 0x43004300u;
            const uint32_t a_lo1 = ((r1[j] >> (8 * h)) & 0x000F000Fu) | 0x43004300u;
            const uint32_t a_hi1 = ((r1[j] >> (8 * h + 4)) & 0x000F000Fu) | 0x43004300u;
            const uint32_t a[4] = {a_lo0, a_lo1, a_hi0, a_hi1};
#pragma unroll
            for (int t = 0; t < NT; ++t)
                mma_bf16_16816(cacc[h][t], a, bq[t][2 * h], bq[t][2 * h + 1], cacc[h][t]);
        }
    }
    const float s0 = __uint_as_float(L.sz0 << 16);
    const float s1 = __uint_as_float(L.sz1 << 16);
    const float o0 = __uint_as_float(__byte_perm(L.sz0, 0x4B000000u, 0x7542)) - (8388608.f - 128.f);
    const float o1 = __uint_as_float(__byte_perm(L.sz1, 0x4B000000u, 0x7542)) - (8388608.f - 128.f);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        const float2 xs2 = *reinterpret_cast<const float2*>(xsb + t * 8 + 2 * c);
        acc[t][0] = fmaf(s0, fmaf(-o0, xs2.x, cacc[0][t][0] + cacc[1][t][0]), acc[t][0]);
        acc[t][1] = fmaf(s0, fmaf(-o0, xs2.y, cacc[0][t][1] + cacc[1][t][1]), acc[t][1]);
        acc[t][2] = fmaf(s1, fmaf(-o1, xs2.x, cacc[0][t][2] + cacc[1][t][2]), acc[t][2]);
        acc[t][3] = fmaf(s1, fmaf(-o1, xs2.y, cacc[0][t][3] + cacc[1][t][3]), acc[t][3]);
    }
}


}  // namespace w4a16
