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
// on it), so the activations are staged in shared memory to match whatever
// words each lane holds.  Within a 32-bit word of codes k..k+7 the LOP3 above
// produces the pairs (k0,k4), (k1,k5), (k2,k6), (k3,k7), so every 16-byte
// piece of eight activations is stored as those four pairs.  Which word of
// which row a lane holds depends on how the weights were loaded:
//  - ldmatrix from shared memory (dense GEMV): lane (r, c) holds word c of
//    each 16-byte chunk j of the block, k = 32 j + 8 c + e, so the pieces stay
//    in their natural order (pair_x_in_place);
//  - one 16-byte global load per row (expert GEMV): lane (r, c) holds chunk c,
//    k = 32 c + 8 j + e, so piece (c, j) moves to position (j, c)
//    (stage_x_permuted).
//
#pragma once

#include "common.cuh"

namespace w4a16 {

// Bytes between tokens in the permuted activation layout for nb 128-k blocks
// (== 64 mod 128, so the two tokens a quarter-warp reads hit different banks).
__host__ __device__ inline int mma_token_stride(int nb) { return nb * 256 + 64; }

// Stage activation rows for k in [kbeg, kbeg + nb*128) into the permuted
// layout (m tokens, token stride tok_stride bytes) and their per-block sums
// xsum[b][Mpad] (tokens >= m get 0).  Token n is row rowsel[n] of x (row
// stride K, bf16), or row n when rowsel is null; rowsel[n] < 0 means zeros.
template <int NT>
__device__ __forceinline__ void stage_x_permuted(const uint16_t* __restrict__ x,
                                                 const int* rowsel, int m, int K, int kbeg,
                                                 int nb, unsigned char* xs, float* xsum,
                                                 int tok_stride) {
    constexpr int Mpad = 8 * NT;
    // 16-byte pieces: token n, block b, quad c, step-pair q -> 8 consecutive k.
    // The 16 pieces of one (token, block) are 16 consecutive i, i.e. 16
    // consecutive lanes of one warp, so the block sum is a 16-lane shuffle
    // reduction in the same pass (blockDim is a multiple of 32).
    const int pieces = m * nb * 16;
    for (int base = 0; base < pieces; base += blockDim.x) {
        const int i = base + threadIdx.x;
        const bool ok = i < pieces;
        const int n = ok ? i / (nb * 16) : 0;
        const int rem = i - n * nb * 16;
        const int b = rem >> 4;
        const int c = (rem >> 2) & 3;
        const int q = rem & 3;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        const int row = ok ? (rowsel ? rowsel[n] : n) : -1;
        if (row >= 0) {
            const int k = kbeg + b * 128 + c * 32 + q * 8;
            v = __ldg(reinterpret_cast<const uint4*>(x + static_cast<size_t>(row) * K + k));
        }
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        float sum = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) sum += bf16_to_f32(w[e] & 0xFFFFu) + bf16_to_f32(w[e] >> 16);
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (ok) {
            uint4 o4;
            o4.x = __byte_perm(v.x, v.z, 0x5410);  // (x0, x4)
            o4.y = __byte_perm(v.x, v.z, 0x7632);  // (x1, x5)
            o4.z = __byte_perm(v.y, v.w, 0x5410);  // (x2, x6)
            o4.w = __byte_perm(v.y, v.w, 0x7632);  // (x3, x7)
            *reinterpret_cast<uint4*>(xs + n * tok_stride + b * 256 + q * 64 + c * 16) = o4;
            if ((rem & 15) == 0) xsum[b * Mpad + n] = sum;
        }
    }
    // tokens m..Mpad-1 contribute nothing
    for (int i = threadIdx.x; i < nb * (Mpad - m); i += blockDim.x) {
        const int b = i / (Mpad - m);
        xsum[b * Mpad + m + (i - b * (Mpad - m))] = 0.f;
    }
}

// In-place form for the dense GEMV: m token rows of nb 128-k blocks were
// copied verbatim to xs (token stride tok_stride bytes); pair the values
// inside every 16-byte piece and write the per-block sums xsum[b][Mpad]
// (tokens >= m get 0).  A thread takes a quarter block (four pieces, loaded
// together); the quarters of a block are four consecutive lanes, so the block
// sum is a 4-lane shuffle reduction.
template <int NT>
__device__ __forceinline__ void pair_x_in_place(int m, int nb, unsigned char* xs, float* xsum,
                                                int tok_stride) {
    constexpr int Mpad = 8 * NT;
    const int per_tok = nb * 4;
    const int items = m * per_tok;
    for (int base = 0; base < items; base += blockDim.x) {
        const int i = base + threadIdx.x;
        const bool ok = i < items;
        const int n = ok ? i / per_tok : 0;
        const int rem = ok ? i - n * per_tok : 0;  // block * 4 + quarter
        uint4* p = reinterpret_cast<uint4*>(xs + n * tok_stride + rem * 64);
        // piece order rotated by lane pair: the eight lanes of a 16-byte load
        // phase then touch eight different bank groups
        const int rot = (rem >> 1) & 3;
        uint4 v[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) v[q] = ok ? p[(q + rot) & 3] : make_uint4(0u, 0u, 0u, 0u);
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint32_t w[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                s0 += bf16_to_f32(w[e] & 0xFFFFu);
                s1 += bf16_to_f32(w[e] >> 16);
            }
        }
        float sum = s0 + s1;
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
            if ((rem & 3) == 0) xsum[(rem >> 2) * Mpad + n] = sum;
        }
    }
    for (int i = threadIdx.x; i < nb * (Mpad - m); i += blockDim.x) {
        const int b = i / (Mpad - m);
        xsum[b * Mpad + m + (i - b * (Mpad - m))] = 0.f;
    }
}

// Packed codes, scale and zero of one thread for one 128-k block of a 16-row
// tile: rows r and r + 8 (r = lane / 4), 32 consecutive k each.
struct MmaBlockLoad {
    uint4 w0, w1;
    uint32_t sz0, sz1;  // scale bits | zero << 16
};

__device__ __forceinline__ void mma_block_issue(MmaBlockLoad& L, const uint4* wq,
                                                const uint16_t* scale, const uint8_t* zero,
                                                int N, int Q, int G, int g, int tile, int blk,
                                                int lane) {
    const int r = lane >> 2;
    const int c = lane & 3;
    const int grp = (blk << 7) / g;
    const int n0 = tile * 16 + r;
    const int n1 = n0 + 8;
    const int chunk = blk * 4 + c;
    if (n0 < N) {
        L.w0 = ldg_stream_u4(wq + static_cast<size_t>(n0) * Q + chunk);
        const size_t gi = static_cast<size_t>(n0) * G + grp;
        L.sz0 = ldg_nc_u16(scale + gi) | (ldg_nc_u8(zero + gi) << 16);
    } else {
        L.w0 = make_uint4(0u, 0u, 0u, 0u);
        L.sz0 = 0u;
    }
    if (n1 < N) {
        L.w1 = ldg_stream_u4(wq + static_cast<size_t>(n1) * Q + chunk);
        const size_t gi = static_cast<size_t>(n1) * G + grp;
        L.sz1 = ldg_nc_u16(scale + gi) | (ldg_nc_u8(zero + gi) << 16);
    } else {
        L.w1 = make_uint4(0u, 0u, 0u, 0u);
        L.sz1 = 0u;
    }
}

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
