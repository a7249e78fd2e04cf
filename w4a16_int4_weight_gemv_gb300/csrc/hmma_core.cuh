// Device helpers shared by the fp16 warp-MMA kernels (the dense GEMV and the
// routed expert FFN): activation scaling, zero points, cp.async group
// control and the hand-off of a split tile's partials.
#pragma once

#include <cuda_fp16.h>

#include "common.cuh"

namespace w4a16 {
namespace {

// exact 2^e for any integer e in [-252, 254], as the product of two normal
// powers of two (applied one after the other by the callers)
__device__ __forceinline__ void pow2_pair(int e, float& f1, float& f2) {
    const int e1 = e / 2;
    f1 = exp2i(e1);
    f2 = exp2i(e - e1);
}

// Shift of a block whose largest |x| has bf16 bits mb: the largest lands in
// [2^14, 2^15); blocks of subnormals or zeros get 2^126 (their products are
// below 2^-100 and exactness there is moot), so 2^-sh is a normal float.
__device__ __forceinline__ int block_shift(uint32_t mb) {
    int eb = static_cast<int>(mb >> 7);  // biased exponent of the largest |x|
    if (eb > 254) eb = 254;              // Inf / NaN: any shift, the result is not finite
    const int sh = 141 - eb;
    return sh > 126 ? 126 : sh;
}

// Largest |x| bits (bf16, sign cleared) of NP 8-k pieces of activations.
template <int NP>
__device__ __forceinline__ uint32_t pieces_absmax(const uint4 (&v)[NP]) {
    uint32_t m2 = 0u;
#pragma unroll
    for (int b = 0; b < NP; ++b) {
        m2 = __vmaxu2(m2, v[b].x & 0x7FFF7FFFu);
        m2 = __vmaxu2(m2, v[b].y & 0x7FFF7FFFu);
        m2 = __vmaxu2(m2, v[b].z & 0x7FFF7FFFu);
        m2 = __vmaxu2(m2, v[b].w & 0x7FFF7FFFu);
    }
    return max(m2 & 0xFFFFu, m2 >> 16);
}

// B fragments of an INT4 unit for NP consecutive 8-k pieces of one column
// (v[q] = the piece's x, bf16): a piece becomes the fp16 pairs
// {(x0, x4), (x1, x5) / 16, (x2, x6), (x3, x7) / 16} times 2^sh = fa * fb --
// the k order and scaling of the codes one LOP3 per two makes (odd codes
// carry a factor 16).  c1 and c2 gain the pieces' sum of B and of B times
// its code factor.
template <int NP>
__device__ __forceinline__ void int4_piece_fragments(const uint4 (&v)[NP], float fa, float fb, uint4 (&o)[NP],
                                                     float& c1, float& c2) {
    const float fo = fb * 0.0625f;
#pragma unroll
    for (int q = 0; q < NP; ++q) {
        const uint32_t w[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
            x[e] = __uint_as_float((e & 1) ? (w[e >> 1] & 0xFFFF0000u) : (w[e >> 1] << 16)) * fa;
        const __half2 h0 = __floats2half2_rn(x[0] * fb, x[4] * fb);
        const __half2 h1 = __floats2half2_rn(x[1] * fo, x[5] * fo);
        const __half2 h2 = __floats2half2_rn(x[2] * fb, x[6] * fb);
        const __half2 h3 = __floats2half2_rn(x[3] * fo, x[7] * fo);
        o[q] = make_uint4(*reinterpret_cast<const uint32_t*>(&h0), *reinterpret_cast<const uint32_t*>(&h1),
                          *reinterpret_cast<const uint32_t*>(&h2), *reinterpret_cast<const uint32_t*>(&h3));
        const float2 f0 = __half22float2(h0), f1 = __half22float2(h1);
        const float2 f2 = __half22float2(h2), f3 = __half22float2(h3);
        const float ev = (f0.x + f0.y) + (f2.x + f2.y);
        const float od = (f1.x + f1.y) + (f3.x + f3.y);
        c1 += ev + od;
        c2 += fmaf(16.f, od, ev);
    }
}

__device__ __forceinline__ float zero_point_f32(uint32_t bytes4, int b) {
    // byte b of bytes4 placed under the exponent of 2^23, minus 2^23
    return __uint_as_float(__byte_perm(bytes4, 0x4B000000u, 0x7540u + b)) - 8388608.f;
}

// wait until at most n of this thread's cp.async commit groups are pending
__device__ __forceinline__ void cp_async_wait_pending(int n) {
    switch (n) {
        case 0: asm volatile("cp.async.wait_group 0;" ::: "memory"); break;
        case 1: asm volatile("cp.async.wait_group 1;" ::: "memory"); break;
        case 2: asm volatile("cp.async.wait_group 2;" ::: "memory"); break;
        case 3: asm volatile("cp.async.wait_group 3;" ::: "memory"); break;
        case 4: asm volatile("cp.async.wait_group 4;" ::: "memory"); break;
        default: asm volatile("cp.async.wait_group 5;" ::: "memory"); break;
    }
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// Part `part` (> 0) of tile group `grp` (wpt parts) hands its partial of
// the group's ti-th tile to part 0 through buffer ti % 2 of `red` (W warps
// per CTA): it first waits until part 0 has read that buffer's previous
// contents (tile ti - 2), then writes and arrives on the buffer's `full`
// barrier.  False if the wait gave up.
// With NT 8-token MMA tiles the partials of tile t go to red + t * 2 * W * 32.
template <int W, int NT>
__device__ __forceinline__ bool hand_partials(float4* red, uint64_t* gbar, int grp, int wpt, int part,
                                              int ti, int lane, const float4 (&v)[NT]) {
    const int b = ti & 1;
    uint64_t* full = gbar + (grp * 2 + b) * 2;
    bool ok = true;
    if (ti >= 2) ok = mbar_wait_bounded(full + 1, ((ti >> 1) - 1) & 1);
#pragma unroll
    for (int t = 0; t < NT; ++t) red[t * 2 * W * 32 + (b * W + grp * wpt + part) * 32 + lane] = v[t];
    mbar_arrive(full);
    return ok;
}
template <int W>
__device__ __forceinline__ bool hand_partial(float4* red, uint64_t* gbar, int grp, int wpt, int part,
                                             int ti, int lane, float4 v) {
    const float4 one[1] = {v};
    return hand_partials<W, 1>(red, gbar, grp, wpt, part, ti, lane, one);
}

}  // namespace
}  // namespace w4a16
