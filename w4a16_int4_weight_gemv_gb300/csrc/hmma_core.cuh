// Device helpers shared by the fp16 warp-MMA kernels (the dense GEMV and the
// routed expert FFN): activation scaling, zero points, cp.async group
// control and the hand-off of a split tile's partials.
#pragma once

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
template <int W>
__device__ __forceinline__ bool hand_partial(float4* red, uint64_t* gbar, int grp, int wpt, int part,
                                             int ti, int lane, float4 v) {
    const int b = ti & 1;
    uint64_t* full = gbar + (grp * 2 + b) * 2;
    bool ok = true;
    if (ti >= 2) ok = mbar_wait_bounded(full + 1, ((ti >> 1) - 1) & 1);
    red[(b * W + grp * wpt + part) * 32 + lane] = v;
    mbar_arrive(full);
    return ok;
}

}  // namespace
}  // namespace w4a16
