// Device-side helpers shared by the W4A16 kernels (sm_103a).
//
// Everything here is either a thin inline-PTX wrapper (bulk copies,
// mbarriers, cluster shared memory, streaming loads, warp MMA) or a bit-level
// conversion.  None of it is numerical library code.
#pragma once

#include <cstdint>
#include <cuda.h>  // CUtensorMap (the type only; no driver library is linked)
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "w4a16.h"

namespace w4a16 {

// ---------------------------------------------------------------------------
// bf16 <-> fp32 (bit level; bf16 is the top half of a binary32)
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_to_f32(uint32_t bits16) {
    return __uint_as_float(bits16 << 16);
}
__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}
// Output element idx of y: fp32, or bf16 rounded to nearest even.
__device__ __forceinline__ void store_out(void* y, int out_f32, size_t idx, float v) {
    if (out_f32) static_cast<float*>(y)[idx] = v;
    else static_cast<uint16_t*>(y)[idx] = f32_to_bf16_rn(v);
}
// SwiGLU element in fp32: silu(gate) * up with silu(v) = v / (1 + e^-v).
// Shared by the elementwise kernel and the expert kernel's fused staging so
// both round the same fp32 value to bf16.
__device__ __forceinline__ float silu_mul(float gte, float up) {
    return gte / (1.0f + expf(-gte)) * up;
}
// SwiGLU of a gate and an up product accumulated in fp32: both rounded to
// bf16 first (as a GEMV storing them would), then bf16(silu(gate) * up)
__device__ __forceinline__ uint16_t swiglu_of_sums(float gate, float up) {
    return f32_to_bf16_rn(silu_mul(bf16_to_f32(f32_to_bf16_rn(gate)), bf16_to_f32(f32_to_bf16_rn(up))));
}
// exact power of two 2^e for a normal exponent e in [-126, 127]
__device__ __forceinline__ float exp2i(int e) { return __int_as_float((127 + e) << 23); }

// ---------------------------------------------------------------------------
// Global loads
// ---------------------------------------------------------------------------
// Streamed, read-once data (packed weights): bypass L1 allocation.
__device__ __forceinline__ uint4 ldg_stream_u4(const uint4* p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ldg_nc_u16(const uint16_t* p) {
    unsigned short v;
    asm("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ldg_nc_u8(const uint8_t* p) {
    unsigned short v;
    asm("ld.global.nc.u8 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

// ---------------------------------------------------------------------------
// Shared memory, mbarrier and bulk (TMA engine) copies
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}
// As mbar_try_wait, but the thread may sleep up to `hint_ns` nanoseconds for
// the phase to complete instead of returning at once, so waiting warps do not
// take issue slots from working ones.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity,
                                                    uint32_t hint_ns) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return done != 0;
}
// Wait for phase `parity` of `bar`, bounded: at most max_iters sleeps of up to
// 100 microseconds each (about 0.8 s in all); false on timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint32_t max_iters = 8192) {
    for (uint32_t i = 0; i < max_iters; ++i)
        if (mbar_try_wait_sleep(bar, parity, 100000u)) return true;
    return false;
}
// Order this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (bulk copy) accesses to the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// 1-D bulk copy global -> this CTA's shared memory, completing on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Asynchronous copies of 16, 8 or 4 bytes global -> shared (cp.async), and an
// arrive on `bar` once all of this thread's earlier cp.async copies landed.
// The arrive does not raise the barrier's expected count, so the barrier's
// initial count must include every thread that performs it.
__device__ __forceinline__ void cp_async_16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_8(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_addr(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_4(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)), "l"(src)
                 : "memory");
}
// Wait until every cp.async this thread issued has landed.
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

// 2-D tiled bulk tensor copy global -> this CTA's shared memory through the
// tensor map `map` (a kernel parameter), box origin (c0, c1) in elements,
// completing on `bar` with the full box size in bytes (elements outside the
// tensor are filled with zeros).  c0 * element size must be a multiple of 16
// bytes; dst must be aligned as the map's swizzle mode requires (1024 bytes
// for the 128-byte swizzle).
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_addr(bar))
        : "memory");
}

// Fetch a tensor map (a __grid_constant__ kernel parameter) into the TMA
// unit's descriptor cache ahead of its first copy.
__device__ __forceinline__ void prefetch_tensor_map(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Four 8x8 matrices of 16-bit elements from shared memory: lanes 8i..8i+7
// give the 16-byte row addresses of matrix i; lane l receives, from each
// matrix, the 32-bit word at row l / 4, bytes 4 * (l % 4) .. + 3.
__device__ __forceinline__ void ldmatrix_x4(uint32_t (&d)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
                 : "r"(addr)
                 : "memory");
}

// ---------------------------------------------------------------------------
// Thread-block clusters (split-K partials are combined through DSMEM)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_barrier() {
    asm volatile(
        "barrier.cluster.arrive.release.aligned;\n\t"
        "barrier.cluster.wait.acquire.aligned;" ::
            : "memory");
}

// The two halves of a cluster barrier.  A kernel that stores into a peer
// CTA's shared memory arrives (relaxed) once its own shared memory is set up
// and waits before its first remote store, so every peer has started; the
// pair also makes one phase of the barrier, to be completed by every thread
// before the next arrive.
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

// Store into the shared memory of CTA `rank` of the cluster, at the offset
// local_ptr has in this CTA (fire-and-forget; a cluster barrier makes it
// visible to the owner).
__device__ __forceinline__ void st_dsmem_f32(float* local_ptr, uint32_t rank, float v) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                 : "=r"(remote)
                 : "r"(smem_addr(local_ptr)), "r"(rank));
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}

// Four floats into the shared memory of CTA `rank` of the cluster (16-byte
// aligned offset), fire-and-forget like st_dsmem_f32.
__device__ __forceinline__ void st_dsmem_f32x4(float* local_ptr, uint32_t rank, float4 v) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                 : "=r"(remote)
                 : "r"(smem_addr(local_ptr)), "r"(rank));
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(remote), "f"(v.x),
                 "f"(v.y), "f"(v.z), "f"(v.w)
                 : "memory");
}

// ---------------------------------------------------------------------------
// Warp MMA: D[16x8] (fp32) = A[16x16] (fp16, row) * B[16x8] (fp16, col) + D
// (A operand: a0 rows r, a1 rows r + 8, k pairs 2c, 2c+1; a2/a3 the same at
// k + 8; B: b0 k pairs 2c, 2c+1 of column r, b1 at k + 8; r = lane / 4,
// c = lane % 4, lower k in the low half of each register)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                              uint32_t a2, uint32_t a3, uint32_t b0,
                                              uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The same with a zero accumulator (the first product of a chain).
__device__ __forceinline__ void mma_f16_16816_zero(float (&d)[4], uint32_t a0, uint32_t a1,
                                                   uint32_t a2, uint32_t a3, uint32_t b0,
                                                   uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%10, %10, %10, %10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}

// Two 4-bit codes of a packed word as an fp16 pair, by one LOP3 with the
// exponent of 1024 (0x6400): (w & 0x000F000F) | 0x64006400 is
// {1024 + code at bits 0..3, 1024 + code at bits 16..19}, and
// (w & 0x00F000F0) | 0x64006400 is {1024 + 16 code(bits 4..7), 1024 + 16 code
// (bits 20..23)} -- both exact, as fp16 has ten fraction bits.
__device__ __forceinline__ uint32_t f16_codes_lo(uint32_t w) {
    uint32_t d;
    asm("lop3.b32 %0, %1, 0x000F000F, 0x64006400, 0xEA;" : "=r"(d) : "r"(w));
    return d;
}
__device__ __forceinline__ uint32_t f16_codes_hi(uint32_t w) {
    uint32_t d;
    asm("lop3.b32 %0, %1, 0x00F000F0, 0x64006400, 0xEA;" : "=r"(d) : "r"(w));
    return d;
}

// ---------------------------------------------------------------------------
// Warp MMA: D[16x8] (fp32) = A[16x16] (bf16, row) * B[16x8] (bf16, col) + C
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4],
                                               uint32_t b0, uint32_t b1, const float (&c)[4]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%10, %11, %12, %13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]),
          "f"(c[2]), "f"(c[3]));
}

// Programmatic dependent launch: let the next grid on the stream start its
// CTAs, and wait until the preceding grid has completed and its memory
// operations are visible (a no-op when launched without the attribute).
__device__ __forceinline__ void grid_dependents_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Barrier among `threads` threads (whole warps) of the CTA, id 1..15.
__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ void raise_device_error(uint32_t* err, uint32_t bits) {
    if (err) atomicOr(err, bits);
}

}  // namespace w4a16
