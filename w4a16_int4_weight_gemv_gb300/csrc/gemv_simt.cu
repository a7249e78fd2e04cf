// M = 1 W4A16 GEMV on CUDA cores (sm_103a).
//
// The decode-time product of the local-kimi README, technical-detail section:
// one activation row against a group-quantised INT4 matrix, done as a true
// GEMV -- every lane walks the reduction axis K of its rows with 128-bit
// coalesced loads and keeps one fp32 accumulator per output row.
//
// Arithmetic.  For one 16-byte chunk (32 consecutive k of one row, all in one
// quantisation group because g % 32 == 0) the kernel forms
//     acc = sum_k code_k * x_k
// exactly-per-product in fp32 and then applies the group's zero point and
// scale once:  partial += s * (acc - z * sum_k x_k),  which equals
// sum_k (code_k - z) * s * x_k.
//
// Nibble -> float without conversion instructions: the bit pattern
// (word & (0xF << p)) read as a binary32 is code * 2^(p - 149) (a subnormal,
// or for p = 20 and code >= 8 the smallest normals, whose value is still the
// integer pattern times 2^-149).  Multiplying it by x * 2^(85 - p) gives
// code * x * 2^-64 exactly, so each weight costs one LOP3 and one FFMA (plus
// one shift per word for the top two nibbles, which are brought down by 8
// bits).  The 2^(85 - p) factors are folded into the staged activations once
// per CTA; the 2^64 is restored on the output.  FFMA keeps subnormal inputs
// (the library is built without flush-to-zero), and the exact product of an
// 8-bit-significand x and a 4-bit code is normal unless |code * x| < 2^-62.
// Inputs must satisfy |x| < 2^40 so that x * 2^85 stays finite.
//
// Data movement.  The CTA's slice of x is copied to shared memory with one
// bulk (TMA engine) copy, then expanded to the pre-scaled fp32 form x' with
// an XOR swizzle so that the 8 lanes of a quarter-warp read 8 distinct bank
// groups.  Weight loads for the first steps are issued before the copy is
// waited on, so DRAM latency overlaps the staging.  Each lane then reuses its
// 32 x' values across the TR rows of a tile.  When K is split (small N, or a
// slice too large for shared memory) the CTAs of a thread-block cluster take
// disjoint K slices of the same rows and the partial sums are added through
// distributed shared memory in rank order (deterministic, no workspace).
#include "common.cuh"
#include "launch.h"

namespace w4a16 {
namespace {

constexpr int kTR = 8;  // rows per tile
constexpr int kPD = 2;  // steps of loads kept in flight per lane
constexpr int kMaxWarps = 8;

struct SimtKernelArgs {
    const uint16_t* x;
    const uint4* wq;
    const uint16_t* scale;
    const uint8_t* zero;
    void* y;
    int out_f32;
    int N;
    int K;
    int g;
    int ksplit;
    int spans_per_cta;
    int tiles_per_cluster;
    uint32_t* err;
};

// x'[k] = x[k] * 2^(85 - p), p the bit offset the code of k sits at after the
// kernel's masking: nibbles 0..5 at 4*i, nibbles 6 and 7 (shifted down by 8) at 16 and 20.
__device__ __forceinline__ float position_factor(int i) {
    const int p = (i < 6) ? 4 * i : 4 * i - 8;
    return exp2i(85 - p);
}

__device__ __forceinline__ float dot_chunk(const uint4 w, const float (&xr)[32]) {
    float a0 = 0.f, a1 = 0.f;
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t v = ws[j];
        const uint32_t t = v >> 8;
        a0 = fmaf(__uint_as_float(v & 0x0000000Fu), xr[8 * j + 0], a0);
        a1 = fmaf(__uint_as_float(v & 0x000000F0u), xr[8 * j + 1], a1);
        a0 = fmaf(__uint_as_float(v & 0x00000F00u), xr[8 * j + 2], a0);
        a1 = fmaf(__uint_as_float(v & 0x0000F000u), xr[8 * j + 3], a1);
        a0 = fmaf(__uint_as_float(v & 0x000F0000u), xr[8 * j + 4], a0);
        a1 = fmaf(__uint_as_float(v & 0x00F00000u), xr[8 * j + 5], a1);
        a0 = fmaf(__uint_as_float(t & 0x000F0000u), xr[8 * j + 6], a0);
        a1 = fmaf(__uint_as_float(t & 0x00F00000u), xr[8 * j + 7], a1);
    }
    return a0 + a1;
}

struct SimtSmem {
    uint64_t* bar;
    uint16_t* xraw;  // bf16 slice as copied
    float* xs;       // pre-scaled, swizzled x' (1024 floats per span)
    float* xsum;     // per chunk: sum of x * 2^-64
    float* red;      // [warps][kTR]
    float* part;     // [tiles_per_cluster][kTR] split-K partials
};

__device__ __forceinline__ SimtSmem carve(unsigned char* smem, int spans, int warps) {
    SimtSmem s;
    s.bar = reinterpret_cast<uint64_t*>(smem);
    s.xraw = reinterpret_cast<uint16_t*>(smem + 16);
    s.xs = reinterpret_cast<float*>(smem + 16 + spans * 2048);
    s.xsum = s.xs + spans * 1024;
    s.red = s.xsum + spans * 32;
    s.part = s.red + warps * kTR;
    return s;
}

__global__ void __launch_bounds__(kMaxWarps * 32)
k_gemv_m1(const SimtKernelArgs a) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int W = blockDim.x >> 5;
    const int Q = a.K >> 5;                   // 16-byte chunks per row
    const int nspan_all = (Q + 31) >> 5;      // 32-chunk spans per row
    const int S = a.ksplit;
    const int rank = (S > 1) ? static_cast<int>(cluster_rank()) : 0;
    const int cid = blockIdx.x / S;
    const int ncl = gridDim.x / S;
    const int SP = a.spans_per_cta;
    const int span0 = rank * SP;
    const int nspan = max(0, min(nspan_all, span0 + SP) - span0);
    const int kbeg = span0 << 10;
    const int kend = min(a.K, (span0 + nspan) << 10);
    const int ntiles = (a.N + kTR - 1) / kTR;
    const int G = a.K / a.g;
    const int cpg = a.g >> 5;                 // chunks per quantisation group
    SimtSmem sm = carve(smem_raw, SP, W);

    // 1. bulk copy of this CTA's x slice
    if (threadIdx.x == 0) {
        mbar_init(sm.bar, 1);
        mbar_init_fence();
    }
    __syncthreads();
    if (threadIdx.x == 0 && kend > kbeg) {
        const uint32_t bytes = static_cast<uint32_t>(kend - kbeg) * 2u;
        mbar_arrive_expect_tx(sm.bar, bytes);
        bulk_copy_g2s(sm.xraw, a.x + kbeg, bytes, sm.bar);
    }

    // 2. work of this warp: tiles cid, cid + ncl, ...; spans warp, warp + W, ...
    const int my_tiles = (ntiles > cid) ? (ntiles - cid + ncl - 1) / ncl : 0;
    const int my_spans = (nspan > warp) ? (nspan - warp + W - 1) / W : 0;
    const int nsteps = my_tiles * my_spans;

    uint4 wb[kPD][kTR];
    uint32_t sz[kPD][kTR];  // scale bits | zero << 16

    auto issue = [&](int s, uint4 (&wv)[kTR], uint32_t (&szv)[kTR]) {
        const int ti = s / my_spans;
        const int si = s - ti * my_spans;
        const int tile = cid + ti * ncl;
        const int c = ((span0 + warp + si * W) << 5) + lane;  // global chunk
        const bool cok = c < Q;
        const int grp = c / cpg;
#pragma unroll
        for (int r = 0; r < kTR; ++r) {
            const int n = tile * kTR + r;
            if (cok && n < a.N) {
                wv[r] = ldg_stream_u4(a.wq + static_cast<size_t>(n) * Q + c);
                const size_t gi = static_cast<size_t>(n) * G + grp;
                szv[r] = ldg_nc_u16(a.scale + gi) | (ldg_nc_u8(a.zero + gi) << 16);
            } else {
                wv[r] = make_uint4(0u, 0u, 0u, 0u);
                szv[r] = 0u;
            }
        }
    };

#pragma unroll
    for (int p = 0; p < kPD; ++p)
        if (p < nsteps) issue(p, wb[p], sz[p]);

    // 3. wait for x, expand to x' and chunk sums
    bool ok = true;
    if (kend > kbeg) ok = mbar_wait_bounded(sm.bar, 0);
    if (!ok && threadIdx.x == 0) raise_device_error(a.err, W4A16_DEVERR_TIMEOUT);
    ok = __syncthreads_and(ok);
    const int nk = nspan << 10;
    for (int i = threadIdx.x; i < (nk >> 2); i += blockDim.x) {
        const int k0 = i << 2;
        const int cl = k0 >> 5;
        const int q = (k0 >> 2) & 7;
        float v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int k = k0 + e;
            const float xv = (ok && kbeg + k < kend) ? bf16_to_f32(sm.xraw[k]) : 0.f;
            v[e] = xv * position_factor(k & 7);
        }
        *reinterpret_cast<float4*>(sm.xs + cl * 32 + ((q ^ (cl & 7)) << 2)) =
            make_float4(v[0], v[1], v[2], v[3]);
    }
    for (int cl = threadIdx.x; cl < (nk >> 5); cl += blockDim.x) {
        float sum = 0.f;
        for (int i = 0; i < 32; ++i) {
            const int k = (cl << 5) + i;
            sum += (ok && kbeg + k < kend) ? bf16_to_f32(sm.xraw[k]) : 0.f;
        }
        sm.xsum[cl] = sum * exp2i(-64);
    }
    __syncthreads();

    // 4. stream the weights
    float acc[kTR];
#pragma unroll
    for (int r = 0; r < kTR; ++r) acc[r] = 0.f;
    int ti = 0, si = 0;

    auto tile_end = [&]() {
#pragma unroll
        for (int r = 0; r < kTR; ++r) {
            float v = acc[r];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if (lane == 0) sm.red[warp * kTR + r] = v;
            acc[r] = 0.f;
        }
        __syncthreads();
        if (threadIdx.x < kTR) {
            float v = 0.f;
            for (int w = 0; w < W; ++w) v += sm.red[w * kTR + threadIdx.x];
            const int tile = cid + ti * ncl;
            const int n = tile * kTR + threadIdx.x;
            if (S == 1) {
                if (n < a.N) {
                    v *= exp2i(64);
                    if (a.out_f32) static_cast<float*>(a.y)[n] = v;
                    else static_cast<uint16_t*>(a.y)[n] = f32_to_bf16_rn(v);
                }
            } else {
                sm.part[ti * kTR + threadIdx.x] = v;
            }
        }
        __syncthreads();
    };

    for (int s0 = 0; s0 < nsteps; s0 += kPD) {
#pragma unroll
        for (int p = 0; p < kPD; ++p) {
            const int s = s0 + p;
            if (s < nsteps) {
                const int cl = ((warp + si * W) << 5) + lane;  // chunk within the slice
                if (((span0 << 5) + cl) < Q) {
                    float xr[32];
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const float4 t = *reinterpret_cast<const float4*>(
                            sm.xs + cl * 32 + ((q ^ (cl & 7)) << 2));
                        xr[4 * q + 0] = t.x;
                        xr[4 * q + 1] = t.y;
                        xr[4 * q + 2] = t.z;
                        xr[4 * q + 3] = t.w;
                    }
                    const float xc = sm.xsum[cl];
#pragma unroll
                    for (int r = 0; r < kTR; ++r) {
                        const float d = dot_chunk(wb[p][r], xr);
                        const float sc = __uint_as_float(sz[p][r] << 16);
                        const float zf =
                            __uint_as_float(__byte_perm(sz[p][r], 0x4B000000u, 0x7542)) -
                            8388608.f;
                        acc[r] = fmaf(sc, fmaf(-zf, xc, d), acc[r]);
                    }
                }
                if (s + kPD < nsteps) issue(s + kPD, wb[p], sz[p]);
                if (++si == my_spans) {
                    si = 0;
                    tile_end();
                    ++ti;
                }
            }
        }
    }
    // warps with no span still take part in every tile's reduction
    if (my_spans == 0)
        for (; ti < my_tiles; ++ti) tile_end();

    // 5. split-K: add the cluster's partials in rank order through DSMEM
    if (S > 1) {
        cluster_barrier();
        for (int idx = threadIdx.x; idx < my_tiles * kTR; idx += blockDim.x) {
            const int t = idx / kTR;
            if (t % S != rank) continue;
            float v = 0.f;
            for (int r = 0; r < S; ++r) v += ld_dsmem_f32(sm.part + idx, static_cast<uint32_t>(r));
            const int n = (cid + t * ncl) * kTR + (idx - t * kTR);
            if (n < a.N) {
                v *= exp2i(64);
                if (a.out_f32) static_cast<float*>(a.y)[n] = v;
                else static_cast<uint16_t*>(a.y)[n] = f32_to_bf16_rn(v);
            }
        }
        cluster_barrier();
    }
}

int smem_bytes_simt(int spans, int warps, int tiles_per_cluster, int S) {
    return 16 + spans * (2048 + 4096 + 128) + warps * kTR * 4 +
           (S > 1 ? tiles_per_cluster * kTR * 4 : 0);
}

}  // namespace

GemvPlan plan_gemv_simt(const DeviceInfo& dev, int N, int K, int k_split_req) {
    GemvPlan p{};
    p.kernel_id = 1;
    const int Q = K / 32;
    const int nspan_all = (Q + 31) / 32;
    const int ntiles = (N + kTR - 1) / kTR;
    const int budget = dev.max_smem_optin - 1024;
    // K split: forced, or enough to fit shared memory, or to fill the SMs when N is small
    int S = 1;
    if (k_split_req > 0) {
        S = k_split_req;
    } else {
        while (S < 8 && smem_bytes_simt((nspan_all + S - 1) / S, kMaxWarps, 0, 1) > budget) ++S;
        while (S < 8 && S * 2 <= nspan_all && ntiles * S * 2 <= dev.sms) S *= 2;
    }
    if (S > nspan_all) S = nspan_all;
    if (S < 1) S = 1;
    const int spans = (nspan_all + S - 1) / S;
    int warps = spans < kMaxWarps ? spans : kMaxWarps;
    if (warps < 1) warps = 1;
    // persistent clusters: up to the tile count, about two CTAs per SM
    int clusters = (2 * dev.sms) / S;
    if (clusters > ntiles) clusters = ntiles;
    if (clusters < 1) clusters = 1;
    const int tpc = (ntiles + clusters - 1) / clusters;
    p.k_split = S;
    p.units_per_cta = spans;
    p.threads = warps * 32;
    p.ctas = clusters * S;
    p.tiles_per_cluster = tpc;
    p.smem_bytes = smem_bytes_simt(spans, warps, tpc, S);
    return p;
}

cudaError_t launch_gemv_simt(const GemvArgs& a, const GemvPlan& p, cudaStream_t s) {
    SimtKernelArgs k{};
    k.x = a.x;
    k.wq = reinterpret_cast<const uint4*>(a.wq);
    k.scale = a.scale;
    k.zero = a.zero;
    k.y = a.y;
    k.out_f32 = a.out_f32;
    k.N = a.N;
    k.K = a.K;
    k.g = a.g;
    k.ksplit = p.k_split;
    k.spans_per_cta = p.units_per_cta;
    k.tiles_per_cluster = p.tiles_per_cluster;
    k.err = a.err;
    cudaError_t e = cudaFuncSetAttribute(k_gemv_m1, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         p.smem_bytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(p.ctas);
    cfg.blockDim = dim3(p.threads);
    cfg.dynamicSmemBytes = p.smem_bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = p.k_split;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_gemv_m1, k);
}

}  // namespace w4a16
