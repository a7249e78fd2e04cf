// M = 1 or 2 W4A16 GEMV on CUDA cores (sm_103a).
//
// The decode-time product of the local-kimi README, technical-detail section:
// one (or two) activation rows against a group-quantised INT4 matrix, done as
// a true GEMV -- every lane walks the reduction axis K of its rows with
// 128-bit coalesced loads and keeps one fp32 accumulator per output.
//
// Arithmetic.  For one 16-byte chunk (32 consecutive k of one row, all in one
// quantisation group because g % 32 == 0) the kernel forms
//     acc = sum_k code_k * x_k
// with every product exact in fp32, then applies the group's zero point and
// scale once:  partial += s * (acc - z * sum_k x_k),  which equals
// sum_k (code_k - z) * s * x_k.
//
// Nibble -> float without conversion instructions: the bit pattern
// (word & (0xF << p)) read as a binary32 is code * 2^(p - 149) (a subnormal,
// or for p = 20 and code >= 8 one of the smallest normals, whose value is
// still the integer pattern times 2^-149).  Multiplying it by x * 2^(85 - p)
// gives code * x * 2^-64 exactly, so a weight costs one LOP3 and one FFMA per
// token, plus one shift per word that brings the top two nibbles down by 8
// bits.  The integer ALU pipe issues LOP3 at half the FFMA rate, so this mask
// is the per-weight cost that bounds the kernel; everything else is kept off
// that pipe or amortised over a span of rows.  The 2^(85 - p) factors are
// folded into the staged activations and the 2^64 is restored on the output.
// The FMAs keep subnormal operands (the library is built without
// flush-to-zero); the exact product of a bf16 x and a 4-bit code stays normal
// unless |code * x| < 2^-62.  Inputs need |x| < 2^40 so x * 2^85 stays finite.
//
// Work split.  One persistent CTA of 16 warps per SM.  Warps own tiles of kTR
// rows and stream their packed words through a ring of kSP spans x kTR rows of
// 16-byte loads per lane (a span = 32 consecutive chunks = 512 contiguous
// bytes of a row, one chunk per lane).  When rows are few, the K range of a
// tile is split over WPT warps of the CTA (partials added in shared memory
// behind a named barrier, once per tile) and over the CTAs of a thread-block
// cluster (added through distributed shared memory, once per kernel), always
// in a fixed order, so results are deterministic.
//
// Activations.  The CTA's K slice of x is read once with 16-byte loads,
// scaled per nibble position into fp32 x' and stored in shared memory with an
// XOR swizzle (the 8 lanes of a quarter-warp read 8 distinct bank groups);
// per-chunk sums are reduced with warp shuffles in the same pass.
//
// Launch.  Kernels are launched with programmatic stream serialisation: the
// next launch on the stream may start its CTAs as this grid drains, and every
// CTA waits (griddepcontrol.wait) for the preceding grid before it reads or
// writes global memory -- or, when the caller declares the weights constant,
// only before it reads x or writes y, so its first weight loads overlap the
// previous kernel.
#include "common.cuh"
#include "launch.h"

namespace w4a16 {
namespace {

constexpr int kTR = 4;  // rows per warp tile
constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;

template <int MT>
struct SimtTraits;
template <>
struct SimtTraits<1> {
    static constexpr int kSP = 4;  // spans of loads in flight per warp
};
template <>
struct SimtTraits<2> {
    static constexpr int kSP = 3;
};

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
    int wpt;              // warps per tile (K split inside the CTA)
    int ksplit;           // CTAs per cluster (K split across the cluster)
    int spans_per_cta;    // 32-chunk spans in one CTA's K slice
    int tiles_per_group;  // upper bound of tiles any tile group processes
    int weights_static;   // weights may be read before the preceding grid completes
    uint32_t* err;
};

// x'[k] = x[k] * 2^(85 - p), p the bit offset the code of k sits at after the
// masking: nibbles 0..5 at 4*i, nibbles 6 and 7 (shifted down by 8) at 16, 20.
__device__ __forceinline__ float position_factor(int i) {
    const int p = (i < 6) ? 4 * i : 4 * i - 8;
    return exp2i(85 - p);
}

// acc += sum over the 16 codes of two words of code * x'
__device__ __forceinline__ void dot_words(float& a0, float& a1, uint32_t v0, uint32_t v1,
                                          const float* xr) {
    const uint32_t vs[2] = {v0, v1};
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const uint32_t v = vs[j];
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
}

__device__ __forceinline__ void store_y(void* y, int out_f32, size_t i, float v) {
    v *= exp2i(64);
    if (out_f32) static_cast<float*>(y)[i] = v;
    else static_cast<uint16_t*>(y)[i] = f32_to_bf16_rn(v);
}

template <int MT>
__global__ void __launch_bounds__(kThreads, 1)
k_gemv_simt(const SimtKernelArgs a) {
    constexpr int kSP = SimtTraits<MT>::kSP;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int WPT = a.wpt;
    const int TG = kWarps / WPT;     // tile groups per CTA
    const int tg = warp / WPT;
    const int kp = warp - tg * WPT;  // this warp's part of the K slice
    const int Q = a.K >> 5;          // 16-byte chunks per row
    const int nspan_all = (Q + 31) >> 5;
    const int S = a.ksplit;
    const int rank = (S > 1) ? static_cast<int>(cluster_rank()) : 0;
    const int cid = blockIdx.x / S;
    const int ncl = gridDim.x / S;
    const int SP = a.spans_per_cta;
    const int span0 = rank * SP;
    const int nspan = max(0, min(nspan_all, span0 + SP) - span0);
    const int ntiles = (a.N + kTR - 1) / kTR;
    const int G = a.K / a.g;
    const int cpg = a.g >> 5;  // chunks per quantisation group

    float* xs = reinterpret_cast<float*>(smem_raw);  // [MT][SP * 1024] swizzled x'
    float* xsum = xs + MT * SP * 1024;              // [MT][SP * 32] chunk sums * 2^-64
    float* red = xsum + MT * SP * 32;               // [2][TG][WPT][kTR * MT]
    float* part = red + 2 * TG * WPT * kTR * MT;    // [tpg][TG][kTR * MT] (S > 1)

    const int gid = cid * TG + tg;
    const int NG = ncl * TG;
    const int my_tiles = (ntiles > gid) ? (ntiles - gid + NG - 1) / NG : 0;
    const int my_spans = (nspan > kp) ? (nspan - kp + WPT - 1) / WPT : 0;
    const int nss = my_tiles * my_spans;  // (tile, span) steps of this warp

    grid_dependents_launch();

    // load cursor: tile and span (within the slice) of the next step to issue
    int l_tile = gid, l_span = kp;
    uint4 ring[kSP][kTR];
    uint32_t szr[kSP][kTR];  // scale bits | zero << 16

    auto issue = [&](uint4 (&wv)[kTR], uint32_t (&szv)[kTR]) {
        const int c = ((span0 + l_span) << 5) + lane;  // global chunk
        const bool cok = c < Q;
        const int grp = c / cpg;
        const uint4* wp = a.wq + static_cast<size_t>(l_tile) * kTR * Q + c;
        const size_t gb = static_cast<size_t>(l_tile) * kTR * G + grp;
#pragma unroll
        for (int r = 0; r < kTR; ++r) {
            const int n = l_tile * kTR + r;
            if (cok && n < a.N) {
                wv[r] = ldg_stream_u4(wp + static_cast<size_t>(r) * Q);
                szv[r] = ldg_nc_u16(a.scale + gb + r * G) | (ldg_nc_u8(a.zero + gb + r * G) << 16);
            } else {
                wv[r] = make_uint4(0u, 0u, 0u, 0u);
                szv[r] = 0u;
            }
        }
        l_span += WPT;
        if (l_span >= nspan) {
            l_span = kp;
            l_tile += NG;
        }
    };

    if (a.weights_static) {
#pragma unroll
        for (int j = 0; j < kSP; ++j)
            if (j < nss) issue(ring[j], szr[j]);
        grid_dependency_wait();
    } else {
        grid_dependency_wait();
#pragma unroll
        for (int j = 0; j < kSP; ++j)
            if (j < nss) issue(ring[j], szr[j]);
    }

    // stage x' and the chunk sums of this CTA's K slice (one pass)
    {
        const int kbeg = span0 << 10;
        const int kend = min(a.K, (span0 + nspan) << 10);
        const int pieces = nspan << 7;  // 8 consecutive k per piece, 4 pieces per chunk
        for (int m = 0; m < MT; ++m) {
            for (int base = 0; base < pieces; base += blockDim.x) {
                const int i = base + threadIdx.x;
                const int k0 = i << 3;   // local k
                const int cl = k0 >> 5;  // local chunk
                const int q0 = (k0 >> 2) & 7;
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                if (i < pieces && kbeg + k0 < kend)
                    v = __ldg(reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(m) * a.K +
                                                             kbeg + k0));
                const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
                float f[8];
                float sum = 0.f;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float lo = bf16_to_f32(wv[e] & 0xFFFFu);
                    const float hi = bf16_to_f32(wv[e] >> 16);
                    sum += lo + hi;
                    f[2 * e] = lo * position_factor(2 * e);
                    f[2 * e + 1] = hi * position_factor(2 * e + 1);
                }
                sum += __shfl_xor_sync(0xffffffffu, sum, 1);
                sum += __shfl_xor_sync(0xffffffffu, sum, 2);
                if (i < pieces) {
                    float* base_p = xs + m * SP * 1024 + cl * 32;
                    *reinterpret_cast<float4*>(base_p + ((q0 ^ (cl & 7)) << 2)) =
                        make_float4(f[0], f[1], f[2], f[3]);
                    *reinterpret_cast<float4*>(base_p + (((q0 + 1) ^ (cl & 7)) << 2)) =
                        make_float4(f[4], f[5], f[6], f[7]);
                    if ((i & 3) == 0) xsum[m * SP * 32 + cl] = sum * exp2i(-64);
                }
            }
        }
    }
    __syncthreads();

    float acc[kTR][MT];
#pragma unroll
    for (int r = 0; r < kTR; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[r][m] = 0.f;
    int c_tile = gid, c_span = kp, ti = 0;

    // lane l < kTR * MT owns output (row l / MT, token l % MT) of the tile
    auto tile_end = [&]() {
        float mine = 0.f;
#pragma unroll
        for (int r = 0; r < kTR; ++r)
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                float s = acc[r][m];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
                if (lane == r * MT + m) mine = s;
                acc[r][m] = 0.f;
            }
        const int orow = lane / MT;
        const int otok = lane - orow * MT;
        if (WPT > 1) {
            float* rb = red + ((ti & 1) * TG + tg) * WPT * kTR * MT;
            if (lane < kTR * MT) rb[kp * kTR * MT + lane] = mine;
            named_barrier_sync(1 + tg, WPT * 32);
            if (kp == 0 && lane < kTR * MT) {
                mine = 0.f;
                for (int q = 0; q < WPT; ++q) mine += rb[q * kTR * MT + lane];
            }
        }
        if (kp == 0 && lane < kTR * MT) {
            if (S == 1) {
                const int n = c_tile * kTR + orow;
                if (n < a.N) store_y(a.y, a.out_f32, static_cast<size_t>(otok) * a.N + n, mine);
            } else {
                part[(ti * TG + tg) * kTR * MT + lane] = mine;
            }
        }
    };

    for (int ss0 = 0; ss0 < nss; ss0 += kSP) {
#pragma unroll
        for (int j = 0; j < kSP; ++j) {
            const int ss = ss0 + j;
            if (ss < nss) {
                const int cl = (c_span << 5) + lane;  // chunk within the slice
                if (((span0 << 5) + cl) < Q) {
                    float d0[kTR][MT], d1[kTR][MT];
#pragma unroll
                    for (int r = 0; r < kTR; ++r)
#pragma unroll
                        for (int m = 0; m < MT; ++m) d0[r][m] = d1[r][m] = 0.f;
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        const float* xb = xs + m * SP * 1024 + cl * 32;
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            float xr[16];
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const float4 t = *reinterpret_cast<const float4*>(
                                    xb + (((4 * h + q) ^ (cl & 7)) << 2));
                                xr[4 * q + 0] = t.x;
                                xr[4 * q + 1] = t.y;
                                xr[4 * q + 2] = t.z;
                                xr[4 * q + 3] = t.w;
                            }
#pragma unroll
                            for (int r = 0; r < kTR; ++r) {
                                const uint4 w = ring[j][r];
                                if (h == 0) dot_words(d0[r][m], d1[r][m], w.x, w.y, xr);
                                else dot_words(d0[r][m], d1[r][m], w.z, w.w, xr);
                            }
                        }
                    }
#pragma unroll
                    for (int r = 0; r < kTR; ++r) {
                        const float sc = __uint_as_float(szr[j][r] << 16);
                        const float zf =
                            __uint_as_float(__byte_perm(szr[j][r], 0x4B000000u, 0x7542)) -
                            8388608.f;
#pragma unroll
                        for (int m = 0; m < MT; ++m) {
                            const float xc = xsum[m * SP * 32 + cl];
                            acc[r][m] = fmaf(sc, fmaf(-zf, xc, d0[r][m] + d1[r][m]), acc[r][m]);
                        }
                    }
                }
                if (ss + kSP < nss) issue(ring[j], szr[j]);
                c_span += WPT;
                if (c_span >= nspan) {
                    tile_end();
                    c_span = kp;
                    c_tile += NG;
                    ++ti;
                }
            }
        }
    }
    // a warp with no span in the slice still joins its group's reductions
    if (my_spans == 0)
        for (; ti < my_tiles; ++ti) {
            tile_end();
            c_tile += NG;
        }

    // cluster K split: add the ranks' partials in rank order through DSMEM
    if (S > 1) {
        cluster_barrier();
        const int per_t = TG * kTR * MT;
        const int tot = a.tiles_per_group * per_t;
        for (int idx = threadIdx.x; idx < tot; idx += blockDim.x) {
            const int t = idx / per_t;
            const int rem = idx - t * per_t;
            const int g2 = rem / (kTR * MT);
            const int l = rem - g2 * kTR * MT;
            const int gid2 = cid * TG + g2;
            const int mt = (ntiles > gid2) ? (ntiles - gid2 + NG - 1) / NG : 0;
            if (t >= mt || (t % S) != rank) continue;
            float v = 0.f;
            for (int q = 0; q < S; ++q) v += ld_dsmem_f32(part + idx, static_cast<uint32_t>(q));
            const int orow = l / MT;
            const int n = (gid2 + t * NG) * kTR + orow;
            if (n < a.N) store_y(a.y, a.out_f32, static_cast<size_t>(l - orow * MT) * a.N + n, v);
        }
        cluster_barrier();
    }
}

template <int MT>
int smem_bytes_simt(int spans, int tg, int wpt, int tpg, int S) {
    return MT * spans * (4096 + 128) + 2 * tg * wpt * kTR * MT * 4 +
           (S > 1 ? tpg * tg * kTR * MT * 4 : 0);
}

}  // namespace

GemvPlan plan_gemv_simt(const DeviceInfo& dev, int M, int N, int K, int k_split_req) {
    const int nspan_all = (K / 32 + 31) / 32;
    const int ntiles = (N + kTR - 1) / kTR;
    const SplitChoice c = choose_split(dev, ntiles, nspan_all, kWarps, 1, k_split_req,
                                       [M](int upc, int tg, int wpt, int tpg, int S) {
                                           return M == 1 ? smem_bytes_simt<1>(upc, tg, wpt, tpg, S)
                                                         : smem_bytes_simt<2>(upc, tg, wpt, tpg, S);
                                       });
    GemvPlan p{};
    p.kernel_id = 1;
    p.k_split = c.S;
    p.wpt = c.wpt;
    p.units_per_cta = c.units_per_cta;
    p.threads = kThreads;
    p.ctas = c.ctas;
    p.tiles_per_cluster = c.tiles_per_group;
    p.smem_bytes = c.smem_bytes;
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
    k.wpt = p.wpt;
    k.ksplit = p.k_split;
    k.spans_per_cta = p.units_per_cta;
    k.tiles_per_group = p.tiles_per_cluster;
    k.weights_static = a.weights_static;
    k.err = a.err;
    auto kern = (a.M == 1) ? k_gemv_simt<1> : k_gemv_simt<2>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         p.smem_bytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(p.ctas);
    cfg.blockDim = dim3(p.threads);
    cfg.dynamicSmemBytes = p.smem_bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int na = 0;
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (p.k_split > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = p.k_split;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, k);
}

}  // namespace w4a16
