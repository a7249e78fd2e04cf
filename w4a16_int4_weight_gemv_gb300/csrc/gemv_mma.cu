// 1 <= M <= 16 W4A16 GEMV with warp-level MMA (sm_103a).
//
// Same product as the CUDA-core kernel (local-kimi README, technical-detail
// section: a true GEMV with K contiguous), for a few tokens at once.  With
// M >= 2 the per-weight multiply-adds would exceed the CUDA cores' issue rate
// long before HBM is saturated, so the multiply-accumulate moves to
// mma.sync.m16n8k16 (bf16 in, fp32 accumulate): weights are the 16-row A
// operand, the M tokens (padded to 8 or 16) the B operand.  The dense tile is
// tiny (n = 8 or 16), so warp MMA fed from registers is the right tool; the
// weights never touch shared memory.  (Dequantisation and the K permutation
// are described in mma_core.cuh.)
//
// Memory-level parallelism.  Each warp owns 16-row tiles and keeps kPD
// 128-k blocks of 16-byte loads in flight ahead of the MMAs.  Warps work
// independently; when there are too few tiles to occupy the GPU the K range
// of a tile is split over WPT warps of a CTA (partials added in shared memory
// behind a named barrier, once per tile) and over the CTAs of a thread-block
// cluster (added through distributed shared memory, once per kernel), always
// in a fixed order.  Launches use programmatic dependent launch, as the
// CUDA-core kernel does (see gemv_simt.cu).
#include "common.cuh"
#include "launch.h"
#include "mma_core.cuh"

namespace w4a16 {
namespace {

constexpr int kThreads = 128;

template <int NT>
struct MmaTraits;
template <>
struct MmaTraits<1> {
    static constexpr int kPD = 8;
};
template <>
struct MmaTraits<2> {
    static constexpr int kPD = 4;
};

struct MmaKernelArgs {
    const uint16_t* x;
    const uint4* wq;
    const uint16_t* scale;
    const uint8_t* zero;
    void* y;
    int out_f32;
    int M;
    int N;
    int K;
    int g;
    int wpt;
    int ksplit;
    int blocks_per_cta;
    int tiles_per_group;
    int weights_static;
    uint32_t* err;
};

template <int NT>
int smem_bytes_mma(int M, int bpc, int tg, int wpt, int tpg, int S) {
    constexpr int Mpad = 8 * NT;
    return M * mma_token_stride(bpc)                   // permuted activations
           + bpc * Mpad * 4                           // per-block activation sums
           + (wpt > 1 ? 2 * tg * wpt * 16 * Mpad * 4 : 0)  // in-CTA K-split partials
           + (S > 1 ? tpg * tg * 16 * Mpad * 4 : 0);   // cluster K-split partials
}

template <int NT>
__global__ void __launch_bounds__(kThreads, 4)
k_gemv_mma(const MmaKernelArgs a) {
    constexpr int Mpad = 8 * NT;
    constexpr int kPD = MmaTraits<NT>::kPD;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int W = blockDim.x >> 5;
    const int WPT = a.wpt;
    const int TG = W / WPT;
    const int tg = warp / WPT;
    const int kp = warp - tg * WPT;
    const int Q = a.K >> 5;
    const int nblk_all = a.K >> 7;
    const int S = a.ksplit;
    const int rank = (S > 1) ? static_cast<int>(cluster_rank()) : 0;
    const int cid = blockIdx.x / S;
    const int ncl = gridDim.x / S;
    const int BPC = a.blocks_per_cta;
    const int b0 = rank * BPC;
    const int nb = max(0, min(nblk_all, b0 + BPC) - b0);
    const int ntiles = (a.N + 15) >> 4;
    const int G = a.K / a.g;
    const int tok_stride = mma_token_stride(BPC);

    unsigned char* xs = smem_raw;
    float* xsum = reinterpret_cast<float*>(smem_raw + a.M * tok_stride);
    float* red = xsum + BPC * Mpad;                               // [2][TG][WPT][16][Mpad]
    float* part = red + (WPT > 1 ? 2 * TG * WPT * 16 * Mpad : 0);  // [tpg][TG][16][Mpad]

    const int gid = cid * TG + tg;
    const int NG = ncl * TG;
    const int my_tiles = (ntiles > gid) ? (ntiles - gid + NG - 1) / NG : 0;
    const int my_blocks = (nb > kp) ? (nb - kp + WPT - 1) / WPT : 0;
    const int nsteps = my_tiles * my_blocks;
    const int r = lane >> 2;
    const int c = lane & 3;

    MmaBlockLoad ring[kPD];
    auto issue = [&](int s, MmaBlockLoad& L) {
        const int ti = s / my_blocks;
        const int bi = s - ti * my_blocks;
        mma_block_issue(L, a.wq, a.scale, a.zero, a.N, Q, G, a.g, gid + ti * NG,
                        b0 + kp + bi * WPT, lane);
    };
    grid_dependents_launch();
    if (a.weights_static) {
#pragma unroll
        for (int p = 0; p < kPD; ++p)
            if (p < nsteps) issue(p, ring[p]);
        grid_dependency_wait();
    } else {
        grid_dependency_wait();
#pragma unroll
        for (int p = 0; p < kPD; ++p)
            if (p < nsteps) issue(p, ring[p]);
    }

    stage_x_permuted<NT>(a.x, nullptr, a.M, a.K, b0 << 7, nb, xs, xsum, tok_stride);
    __syncthreads();

    float acc[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[t][i] = 0.f;
    int ti = 0, bi = 0;

    // fragment position i of n-tile t: row r (+8 for i >= 2), token t*8 + 2c + (i & 1)
    auto tile_end = [&]() {
        const int tile = gid + ti * NG;
        if (WPT > 1) {
            float* rb = red + ((ti & 1) * TG + tg) * WPT * 16 * Mpad;
#pragma unroll
            for (int t = 0; t < NT; ++t)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int row = r + ((i >> 1) << 3);
                    const int tok = t * 8 + 2 * c + (i & 1);
                    if (kp > 0) rb[(kp * 16 + row) * Mpad + tok] = acc[t][i];
                }
            named_barrier_sync(1 + tg, WPT * 32);
            if (kp == 0) {
#pragma unroll
                for (int t = 0; t < NT; ++t)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int row = r + ((i >> 1) << 3);
                        const int tok = t * 8 + 2 * c + (i & 1);
                        for (int q = 1; q < WPT; ++q) acc[t][i] += rb[(q * 16 + row) * Mpad + tok];
                    }
            }
        }
        if (kp == 0) {
#pragma unroll
            for (int t = 0; t < NT; ++t)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int row = r + ((i >> 1) << 3);
                    const int tok = t * 8 + 2 * c + (i & 1);
                    if (tok >= a.M) continue;
                    if (S == 1) {
                        const int n = tile * 16 + row;
                        if (n < a.N)
                            store_out(a.y, a.out_f32, static_cast<size_t>(tok) * a.N + n, acc[t][i]);
                    } else {
                        part[((ti * TG + tg) * 16 + row) * Mpad + tok] = acc[t][i];
                    }
                }
        }
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[t][i] = 0.f;
    };

    for (int s0 = 0; s0 < nsteps; s0 += kPD) {
#pragma unroll
        for (int p = 0; p < kPD; ++p) {
            const int s = s0 + p;
            if (s < nsteps) {
                const int lb = kp + bi * WPT;  // block within the slice
                mma_block<NT>(acc, ring[p], xs + lb * 256, xsum + lb * Mpad, tok_stride, a.M,
                              lane);
                if (s + kPD < nsteps) issue(s + kPD, ring[p]);
                if (++bi == my_blocks) {
                    bi = 0;
                    tile_end();
                    ++ti;
                }
            }
        }
    }
    if (my_blocks == 0)
        for (; ti < my_tiles; ++ti) tile_end();

    if (S > 1) {
        cluster_barrier();
        const int per_t = TG * 16 * a.M;
        const int tot = a.tiles_per_group * per_t;
        for (int idx = threadIdx.x; idx < tot; idx += blockDim.x) {
            const int t = idx / per_t;
            int rem = idx - t * per_t;
            const int g2 = rem / (16 * a.M);
            rem -= g2 * 16 * a.M;
            const int tok = rem >> 4;
            const int row = rem & 15;
            const int gid2 = cid * TG + g2;
            const int mt = (ntiles > gid2) ? (ntiles - gid2 + NG - 1) / NG : 0;
            if (t >= mt || (t % S) != rank) continue;
            const float* src = part + ((t * TG + g2) * 16 + row) * Mpad + tok;
            float v = 0.f;
            for (int q = 0; q < S; ++q) v += ld_dsmem_f32(src, static_cast<uint32_t>(q));
            const int n = (gid2 + t * NG) * 16 + row;
            if (n < a.N) store_out(a.y, a.out_f32, static_cast<size_t>(tok) * a.N + n, v);
        }
        cluster_barrier();
    }
}

}  // namespace

GemvPlan plan_gemv_mma(const DeviceInfo& dev, int M, int N, int K, int k_split_req) {
    const int W = kThreads / 32;
    const int nblk = K / 128;
    const int ntiles = (N + 15) / 16;
    const bool two = M > 8;
    const SplitChoice c = choose_split(
        dev, ntiles, nblk, W, 4, k_split_req, [M, two](int upc, int tg, int wpt, int tpg, int S) {
            return two ? smem_bytes_mma<2>(M, upc, tg, wpt, tpg, S)
                       : smem_bytes_mma<1>(M, upc, tg, wpt, tpg, S);
        });
    GemvPlan p{};
    p.kernel_id = 2;
    p.k_split = c.S;
    p.wpt = c.wpt;
    p.units_per_cta = c.units_per_cta;
    p.threads = kThreads;
    p.ctas = c.ctas;
    p.tiles_per_cluster = c.tiles_per_group;
    p.smem_bytes = c.smem_bytes;
    return p;
}

cudaError_t launch_gemv_mma(const GemvArgs& a, const GemvPlan& p, cudaStream_t s) {
    MmaKernelArgs k{};
    k.x = a.x;
    k.wq = reinterpret_cast<const uint4*>(a.wq);
    k.scale = a.scale;
    k.zero = a.zero;
    k.y = a.y;
    k.out_f32 = a.out_f32;
    k.M = a.M;
    k.N = a.N;
    k.K = a.K;
    k.g = a.g;
    k.wpt = p.wpt;
    k.ksplit = p.k_split;
    k.blocks_per_cta = p.units_per_cta;
    k.tiles_per_group = p.tiles_per_cluster;
    k.weights_static = a.weights_static;
    k.err = a.err;
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
    cudaError_t e;
    if (a.M <= 8) {
        e = cudaFuncSetAttribute(k_gemv_mma<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 p.smem_bytes);
        if (e != cudaSuccess) return e;
        return cudaLaunchKernelEx(&cfg, k_gemv_mma<1>, k);
    }
    e = cudaFuncSetAttribute(k_gemv_mma<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             p.smem_bytes);
    if (e != cudaSuccess) return e;
    return cudaLaunchKernelEx(&cfg, k_gemv_mma<2>, k);
}

}  // namespace w4a16
