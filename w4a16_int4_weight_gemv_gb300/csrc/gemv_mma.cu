// 1 <= M <= 16 W4A16 GEMV with warp-level MMA (sm_103a).
//
// Same product as the CUDA-core kernel (local-kimi README, technical-detail
// section: a true GEMV with K contiguous), for a few tokens at once.  With
// M >= 2 the per-weight multiply-adds would exceed the CUDA cores' issue rate
// long before HBM is saturated, so the multiply-accumulate moves to
// mma.sync.m16n8k16 (bf16 in, fp32 accumulate): weights are the 16-row A
// operand, the M tokens (padded to 8 or 16) the B operand.  The dense tile is
// tiny (n = 8 or 16), so warp MMA fed from registers is the right tool; the
// weights never touch shared memory.
//
// Work split.  A CTA owns a K slice (all of K unless split across a cluster)
// and loops over 16-row tiles; its warps take interleaved 128-k blocks of the
// slice and their partials are summed through shared memory; cluster K-splits
// are summed through distributed shared memory in rank order.
#include "common.cuh"
#include "launch.h"
#include "mma_core.cuh"

namespace w4a16 {
namespace {

constexpr int kPD = 4;  // 128-k blocks of loads in flight per warp
constexpr int kMaxWarps = 8;

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
    int ksplit;
    int blocks_per_cta;
    int tiles_per_cluster;
    uint32_t* err;
};

template <int NT>
__global__ void __launch_bounds__(kMaxWarps * 32)
k_gemv_mma(const MmaKernelArgs a) {
    constexpr int Mpad = 8 * NT;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int W = blockDim.x >> 5;
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
    const int tok_stride = MmaLayout<NT>::token_stride(BPC);

    unsigned char* xs = smem_raw;
    float* xsum = reinterpret_cast<float*>(smem_raw + Mpad * tok_stride);
    float* red = xsum + BPC * Mpad;
    float* part = red + W * 16 * Mpad;

    const int my_tiles = (ntiles > cid) ? (ntiles - cid + ncl - 1) / ncl : 0;
    const int my_blocks = (nb > warp) ? (nb - warp + W - 1) / W : 0;
    const int nsteps = my_tiles * my_blocks;
    const int r = lane >> 2;
    const int c = lane & 3;

    uint4 wa[kPD], wb[kPD];
    uint32_t sa[kPD], sb[kPD];
    auto issue = [&](int s, uint4& w0, uint4& w1, uint32_t& z0, uint32_t& z1) {
        const int ti = s / my_blocks;
        const int bi = s - ti * my_blocks;
        const int tile = cid + ti * ncl;
        const int blk = b0 + warp + bi * W;  // global 128-k block
        const int grp = (blk << 7) / a.g;
        const int n0 = tile * 16 + r;
        const int n1 = n0 + 8;
        const int chunk = blk * 4 + c;
        if (n0 < a.N) {
            w0 = ldg_stream_u4(a.wq + static_cast<size_t>(n0) * Q + chunk);
            const size_t gi = static_cast<size_t>(n0) * G + grp;
            z0 = ldg_nc_u16(a.scale + gi) | (ldg_nc_u8(a.zero + gi) << 16);
        } else {
            w0 = make_uint4(0u, 0u, 0u, 0u);
            z0 = 0u;
        }
        if (n1 < a.N) {
            w1 = ldg_stream_u4(a.wq + static_cast<size_t>(n1) * Q + chunk);
            const size_t gi = static_cast<size_t>(n1) * G + grp;
            z1 = ldg_nc_u16(a.scale + gi) | (ldg_nc_u8(a.zero + gi) << 16);
        } else {
            w1 = make_uint4(0u, 0u, 0u, 0u);
            z1 = 0u;
        }
    };
#pragma unroll
    for (int p = 0; p < kPD; ++p)
        if (p < nsteps) issue(p, wa[p], wb[p], sa[p], sb[p]);

    stage_x_permuted<NT>(a.x, nullptr, a.M, a.K, b0 << 7, nb, xs, xsum, tok_stride);
    __syncthreads();

    float acc[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[t][i] = 0.f;
    int ti = 0, bi = 0;

    auto tile_end = [&]() {
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const int tok = t * 8 + 2 * c;
            red[(warp * 16 + r) * Mpad + tok] = acc[t][0];
            red[(warp * 16 + r) * Mpad + tok + 1] = acc[t][1];
            red[(warp * 16 + r + 8) * Mpad + tok] = acc[t][2];
            red[(warp * 16 + r + 8) * Mpad + tok + 1] = acc[t][3];
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[t][i] = 0.f;
        }
        __syncthreads();
        const int tile = cid + ti * ncl;
        for (int idx = threadIdx.x; idx < 16 * a.M; idx += blockDim.x) {
            const int tok = idx >> 4;
            const int row = idx & 15;
            float v = 0.f;
            for (int w = 0; w < W; ++w) v += red[(w * 16 + row) * Mpad + tok];
            if (S == 1) {
                const int n = tile * 16 + row;
                if (n < a.N) store_out(a.y, a.out_f32, static_cast<size_t>(tok) * a.N + n, v);
            } else {
                part[(ti * 16 + row) * Mpad + tok] = v;
            }
        }
        __syncthreads();
    };

    for (int s0 = 0; s0 < nsteps; s0 += kPD) {
#pragma unroll
        for (int p = 0; p < kPD; ++p) {
            const int s = s0 + p;
            if (s < nsteps) {
                const int lb = warp + bi * W;  // block within the slice
                mma_block<NT>(acc, wa[p], wb[p], sa[p], sb[p], xs + lb * 256, xsum + lb * Mpad,
                              tok_stride, lane);
                if (s + kPD < nsteps) issue(s + kPD, wa[p], wb[p], sa[p], sb[p]);
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
        for (int idx = threadIdx.x; idx < my_tiles * 16 * a.M; idx += blockDim.x) {
            const int t = idx / (16 * a.M);
            if (t % S != rank) continue;
            const int rem = idx - t * 16 * a.M;
            const int tok = rem >> 4;
            const int row = rem & 15;
            const float* src = part + (t * 16 + row) * Mpad + tok;
            float v = 0.f;
            for (int q = 0; q < S; ++q) v += ld_dsmem_f32(src, static_cast<uint32_t>(q));
            const int n = (cid + t * ncl) * 16 + row;
            if (n < a.N) store_out(a.y, a.out_f32, static_cast<size_t>(tok) * a.N + n, v);
        }
        cluster_barrier();
    }
}

}  // namespace

GemvPlan plan_gemv_mma(const DeviceInfo& dev, int M, int N, int K, int k_split_req) {
    GemvPlan p{};
    p.kernel_id = 2;
    const int NT = (M <= 8) ? 1 : 2;
    const int nblk = K / 128;
    const int ntiles = (N + 15) / 16;
    const int budget = dev.max_smem_optin - 1024;
    auto bytes = [&](int bpc, int warps, int tpc, int S) {
        return NT == 1 ? MmaLayout<1>::bytes(bpc, warps, tpc, S)
                       : MmaLayout<2>::bytes(bpc, warps, tpc, S);
    };
    int S = 1;
    if (k_split_req > 0) {
        S = k_split_req;
    } else {
        // keep the activation slice to about 100 KB so two CTAs fit on an SM
        while (S < 8 && bytes((nblk + S - 1) / S, kMaxWarps, 0, 1) > 100 * 1024) ++S;
        while (S < 8 && S * 2 <= nblk && ntiles * S * 2 <= dev.sms) S *= 2;
    }
    if (S > nblk) S = nblk;
    if (S < 1) S = 1;
    const int bpc = (nblk + S - 1) / S;
    int warps = bpc < kMaxWarps ? bpc : kMaxWarps;
    if (warps < 1) warps = 1;
    int clusters = (2 * dev.sms) / S;
    if (clusters > ntiles) clusters = ntiles;
    if (clusters < 1) clusters = 1;
    int tpc = (ntiles + clusters - 1) / clusters;
    // the split-K partial buffer must fit too; otherwise use more clusters
    while (S > 1 && bytes(bpc, warps, tpc, S) > budget && clusters < ntiles) {
        clusters *= 2;
        if (clusters > ntiles) clusters = ntiles;
        tpc = (ntiles + clusters - 1) / clusters;
    }
    p.k_split = S;
    p.units_per_cta = bpc;
    p.threads = warps * 32;
    p.ctas = clusters * S;
    p.tiles_per_cluster = tpc;
    p.smem_bytes = bytes(bpc, warps, tpc, S);
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
    k.ksplit = p.k_split;
    k.blocks_per_cta = p.units_per_cta;
    k.tiles_per_cluster = p.tiles_per_cluster;
    k.err = a.err;
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
