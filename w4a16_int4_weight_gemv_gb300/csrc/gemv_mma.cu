// 1 <= M <= 16 W4A16 GEMV with warp-level MMA (sm_103a).
//
// Same product as the CUDA-core kernel (local-kimi README, technical-detail
// section: a true GEMV with K contiguous), for a few tokens at once.  With
// M >= 2 the per-weight multiply-adds would exceed the CUDA cores' issue rate
// long before HBM is saturated, so the multiply-accumulate moves to
// mma.sync.m16n8k16 (bf16 in, fp32 accumulate): weights are the 16-row A
// operand, the M tokens (padded to 8 or 16) the B operand.  The dense tile is
// tiny (n = 8 or 16), so warp MMA fed from registers is the right tool.
// (Dequantisation is described in mma_core.cuh.)
//
// Memory path.  Each warp owns 16-row tiles; a step is 512 k of the tile
// (kSB 128-k blocks, 4 KB of packed words).  The step reaches a per-warp ring
// of shared-memory stages as two 2-D tensor copies (16 rows x 128 bytes each,
// 128-byte swizzle) issued by one lane; its scales and zero points follow by
// cp.async; all complete on the stage's mbarrier.  Fragments are read with
// ldmatrix: lane (r, c) gets word c of every 16-byte chunk of rows r and
// r + 8, i.e. 8 consecutive k per chunk, and the swizzle puts the eight rows
// of an ldmatrix phase in eight bank groups.  With that assignment the
// activations need no reordering beyond the pairing inside each 16-byte piece,
// so each token's K slice is one bulk copy, issued before any weight copy so
// that it is not queued behind the weight stream, then paired in place.
//
// Work split.  Warps work independently; when there are too few tiles to
// occupy the GPU the K range of a tile is split over WPT warps of a CTA
// (partials added in shared memory behind a named barrier, once per tile) and
// over the CTAs of a thread-block cluster (added through distributed shared
// memory, once per kernel), always in a fixed order.  Launches use
// programmatic dependent launch.
#include "common.cuh"
#include "launch.h"
#include "mma_core.cuh"

namespace w4a16 {
namespace {

// Warps per CTA: 12 when the tokens fit one 8-column MMA tile and the
// activation slice is small (more warps to cover the MMA and dequant
// latencies), else 8 (shared memory goes to the activations and the rings).
int mma_warps_for(int M, int K) { return (M <= 8 && K <= 8192) ? 12 : 8; }
constexpr int kSB = 4;           // 128-k blocks per step (512 k)
constexpr int kHalfBytes = 2048;  // one tensor box: 16 rows x 128 bytes
constexpr int kStageA = 2 * kHalfBytes;
constexpr int kStageSZ = 256;    // 16 rows x 4 zero points, then 16 rows x 4 scales
constexpr int kSZScales = 64;
constexpr int kMaxStages = 8;
constexpr unsigned kBoxRows = 16;
static_assert(kWeightBoxWords * 4 * kBoxRows == kHalfBytes, "box geometry");

struct MmaKernelArgs {
    const uint16_t* x;
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
    int steps_per_cta;
    int tiles_per_group;
    int stages;
    int weights_static;
    int swiglu_out;  // rows 16t..+7 gate, 16t+8..+15 up: y = bf16 SwiGLU [M][N/2]
    uint32_t* err;
};

// Bytes of the CTA's shared memory before the stage rings: permuted
// activations, block sums, the in-CTA reduction buffer and (K split over a
// cluster) the partials the cluster adds.
__host__ __device__ inline int mma_base_bytes(int M, int NT, int upc, int tg, int wpt, int tpg,
                                              int S) {
    const int Mpad = 8 * NT;
    const int bpc = upc * kSB;
    const int b = M * mma_token_stride(bpc) + bpc * Mpad * 4 +
                  (wpt > 1 ? 2 * tg * wpt * 16 * Mpad * 4 : 0) +
                  (S > 1 ? tpg * S * tg * 16 * Mpad * 4 : 0);
    return (b + 127) & ~127;
}

// Whole dynamic shared memory for NS stages per warp; 1024 bytes of slack
// let the A rings start on the 1024-byte boundary the swizzle needs.
__host__ __device__ inline int mma_smem_bytes(int base, int ns, int warps) {
    return base + 1024 + warps * ns * (kStageA + kStageSZ + 8) + 16;
}

// kFast: g == 128 and K % 512 == 0 -- a step's scales and zero points are
// whole 8- and 4-byte pieces per row, copied with cp.async into the stage.
// Otherwise the consumer loads the two rows' pair for each block itself.
template <int NT, bool kFast, int W>
__global__ void __launch_bounds__(W * 32, 1)
k_gemv_mma(const MmaKernelArgs a, const __grid_constant__ CUtensorMap wmap) {
    constexpr int Mpad = 8 * NT;
    constexpr int kWarps = W;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int WPT = a.wpt;
    const int TG = kWarps / WPT;
    const int tg = warp / WPT;
    const int kp = warp - tg * WPT;
    const int nblk_all = a.K >> 7;
    const int S = a.ksplit;
    const int rank = (S > 1) ? static_cast<int>(cluster_rank()) : 0;
    const int cid = blockIdx.x / S;
    const int ncl = gridDim.x / S;
    const int BPC = a.steps_per_cta * kSB;          // blocks per CTA slice
    const int b0 = rank * BPC;
    const int nb = max(0, min(nblk_all, b0 + BPC) - b0);
    const int nsteps_slice = (nb + kSB - 1) / kSB;
    const int ntiles = (a.N + 15) >> 4;
    const int G = a.K / a.g;
    const int tok_stride = mma_token_stride(BPC);
    const int NS = a.stages;
    const int r = lane >> 2;
    const int c = lane & 3;

    unsigned char* xs = smem_raw;
    float* xsum = reinterpret_cast<float*>(smem_raw + a.M * tok_stride);
    float* red = xsum + BPC * Mpad;                                 // [2][TG][WPT][16][Mpad]
    float* part = red + (WPT > 1 ? 2 * TG * WPT * 16 * Mpad : 0);    // [tpg][S][TG][16][Mpad]
    const int base = mma_base_bytes(a.M, NT, a.steps_per_cta, TG, WPT, a.tiles_per_group, S);
    const uint32_t raw_addr = smem_addr(smem_raw);
    const int a_off = static_cast<int>(((raw_addr + base + 1023u) & ~1023u) - raw_addr);
    unsigned char* ring_a = smem_raw + a_off + warp * NS * kStageA;
    unsigned char* ring_sz = smem_raw + a_off + kWarps * NS * kStageA + warp * NS * kStageSZ;
    uint64_t* bars0 =
        reinterpret_cast<uint64_t*>(smem_raw + a_off + kWarps * NS * (kStageA + kStageSZ));
    uint64_t* bars = bars0 + warp * NS;
    uint64_t* xbar = bars0 + kWarps * NS;

    // tile groups are dealt round-robin over the CTAs (group tg of CTA cid is
    // tg * ncl + cid), so with more CTAs than a full group layout needs the
    // tiles spread over all of them instead of filling the first ones
    const int gid = tg * ncl + cid;
    const int NG = ncl * TG;
    const int my_tiles = (ntiles > gid) ? (ntiles - gid + NG - 1) / NG : 0;
    const int my_steps = (nsteps_slice > kp) ? (nsteps_slice - kp + WPT - 1) / WPT : 0;
    const int nss = my_tiles * my_steps;

    if (threadIdx.x == 0) prefetch_tensor_map(&wmap);
    grid_dependents_launch();
    if (lane == 0) {
        for (int i = 0; i < NS; ++i) mbar_init(bars + i, 1 + (kFast ? 32 : 0));
        if (warp == 0) mbar_init(xbar, 1);
        mbar_init_fence();
    }
    __syncthreads();
    // K split over a cluster: this CTA is running; the matching wait comes
    // before the first store into a peer's shared memory
    if (S > 1) cluster_arrive_relaxed();

    // producer cursor
    int w_tile = gid, w_step = kp, w_stage = 0, w_issued = 0;
    auto issue = [&]() {
        uint64_t* bar = bars + w_stage;
        unsigned char* dst = ring_a + w_stage * kStageA;
        const int blk0 = b0 + w_step * kSB;        // first global block of the step
        const int nbs = min(kSB, b0 + nb - blk0);  // blocks in this step
        const int nh = (nbs + 1) >> 1;             // boxes (two blocks each)
        const int row0 = w_tile * 16;
        if (lane == 0) {
            if (w_issued >= NS) fence_proxy_async_smem();
            mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nh * kHalfBytes));
            tma_load_2d(dst, &wmap, blk0 * 16, row0, bar);
            if (nh > 1) tma_load_2d(dst + kHalfBytes, &wmap, blk0 * 16 + 32, row0, bar);
        }
        if constexpr (kFast) {
            // lanes 0..15 copy row lane's 4 zero points, lanes 16..31 its 4 scales
            unsigned char* sz = ring_sz + w_stage * kStageSZ;
            const int rr = lane & 15;
            if (row0 + rr < a.N) {
                const size_t gi = static_cast<size_t>(row0 + rr) * G + blk0;  // block == group
                if (lane < 16) cp_async_4(sz + rr * 4, a.zero + gi);
                else cp_async_8(sz + kSZScales + rr * 8, a.scale + gi);
            }
            cp_async_arrive_noinc(bar);
        }
        if (++w_stage == NS) w_stage = 0;
        ++w_issued;
        w_step += WPT;
        if (w_step >= nsteps_slice) {
            w_step = kp;
            w_tile += NG;
        }
    };

    // Activations first (they gate every MMA), then the weight rings.  With
    // static weights one stage per warp is already requested while the
    // preceding grid finishes.
    if (a.weights_static && nss > 0) issue();
    grid_dependency_wait();
    if (warp == 0) {
        if (lane == 0) mbar_arrive_expect_tx(xbar, static_cast<uint32_t>(a.M * nb * 256));
        __syncwarp();
        if (lane < a.M && nb > 0)
            bulk_copy_g2s(xs + lane * tok_stride,
                          a.x + static_cast<size_t>(lane) * a.K + (static_cast<size_t>(b0) << 7),
                          static_cast<uint32_t>(nb * 256), xbar);
    }
    __syncthreads();
    // one stage per warp before the pairing pass, the rest after it: issuing
    // whole rings here stalls the warps on memory back-pressure before they
    // reach the pass
    if (w_issued == 0 && nss > 0) issue();

    bool timed_out = !mbar_wait_bounded(xbar, 0);
    pair_x_in_place<NT>(a.M, nb, xs, xsum, tok_stride);
    __syncthreads();
    while (w_issued < NS && w_issued < nss) issue();
    if (S > 1) cluster_wait();  // every peer CTA has started

    float acc[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[t][i] = 0.f;
    int c_tile = gid, c_step = kp, ti = 0, c_stage = 0;
    uint32_t c_phase = 0;

    // fragment position i of n-tile t: row r (+8 for i >= 2), token t*8 + 2c + (i & 1)
    auto tile_end = [&]() {
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
        if (kp == 0 && S == 1 && a.swiglu_out) {
            // rows r and r + 8 of the tile are gate and up row 8 tile + r
            const size_t nh = static_cast<size_t>(a.N >> 1);
            uint16_t* y = static_cast<uint16_t*>(a.y);
#pragma unroll
            for (int t = 0; t < NT; ++t)
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int tok = t * 8 + 2 * c + i;
                    if (tok < a.M)
                        y[tok * nh + static_cast<size_t>(c_tile) * 8 + r] =
                            swiglu_of_sums(acc[t][i], acc[t][i + 2]);
                }
        } else if (kp == 0) {
#pragma unroll
            for (int t = 0; t < NT; ++t)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int row = r + ((i >> 1) << 3);
                    const int tok = t * 8 + 2 * c + (i & 1);
                    if (tok >= a.M) continue;
                    if (S == 1) {
                        const int n = c_tile * 16 + row;
                        if (n < a.N)
                            store_out(a.y, a.out_f32, static_cast<size_t>(tok) * a.N + n, acc[t][i]);
                    } else {
                        // into the owner's shared memory (CTA ti % S of the cluster)
                        st_dsmem_f32(part + (((ti * S + rank) * TG + tg) * 16 + row) * Mpad + tok,
                                     static_cast<uint32_t>(ti % S), acc[t][i]);
                    }
                }
        }
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[t][i] = 0.f;
    };

    // ldmatrix addressing: lane l supplies row (l & 7) + 8 * ((l >> 3) & 1) of
    // chunk (l >> 4) (+ 2 for the second load) of the block's four chunks.
    const int lrow = (lane & 7) + (((lane >> 3) & 1) << 3);
    const uint32_t lbase = static_cast<uint32_t>(lrow * 128);
    const int lsw = lane & 7;  // swizzle term: row % 8
    const int lch = lane >> 4;

#pragma unroll 1
    for (int ss = 0; ss < nss; ++ss) {
        if (!mbar_wait_bounded(bars + c_stage, c_phase)) timed_out = true;
        const uint32_t stg = smem_addr(ring_a + c_stage * kStageA);
        const unsigned char* sz = ring_sz + c_stage * kStageSZ;
        const int lb0 = c_step * kSB;  // first block of the step within the slice
        const int nbs = min(kSB, nb - lb0);
        const int n0 = c_tile * 16 + r;
#pragma unroll
        for (int bb = 0; bb < kSB; ++bb) {
            if (bb < nbs) {
                const uint32_t hb = stg + (bb >> 1) * kHalfBytes + lbase;
                const int cb = (bb & 1) * 4 + lch;
                uint32_t q0[4], q1[4];
                ldmatrix_x4(q0, hb + (static_cast<uint32_t>(cb ^ lsw) << 4));
                ldmatrix_x4(q1, hb + (static_cast<uint32_t>((cb + 2) ^ lsw) << 4));
                MmaBlockLoad L;
                L.w0 = make_uint4(q0[0], q0[2], q1[0], q1[2]);
                L.w1 = make_uint4(q0[1], q0[3], q1[1], q1[3]);
                if constexpr (kFast) {
                    L.sz0 = *reinterpret_cast<const uint16_t*>(sz + kSZScales + r * 8 + bb * 2) |
                            (static_cast<uint32_t>(sz[r * 4 + bb]) << 16);
                    L.sz1 =
                        *reinterpret_cast<const uint16_t*>(sz + kSZScales + (r + 8) * 8 + bb * 2) |
                        (static_cast<uint32_t>(sz[(r + 8) * 4 + bb]) << 16);
                } else {
                    const int grp = ((b0 + lb0 + bb) << 7) / a.g;
                    L.sz0 = 0u;
                    L.sz1 = 0u;
                    if (n0 < a.N) {
                        const size_t gi = static_cast<size_t>(n0) * G + grp;
                        L.sz0 = ldg_nc_u16(a.scale + gi) | (ldg_nc_u8(a.zero + gi) << 16);
                    }
                    if (n0 + 8 < a.N) {
                        const size_t gi = static_cast<size_t>(n0 + 8) * G + grp;
                        L.sz1 = ldg_nc_u16(a.scale + gi) | (ldg_nc_u8(a.zero + gi) << 16);
                    }
                }
                mma_block<NT>(acc, L, xs + (lb0 + bb) * 256, xsum + (lb0 + bb) * Mpad, tok_stride,
                              a.M, lane);
            }
        }
        __syncwarp();  // every lane is done with stage c_stage
        if (w_issued < nss) issue();
        if (++c_stage == NS) {
            c_stage = 0;
            c_phase ^= 1u;
        }
        c_step += WPT;
        if (c_step >= nsteps_slice) {
            tile_end();
            c_step = kp;
            c_tile += NG;
            ++ti;
        }
    }
    if (timed_out && lane == 0) raise_device_error(a.err, W4A16_DEVERR_TIMEOUT);
    if (my_steps == 0)
        for (; ti < my_tiles; ++ti) tile_end();

    // cluster K split: every rank stored its partials of tile t into the
    // shared memory of the owner, rank t % S; after one cluster barrier the
    // owner adds them in rank order (deterministic) and stores y
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
            const int gid2 = g2 * ncl + cid;
            const int mt = (ntiles > gid2) ? (ntiles - gid2 + NG - 1) / NG : 0;
            if (t >= mt || (t % S) != rank) continue;
            if (a.swiglu_out && row >= 8) continue;  // the up row goes with its gate row
            float v = 0.f, u = 0.f;
            for (int q = 0; q < S; ++q) v += part[(((t * S + q) * TG + g2) * 16 + row) * Mpad + tok];
            const int n = (gid2 + t * NG) * 16 + row;
            if (a.swiglu_out) {
                for (int q = 0; q < S; ++q)
                    u += part[(((t * S + q) * TG + g2) * 16 + row + 8) * Mpad + tok];
                static_cast<uint16_t*>(a.y)[static_cast<size_t>(tok) * (a.N >> 1) +
                                            static_cast<size_t>(gid2 + t * NG) * 8 + row] =
                    swiglu_of_sums(v, u);
                continue;
            }
            if (n < a.N) store_out(a.y, a.out_f32, static_cast<size_t>(tok) * a.N + n, v);
        }
    }
}

using MmaKernel = void (*)(MmaKernelArgs, CUtensorMap);

MmaKernel pick_mma_kernel(int M, int K, int g, int warps) {
    const bool fast = (g == 128) && (K % 512 == 0);
    if (warps == 12)
        return (M <= 8) ? (fast ? k_gemv_mma<1, true, 12> : k_gemv_mma<1, false, 12>)
                        : (fast ? k_gemv_mma<2, true, 12> : k_gemv_mma<2, false, 12>);
    return (M <= 8) ? (fast ? k_gemv_mma<1, true, 8> : k_gemv_mma<1, false, 8>)
                    : (fast ? k_gemv_mma<2, true, 8> : k_gemv_mma<2, false, 8>);
}

}  // namespace

GemvPlan plan_gemv_mma(const DeviceInfo& dev, int M, int N, int K, int g, int k_split_req) {
    const int nblk = K / 128;
    const int units_all = (nblk + kSB - 1) / kSB;
    const int ntiles = (N + 15) / 16;
    const int NT = (M <= 8) ? 1 : 2;
    const int W = mma_warps_for(M, K);
    const void* kern = reinterpret_cast<const void*>(pick_mma_kernel(M, K, g, W));
    // the launch fills the CTA's shared memory with stages, so co-residency of
    // clusters is queried at the full budget, not at the two-stage minimum
    const int budget = dev.max_smem_optin;
    const SplitChoice c = choose_split(
        dev, ntiles, units_all, W, 1, k_split_req, 0,
        [M, NT, W](int upc, int tg, int wpt, int tpg, int S) {
            return mma_smem_bytes(mma_base_bytes(M, NT, upc, tg, wpt, tpg, S), 2, W);
        },
        [kern, budget, W](int S, int) { return max_active_clusters(kern, W * 32, budget, S); });
    GemvPlan p{};
    p.kernel_id = 2;
    p.k_split = c.S;
    p.wpt = c.wpt;
    p.units_per_cta = c.units_per_cta;
    p.threads = W * 32;
    p.ctas = c.ctas;
    p.tiles_per_cluster = c.tiles_per_group;
    if (c.ctas > 0) {
        const int base = mma_base_bytes(M, NT, c.units_per_cta, W / c.wpt, c.wpt,
                                        c.tiles_per_group, c.S);
        const int max_steps = c.tiles_per_group * ((c.units_per_cta + c.wpt - 1) / c.wpt);
        int ns = 2;
        while (ns < kMaxStages && ns < max_steps && mma_smem_bytes(base, ns + 1, W) <= budget) ++ns;
        p.stages = ns;
        p.smem_bytes = mma_smem_bytes(base, ns, W);
    }
    return p;
}

cudaError_t launch_gemv_mma(const GemvArgs& a, const GemvPlan& p, cudaStream_t s) {
    MmaKernelArgs k{};
    k.x = a.x;
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
    k.steps_per_cta = p.units_per_cta;
    k.tiles_per_group = p.tiles_per_cluster;
    k.stages = p.stages;
    k.weights_static = a.weights_static;
    k.swiglu_out = a.swiglu_out;
    k.err = a.err;
    CUtensorMap wmap;
    if (!encode_weight_map(&wmap, a.wq, a.N, a.K, kBoxRows)) return cudaErrorInvalidValue;
    MmaKernel kern = pick_mma_kernel(a.M, a.K, a.g, p.threads / 32);
    cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), p.smem_bytes);
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
    return cudaLaunchKernelEx(&cfg, kern, k, wmap);
}

}  // namespace w4a16
