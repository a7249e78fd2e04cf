// 1 <= M <= 16 W4A16 GEMV on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// Same product as the other GEMV kernels (local-kimi README, technical-detail
// section: a true GEMV with K contiguous).  The legacy warp MMA (mma.sync)
// and the CUDA cores both spend their issue slots on the multiply-adds as
// well as on unpacking the 4-bit codes, and top out below the rate at which
// HBM delivers weights.  Here the multiply-add leaves the SM's issue ports
// entirely: the CUDA cores only unpack codes into bf16 and write them to
// tensor memory, and one thread issues tcgen05.mma over them.
//
// Tile: 128 weight rows (one per TMEM lane) x the CTA's K slice.  A 128-k
// block of the tile is the MMA's A operand: eight 128 x 16 bf16 steps in 64
// TMEM columns, each value 128 + code (the LOP3 trick of mma_core.cuh: a
// word's nibbles i and i + 4 become one column's pair).  B is the token
// activations in shared memory (K-major, 8 or 16 tokens, values paired the
// same way), D is 16 fp32 columns.  D of a block is the exact fp32 sum
//     C_m = sum_k (128 + q_k) x_mk      (bf16 products are exact in fp32)
// and is folded into the row's accumulator as s * (C_m - (128 + z) * sum_k x_mk)
// because a 128-k block lies in one quantisation group (g % 128 == 0).
//
// Warps: 8 unpacking warps -- TMEM lane quarter (warp % 4) x column half
// (warp / 4), all of them on every block -- one TMA producer warp, one
// MMA-issuing warp.  Pipeline per block: TMA ring stage (16 KB: 128 rows x
// two blocks, 128-byte swizzle) -> unpack to registers -> tcgen05.st into the
// block's A slot -> "ready" mbarrier (8 arrivals) -> 8 MMAs into the block's
// D slot -> tcgen05.commit to that D slot's "done" mbarrier -> one half-warp
// folds the D kLag blocks later.  TMEM holds 4 A slots (64 columns each) and
// 16 D slots (16 columns each): all 512 columns.  The MMAs of a block take
// ~363 cycles to issue (M = 128, N = 16, K = 16 issues at ~45 cycles), which
// bounds the kernel at ~45 weights per clock per SM; the unpacking warps run
// up to 4 blocks ahead of them.
//
// Work split: a cluster of S CTAs shares tiles, rank r taking the r-th K
// slice; partials meet through distributed shared memory in rank order, so
// results are deterministic.  Every wait is bounded; a timeout sets an abort
// flag that releases all other waits and raises W4A16_DEVERR_TIMEOUT.
#include "common.cuh"
#include "launch.h"
#include "tc_core.cuh"

namespace w4a16 {
namespace {

constexpr int kDeqWarps = 8;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kThreads = 320;
constexpr int kRows = 128;                 // tile rows = TMEM lanes = MMA M
constexpr int kStageBytes = kRows * 128;   // 128 rows x 128 bytes: two 128-k blocks
constexpr int kASlots = 4;                 // A slot of block bg: bg % 4
constexpr int kDSlots = 16;                // D slot of block bg: bg % 16
constexpr int kACols = 64;                 // TMEM columns of one block's A
constexpr int kDCol0 = kASlots * kACols;   // first D column
constexpr int kDCols = 16;
constexpr int kLag = 8;                    // blocks between a block's MMAs and its fold
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxStages = 10;
constexpr uint32_t kIdesc = tc_idesc_bf16(128, 16);
static_assert(kDCol0 + kDSlots * kDCols <= static_cast<int>(kTmemCols), "TMEM columns");
static_assert(kLag + kASlots <= kDSlots, "a D slot is folded before it is reused");

struct TcArgs {
    const uint16_t* x;
    const uint16_t* scale;
    const uint8_t* zero;
    void* y;
    int out_f32;
    int M;
    int N;
    int K;
    int g;
    int ksplit;
    int bpc;  // 128-k blocks per CTA slice (even)
    int tiles_per_cluster;
    int stages;
    uint32_t* err;
};

__host__ __device__ inline int tc_ntok(int MR) { return MR <= 8 ? 8 : 16; }

// Shared memory before the TMA ring: B operand (bpc*16 words x ntok tokens x
// 16 bytes), block sums [bpc][MR], tile reduction [2][4][MR][32], per-warp
// rings of the scale | zero words of blocks awaiting their fold
// [8][kDSlots][32], and (K split
// over a cluster) the partials every rank stores here for the tiles this CTA
// owns, [tpg][S][MR][128].
__host__ __device__ inline int tc_base_bytes(int MR, int bpc, int tpg, int S) {
    const int b = bpc * 16 * tc_ntok(MR) * 16 + bpc * MR * 4 + 2 * 4 * MR * 32 * 4 +
                  kDeqWarps * kDSlots * 32 * 4 + (S > 1 ? tpg * S * MR * kRows * 4 : 0);
    return (b + 127) & ~127;
}
// Whole dynamic shared memory: 1024 bytes of slack for the ring's alignment,
// the ring, its mbarriers (full, empty) and the slots' (ready per A slot, done
// per D slot), the TMEM
// base address and the abort flag.
__host__ __device__ inline int tc_smem_bytes(int base, int ns) {
    return base + 1024 + ns * kStageBytes + (2 * ns + kASlots + kDSlots) * 8 + 16;
}

// Bounded mbarrier wait that gives up at once when another thread aborted.
__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
    for (uint32_t i = 0; i < 8192u; ++i) {
        if (mbar_try_wait_sleep(bar, parity, 100000u)) return true;
        if (*abort_flag) return false;
    }
    *abort_flag = 1;
    return false;
}

template <int MR>
__global__ void __launch_bounds__(kThreads, 1)
k_gemv_tc(const TcArgs a, const __grid_constant__ CUtensorMap wmap) {
    constexpr int NTOK = MR <= 8 ? 8 : 16;
    constexpr int kWordBytes = NTOK * 16;  // one 8-k word of every token
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int S = a.ksplit;
    const int rank = (S > 1) ? static_cast<int>(cluster_rank()) : 0;
    const int cid = blockIdx.x / S;
    const int ncl = gridDim.x / S;
    const int nblk_all = a.K >> 7;
    const int b0 = rank * a.bpc;
    const int nb = max(0, min(nblk_all, b0 + a.bpc) - b0);
    const int nss = (nb + 1) >> 1;  // ring stages per tile
    const int ntiles = (a.N + kRows - 1) / kRows;
    const int my_tiles = (ntiles > cid) ? (ntiles - cid + ncl - 1) / ncl : 0;
    const int G = a.K / a.g;
    const int NS = a.stages;

    unsigned char* xs = smem_raw;
    float* xsum = reinterpret_cast<float*>(smem_raw + a.bpc * 16 * kWordBytes);
    float* red = xsum + a.bpc * MR;
    uint32_t* szr = reinterpret_cast<uint32_t*>(red + 2 * 4 * MR * 32);  // [8][kDSlots][32]
    float* part = reinterpret_cast<float*>(szr + kDeqWarps * kDSlots * 32);
    const int base = tc_base_bytes(MR, a.bpc, a.tiles_per_cluster, S);
    const uint32_t raw = smem_addr(smem_raw);
    unsigned char* ring = smem_raw + (((raw + base + 1023u) & ~1023u) - raw);
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + NS * kStageBytes);
    uint64_t* empty = full + NS;
    uint64_t* ready = empty + NS;
    uint64_t* done = ready + kASlots;
    uint32_t* tmem_base = reinterpret_cast<uint32_t*>(done + kDSlots);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_base + 1);

    grid_dependents_launch();
    if (warp == kMmaWarp) {
        tmem_alloc(tmem_base, kTmemCols);
        tmem_relinquish();
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(full + i, 1);
            mbar_init(empty + i, kDeqWarps);
        }
        for (int i = 0; i < kASlots; ++i) mbar_init(ready + i, kDeqWarps);
        for (int i = 0; i < kDSlots; ++i) mbar_init(done + i, 1);
        *abort_flag = 0;
        mbar_init_fence();
    }
    grid_dependency_wait();

    // Activations first (they gate every MMA): raw 16-byte pieces straight to
    // their place in the B layout; tokens M..NTOK-1 are zero.
    {
        const int words = nb * 16;
        const int pieces = a.M * words;
        for (int i = threadIdx.x; i < pieces; i += blockDim.x) {
            const int t = i / words;
            const int w = i - t * words;
            cp_async_16(xs + w * kWordBytes + t * 16,
                        a.x + static_cast<size_t>(t) * a.K + (static_cast<size_t>(b0) << 7) + w * 8);
        }
        const int zpieces = (NTOK - a.M) * words;
        for (int i = threadIdx.x; i < zpieces; i += blockDim.x) {
            const int t = a.M + i / words;
            const int w = i - (t - a.M) * words;
            *reinterpret_cast<uint4*>(xs + w * kWordBytes + t * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
    }
    tc_fence_before();
    __syncthreads();  // barriers initialised, TMEM allocated, activation copies issued
    tc_fence_after();
    // K split over a cluster: this CTA is running; the matching wait comes
    // before the first store into a peer's shared memory
    if (S > 1) cluster_arrive_relaxed();
    const uint32_t tb = *tmem_base;

    // producer: stage st holds blocks 2 s2, 2 s2 + 1 of tile i (st = i * nss + s2)
    const int total_st = my_tiles * nss;
    int p_st = 0;
    auto produce = [&](int upto) {
        for (; p_st < upto; ++p_st) {
            const int sidx = p_st % NS;
            if (p_st >= NS && !tc_wait(empty + sidx, ((p_st / NS) - 1) & 1, abort_flag)) {
                // aborted: stop producing (consumers give up on their waits too)
                p_st = total_st;
                return;
            }
            const int i = p_st / nss;
            const int s2 = p_st - i * nss;
            mbar_arrive_expect_tx(full + sidx, kStageBytes);
            tma_load_2d(ring + sidx * kStageBytes, &wmap, (b0 + 2 * s2) * 16,
                        (cid + i * ncl) * kRows, full + sidx);
        }
    };
    if (warp == kProducerWarp && lane == 0) produce(min(NS, total_st));

    // pair the values inside each 16-byte piece ((x0,x4), (x1,x5), ...) and
    // take the per-block sums; one thread per (block, token)
    cp_async_wait_all();
    __syncthreads();
    for (int i = threadIdx.x; i < a.M * nb; i += blockDim.x) {
        const int j = i / a.M;
        const int t = i - j * a.M;
        uint4* p0 = reinterpret_cast<uint4*>(xs + j * 16 * kWordBytes + t * 16);
        uint4 v[16];
#pragma unroll
        for (int w = 0; w < 16; ++w) v[w] = p0[w * (kWordBytes / 16)];
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int w = 0; w < 16; ++w) {
            const uint32_t u[4] = {v[w].x, v[w].y, v[w].z, v[w].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                s0 += bf16_to_f32(u[e] & 0xFFFFu);
                s1 += bf16_to_f32(u[e] >> 16);
            }
            uint4 o4;
            o4.x = __byte_perm(v[w].x, v[w].z, 0x5410);  // (x0, x4)
            o4.y = __byte_perm(v[w].x, v[w].z, 0x7632);  // (x1, x5)
            o4.z = __byte_perm(v[w].y, v[w].w, 0x5410);  // (x2, x6)
            o4.w = __byte_perm(v[w].y, v[w].w, 0x7632);  // (x3, x7)
            p0[w * (kWordBytes / 16)] = o4;
        }
        xsum[j * MR + t] = s0 + s1;
    }
    for (int i = threadIdx.x; i < nb * (MR - a.M); i += blockDim.x) {
        const int j = i / (MR - a.M);
        xsum[j * MR + a.M + (i - j * (MR - a.M))] = 0.f;
    }
    fence_proxy_async_smem();  // B is read by the tensor cores (async proxy)
    __syncthreads();
    if (S > 1) cluster_wait();  // every peer CTA has started

    if (warp < kDeqWarps) {
        // ------------------------------------------------------------------
        // unpacking warps: lane quarter q (rows 32q..32q+31), column half h
        // (words 8h..8h+7 of every block).  All eight warps take every block,
        // so a block is ready as soon as each has done half of its rows'
        // work.  Block bg (counted over the CTA's tiles) uses A slot bg % 4 and
        // D slot bg % 16; before writing A slot bg % 4 a warp waits for the
        // MMAs of block bg - 4, which is long done in steady state.  Block bf
        // is folded kLag blocks later by the half h == bf & 1; both halves end
        // a tile at the same iteration, so their pairing barrier cannot stall
        // the pipeline.
        // ------------------------------------------------------------------
        const int q = warp & 3;
        const int h = warp >> 2;
        const int row = q * 32 + lane;
        const uint32_t lane_base = tb + (static_cast<uint32_t>(q * 32) << 16);
        const int total = my_tiles * nb;
        const int lag = min(kLag, max(nb, 1));
        // accumulators of even and odd tiles: with lag <= nb, pending folds
        // belong to at most two consecutive tiles
        float acc_e[MR], acc_o[MR];
#pragma unroll
        for (int m = 0; m < MR; ++m) acc_e[m] = acc_o[m] = 0.f;

        auto tile_end = [&](int i, float (&acc)[MR]) {
            float* rb = red + ((i & 1) * 4 + q) * MR * 32;
            if (h == 1) {
#pragma unroll
                for (int m = 0; m < MR; ++m) rb[m * 32 + lane] = acc[m];
            }
            named_barrier_sync(1 + q, 64);
            if (h == 0) {
                const int n = (cid + i * ncl) * kRows + row;
#pragma unroll
                for (int m = 0; m < MR; ++m) {
                    if (m >= a.M) continue;
                    const float v = acc[m] + rb[m * 32 + lane];
                    if (S == 1) {
                        if (n < a.N) store_out(a.y, a.out_f32, static_cast<size_t>(m) * a.N + n, v);
                    } else {
                        // into the owner's shared memory (CTA i % S of the cluster)
                        st_dsmem_f32(part + ((i * S + rank) * MR + m) * kRows + row,
                                     static_cast<uint32_t>(i % S), v);
                    }
                }
            }
#pragma unroll
            for (int m = 0; m < MR; ++m) acc[m] = 0.f;
        };
        // block bf: its half folds acc += s * (D - (128 + z) * sum x); at the
        // tile's last block both halves end the tile
        auto fold_step = [&](int bf) {
            const int ti = bf / nb;
            const int j = bf - ti * nb;
            if ((bf & 1) == h) {
                const uint32_t sz = szr[(warp * kDSlots + bf % kDSlots) * 32 + lane];
                const int dslot = bf % kDSlots;
                tc_wait(done + dslot, (bf / kDSlots) & 1, abort_flag);
                tc_fence_after();
                float d[MR];
                tmem_ld<MR>(lane_base + kDCol0 + dslot * kDCols, d);
                tmem_wait_ld();
                const float s = __uint_as_float(sz << 16);
                const float o = static_cast<float>(128u + (sz >> 16));
                const float* xsb = xsum + j * MR;
                if (ti & 1) {
#pragma unroll
                    for (int m = 0; m < MR; ++m)
                        if (m < a.M) acc_o[m] = fmaf(s, fmaf(-o, xsb[m], d[m]), acc_o[m]);
                } else {
#pragma unroll
                    for (int m = 0; m < MR; ++m)
                        if (m < a.M) acc_e[m] = fmaf(s, fmaf(-o, xsb[m], d[m]), acc_e[m]);
                }
            }
            if (j == nb - 1) {
                if (ti & 1) tile_end(ti, acc_o);
                else tile_end(ti, acc_e);
            }
        };

        int bg = 0;
        for (int st = 0; st < total_st; ++st) {
            const int i = st / nss;
            const int s2 = st - i * nss;
            const int sidx = st % NS;
            tc_wait(full + sidx, (st / NS) & 1, abort_flag);
            const unsigned char* src = ring + sidx * kStageBytes + row * 128;
            for (int half = 0; half < 2; ++half) {
                const int j = 2 * s2 + half;
                if (j >= nb) break;
                // this warp's 8 words of the block: chunks 2h, 2h + 1 of the
                // block's 4 (128-byte swizzle: chunk c of row r at c ^ (r % 8))
                const int c0 = (half << 2) + 2 * h;
                const uint4 w0 = *reinterpret_cast<const uint4*>(src + ((c0 ^ (row & 7)) << 4));
                const uint4 w1 = *reinterpret_cast<const uint4*>(src + (((c0 + 1) ^ (row & 7)) << 4));
                const uint32_t ws[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
                uint32_t A[32];
#pragma unroll
                for (int w = 0; w < 8; ++w) {  // word 8h + w: k = 8 (8h + w) .. + 7 of the block
                    const uint32_t u = ws[w];
                    A[4 * w + 0] = (u & 0x000F000Fu) | 0x43004300u;
                    A[4 * w + 1] = ((u >> 4) & 0x000F000Fu) | 0x43004300u;
                    A[4 * w + 2] = ((u >> 8) & 0x000F000Fu) | 0x43004300u;
                    A[4 * w + 3] = ((u >> 12) & 0x000F000Fu) | 0x43004300u;
                }
                // this half folds the block kLag blocks later: load its scale and
                // zero point now (stored to the ring at the end of the iteration,
                // so the loads' latency overlaps the block's TMEM traffic)
                const bool folds = (bg & 1) == h;
                uint32_t sz_new = 0u;  // rows beyond N: s = 0
                {
                    const int n = (cid + i * ncl) * kRows + row;
                    if (folds && n < a.N) {
                        const size_t gi = static_cast<size_t>(n) * G + (((b0 + j) << 7) / a.g);
                        sz_new = ldg_nc_u16(a.scale + gi) | (ldg_nc_u8(a.zero + gi) << 16);
                    }
                }
                if (bg >= kASlots)  // A slot free: the MMAs of block bg - 4 have completed
                    tc_wait(done + (bg - kASlots) % kDSlots, ((bg - kASlots) / kDSlots) & 1,
                            abort_flag);
                tc_fence_after();
                tmem_st_x32(lane_base + (bg % kASlots) * kACols + h * 32, A);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(ready + bg % kASlots);
                if (bg >= lag) fold_step(bg - lag);
                if (folds) szr[(warp * kDSlots + bg % kDSlots) * 32 + lane] = sz_new;
                ++bg;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty + sidx);  // both blocks of the stage read
        }
        for (int bf = max(0, total - lag); bf < total; ++bf) fold_step(bf);
    } else if (warp == kProducerWarp) {
        if (lane == 0) produce(total_st);
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            const uint32_t xs_addr = smem_addr(xs);
            const int total = my_tiles * nb;
            for (int bg = 0; bg < total; ++bg) {
                const int j = bg % nb;
                const int aslot = bg % kASlots;
                const int dslot = bg % kDSlots;
                tc_wait(ready + aslot, (bg / kASlots) & 1, abort_flag);
                tc_fence_after();
                const uint32_t a_t = tb + aslot * kACols;
                const uint32_t d_t = tb + kDCol0 + dslot * kDCols;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t desc =
                        smem_desc_kmajor(xs_addr + (j * 16 + 2 * kk) * kWordBytes, kWordBytes,
                                         NTOK == 16 ? 128u : 0u);
                    tc_mma_tmem_a(d_t, a_t + kk * 8, desc, kIdesc, kk > 0 ? 1u : 0u);
                }
                tc_commit(done + dslot);
            }
        }
    }

    // K split: every rank stored its partials of tile i into the shared
    // memory of the owner, rank i % S; after one cluster barrier the owner
    // adds them in rank order (deterministic) and stores y
    if (S > 1) {
        cluster_barrier();
        const int per_t = a.M * kRows;
        const int tot = my_tiles * per_t;
        for (int idx = threadIdx.x; idx < tot; idx += blockDim.x) {
            const int i = idx / per_t;
            if ((i % S) != rank) continue;
            const int rem = idx - i * per_t;
            const int m = rem / kRows;
            const int row = rem - m * kRows;
            float v = 0.f;
            for (int r = 0; r < S; ++r) v += part[((i * S + r) * MR + m) * kRows + row];
            const int n = (cid + i * ncl) * kRows + row;
            if (n < a.N) store_out(a.y, a.out_f32, static_cast<size_t>(m) * a.N + n, v);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tb, kTmemCols);
    }
    if (threadIdx.x == 0 && *abort_flag) raise_device_error(a.err, W4A16_DEVERR_TIMEOUT);
}

using TcKernel = void (*)(TcArgs, CUtensorMap);

int tc_mr(int M) { return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : M <= 8 ? 8 : 16; }

TcKernel pick_tc_kernel(int M) {
    switch (tc_mr(M)) {
        case 1: return k_gemv_tc<1>;
        case 2: return k_gemv_tc<2>;
        case 4: return k_gemv_tc<4>;
        case 8: return k_gemv_tc<8>;
        default: return k_gemv_tc<16>;
    }
}

}  // namespace

GemvPlan plan_gemv_tc(const DeviceInfo& dev, int M, int N, int K, int g, int k_split_req) {
    (void)g;
    GemvPlan p{};
    const int nblk = K / 128;
    const int ntiles = (N + kRows - 1) / kRows;
    const int MR = tc_mr(M);
    const void* kern = reinterpret_cast<const void*>(pick_tc_kernel(M));
    const int budget = dev.max_smem_optin;
    long best_cost = -1;
    int bS = 0, bcl = 0, btpg = 0, bbpc = 0;
    for (int S = 1; S <= 8; S *= 2) {
        if (k_split_req > 0 && S != k_split_req) continue;
        int bpc = (nblk + S - 1) / S;
        bpc += bpc & 1;
        if ((S - 1) * bpc >= nblk && S > 1) continue;  // a rank would have no block
        if (tc_smem_bytes(tc_base_bytes(MR, bpc, 1, S), 2) > budget) continue;
        int clusters = dev.sms / S;
        if (S > 1) {
            const int mc = max_active_clusters(kern, kThreads, budget, S);
            if (mc < 1) continue;
            if (clusters > mc) clusters = mc;
        }
        if (clusters > ntiles) clusters = ntiles;
        const int tpg = (ntiles + clusters - 1) / clusters;
        if (tc_smem_bytes(tc_base_bytes(MR, bpc, tpg, S), 2) > budget) continue;
        const long cost = static_cast<long>(tpg) * bpc;
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            bS = S;
            bcl = clusters;
            btpg = tpg;
            bbpc = bpc;
        }
    }
    if (best_cost < 0) return p;  // ctas = 0: not feasible
    const int base = tc_base_bytes(MR, bbpc, btpg, bS);
    const int steps = btpg * ((bbpc + 1) / 2);
    int ns = 2;
    while (ns < kMaxStages && ns < steps && tc_smem_bytes(base, ns + 1) <= budget) ++ns;
    int smem = tc_smem_bytes(base, ns);
    // one CTA per SM: each CTA holds all 512 TMEM columns
    const int floor_one_cta = dev.smem_per_sm / 2 + 1024;
    if (smem < floor_one_cta) smem = floor_one_cta;
    p.kernel_id = 3;
    p.k_split = bS;
    p.wpt = 1;
    p.units_per_cta = bbpc;
    p.threads = kThreads;
    p.ctas = bcl * bS;
    p.tiles_per_cluster = btpg;
    p.stages = ns;
    p.smem_bytes = smem;
    return p;
}

cudaError_t launch_gemv_tc(const GemvArgs& a, const GemvPlan& p, cudaStream_t s) {
    TcArgs k{};
    k.x = a.x;
    k.scale = a.scale;
    k.zero = a.zero;
    k.y = a.y;
    k.out_f32 = a.out_f32;
    k.M = a.M;
    k.N = a.N;
    k.K = a.K;
    k.g = a.g;
    k.ksplit = p.k_split;
    k.bpc = p.units_per_cta;
    k.tiles_per_cluster = p.tiles_per_cluster;
    k.stages = p.stages;
    k.err = a.err;
    CUtensorMap wmap;
    if (!encode_weight_map(&wmap, a.wq, a.N, a.K, kRows)) return cudaErrorInvalidValue;
    TcKernel kern = pick_tc_kernel(a.M);
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
