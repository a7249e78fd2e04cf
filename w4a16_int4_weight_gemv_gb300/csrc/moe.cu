// Expert-indexed W4A16 GEMV (sm_103a): the grouped expert kernel of the
// local-kimi README, technical-detail section, as a true GEMV.
//
// For token t and routed slot j, expert e = ids[t][j] multiplies its own INT4
// matrix W_e by the slot's activation row.  Tokens that route to the same
// expert share one pass over that expert's weights: CTA (chunk, d, bank)
// finds the d-th distinct expert among the routed slots (in order of first
// appearance), gathers the activation rows of every slot routed to it into
// shared memory and streams a chunk of W_e's rows against all of them at
// once.  The routed ids live on the device, so the grid is sized for the
// worst case (min(E, M*topk) distinct experts) and CTAs beyond the actual
// count exit at once.
//
// Transport and arithmetic are those of the dense warp-MMA kernel
// (gemv_mma.cu, mma_core.cuh): one 2-D tensor map over the whole stacked
// bank [E*N rows][K/8 words], per-warp rings of 16-row x 512-k stages filled
// by two 128-byte-swizzled TMA boxes, ldmatrix fragments, mma.sync with the
// 128 + code bf16 trick and the per-block zero-point/scale correction.  A
// chunk is 4 tiles of 16 rows with two warps per tile (K halves, partials
// added in shared memory in a fixed order), or 8 tiles with a warp per tile
// -- and then possibly two or four tiles per warp in turn -- when smaller
// chunks would take more than one wave.  A CTA's scales and zero points (its
// rows are consecutive, so two contiguous byte spans) are copied into
// shared memory once, before its first weight box is issued.
//
// One launch can serve two banks of the same shape against the same
// activations (grid z): the gate and up products of a SwiGLU expert FFN.
// The activations can also be formed while staging, h = bf16(silu(g) * u)
// from per-slot gate and up outputs: the down product of that FFN, without a
// separate SwiGLU pass.
//
// With route weights the per-slot results go to an fp32 workspace; y[t] =
// sum_j r[t][j] d[t][j] is then formed in slot order -- a fixed order, so
// the result is deterministic (no floating-point atomics) -- by a second
// kernel, or, inside the FFN chain, by the last CTA to finish each row
// chunk.
#include <atomic>

#include "common.cuh"
#include "launch.h"
#include "mma_core.cuh"

namespace w4a16 {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kSB = 4;                   // 128-k blocks per step (512 k)
constexpr int kHalfBytes = 2048;         // one TMA box: 16 rows x 128 bytes
constexpr int kStageA = 2 * kHalfBytes;
constexpr unsigned kBoxRows = 16;
constexpr int kMaxSlots = 256;
constexpr int kMaxTableGroups = 64;      // scale/zero table in shared memory up to G = 64
constexpr int kMaxStages = 4;
constexpr int kSwBatch = 2;              // gate/up pieces per thread per load batch

struct MoeKernelArgs {
    const uint16_t* x;
    int x_per_slot;
    const uint16_t* sw_gate;  // non-null: activations are h = bf16(silu(gate) * up), [S][K]
    const uint16_t* sw_up;
    const int32_t* ids;
    MoeBank bank[2];
    float* ws;  // fp32 per-slot outputs [S][N] (a routed sum follows), else bf16 bank[z].y
    int M;
    int topk;
    int E;
    int N;
    int K;
    int g;
    int stages;
    int tpw;    // 16-row tiles per warp, one after another (8-tile CTAs only)
    int early;  // ids, weights, scales may be read before the grid dependency wait
    // Routed sum inside the launch (fused FFN chain): per 64-row chunk, the
    // last CTA to finish its partials adds every token's slots in slot order.
    unsigned* chunk_count;  // [gridDim.x] arrival counters (zero between calls)
    const float* route_w;
    uint16_t* y_routed;     // bf16 [M][N]
    // zero these counters (the next launch's) before anything else
    unsigned* zero_count;
    int zero_n;
    uint32_t* err;
};

// The CTA's scales and zero points, copied verbatim from the bank: its rows'
// bf16 scales [rows][G], then (16-byte aligned) their u8 zero points, each
// placed 0..15 bytes into its area so that it agrees with its source modulo
// 16 (the copy then moves aligned 16-byte pieces).
__host__ __device__ inline int moe_table_scale_bytes(int tiles, int G) {
    return (tiles * 16 * G * 2 + 16 + 15) & ~15;
}
__host__ __device__ inline int moe_table_bytes(int tiles, int G) {
    return moe_table_scale_bytes(tiles, G) + tiles * 16 * G + 16;
}

struct MoeLayout {
    int xsum, red, tab, base;
};
__host__ __device__ inline MoeLayout moe_layout(int Mpad, int nblk, int G, int tiles, int tpw) {
    MoeLayout L;
    L.xsum = Mpad * mma_token_stride(nblk);
    L.red = L.xsum + nblk * Mpad * 4;
    // K-half partials only when two warps share a tile (4-tile CTAs)
    L.tab = L.red + (kWarps / tiles > 1 ? tiles * 16 * Mpad * 4 : 0);
    const int end = L.tab + (G <= kMaxTableGroups ? moe_table_bytes(tiles * tpw, G) : 0);
    L.base = (end + 127) & ~127;
    return L;
}
__host__ __device__ inline int moe_smem_bytes(int Mpad, int nblk, int G, int tiles, int tpw,
                                              int ns) {
    return moe_layout(Mpad, nblk, G, tiles, tpw).base + 1024 + kWarps * ns * (kStageA + 8);
}

// Bytes [src, src + n) of global memory to shared memory at dst, where dst
// and src agree modulo 16: the aligned body by 16-byte cp.async, the ragged
// head and tail by byte loads.  Before reading, the caller waits for its
// cp.async groups and synchronises the CTA.
__device__ __forceinline__ void copy_span_async(unsigned char* dst, const unsigned char* src,
                                                int n) {
    const uintptr_t s0 = reinterpret_cast<uintptr_t>(src);
    const uintptr_t a0 = (s0 + 15) & ~static_cast<uintptr_t>(15);
    const uintptr_t a1 = (s0 + n) & ~static_cast<uintptr_t>(15);
    const int head = (a0 < s0 + n) ? static_cast<int>(a0 - s0) : n;
    const int body = (a0 < s0 + n && a1 > a0) ? static_cast<int>(a1 - a0) : 0;
    for (int i = threadIdx.x; i < body / 16; i += blockDim.x)
        cp_async_16(dst + head + 16 * i, src + head + 16 * i);
    const int tail0 = head + body;
    for (int i = threadIdx.x; i < head + (n - tail0); i += blockDim.x) {
        const int o = i < head ? i : tail0 + (i - head);
        dst[o] = static_cast<unsigned char>(ldg_nc_u8(src + o));
    }
}

// y[t][n] = bf16(sum_j r[t][j] * ws[t][j][n]) over slots with a valid expert
// id, for rows n in [n0, n1): fp32, j ascending (the same order as
// k_moe_route_sum).
__device__ __forceinline__ void moe_route_rows(const float* ws, const float* route_w,
                                               const int* ids, uint16_t* y, int M, int topk,
                                               int E, int N, int n0, int n1) {
    const int rows = n1 - n0;
    for (int i = threadIdx.x; i < M * rows; i += blockDim.x) {
        const int t = i / rows;
        const int n = n0 + (i - t * rows);
        float v = 0.f;
        for (int j = 0; j < topk; ++j) {
            const int e = ids[t * topk + j];
            if (e < 0 || e >= E) continue;
            v = fmaf(route_w[t * topk + j], ws[(static_cast<size_t>(t) * topk + j) * N + n], v);
        }
        y[static_cast<size_t>(t) * N + n] = f32_to_bf16_rn(v);
    }
}

// The chunk's partials of this CTA are written (or it has none): count it;
// the CTA that completes the count forms the chunk's routed sums and resets
// the counter for the next call.
__device__ __forceinline__ void moe_chunk_done(const MoeKernelArgs& a, const int* ids, int rows) {
    if (!a.chunk_count) return;
    __shared__ unsigned s_last;
    __threadfence();  // this CTA's partials are visible device-wide before it is counted
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned total = gridDim.y * gridDim.z;
        s_last = (atomicAdd(a.chunk_count + blockIdx.x, 1u) == total - 1) ? 1u : 0u;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();  // every counted CTA's partials are visible to this one
    const int n0 = blockIdx.x * rows;
    moe_route_rows(a.ws, a.route_w, ids, a.y_routed, a.M, a.topk, a.E, a.N, n0,
                   min(a.N, n0 + rows));
    if (threadIdx.x == 0) a.chunk_count[blockIdx.x] = 0u;
}

template <int NT, int TILES>
__global__ void __launch_bounds__(kThreads, NT == 1 ? 2 : 1)
k_moe_tma(const MoeKernelArgs a, const __grid_constant__ CUtensorMap map0,
          const __grid_constant__ CUtensorMap map1) {
    constexpr int Mpad = 8 * NT;
    constexpr int kTiles = TILES;
    constexpr int kWpt = kWarps / kTiles;  // warps sharing a tile (K halves)
    constexpr int kRowsPerTileSet = kTiles * 16;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __shared__ int s_ids[kMaxSlots];
    __shared__ unsigned char s_slots[kMaxSlots];
    __shared__ unsigned s_mask[kWarps];
    __shared__ int s_expert;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int z = blockIdx.z;
    const CUtensorMap* wmap = z ? &map1 : &map0;
    const MoeBank bank = a.bank[z];
    const int S = a.M * a.topk;
    const int nblk = a.K >> 7;
    const int nsteps = (nblk + kSB - 1) / kSB;
    const int G = a.K / a.g;
    const bool use_table = G <= kMaxTableGroups;
    const int tok_stride = mma_token_stride(nblk);
    const int NS = a.stages;
    const int cta_rows = kRowsPerTileSet * a.tpw;  // rows of expert e this CTA covers

    // Programmatic dependent launch: without `early` everything waits for the
    // preceding grid; with it (a launch inside the FFN chain, whose
    // predecessor signalled only after its own wait) the routed ids, weights
    // and scales -- inputs of the whole chain -- are read first and only the
    // activations and outputs wait.
    if (threadIdx.x == 0) prefetch_tensor_map(wmap);
    if (!a.early) grid_dependency_wait();
    if (a.zero_count && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0)
        for (int i = threadIdx.x; i < a.zero_n; i += blockDim.x) a.zero_count[i] = 0u;

    // 1. which expert does this CTA serve?  One thread per routed slot
    // (S <= kThreads): a slot is its expert's first if no earlier slot names
    // the same expert; the first slots are counted in slot order by ballots.
    const int si = threadIdx.x;
    int my_id = -1;
    if (si < S) {
        my_id = a.ids[si];
        s_ids[si] = my_id;
    }
    if (threadIdx.x == 0) s_expert = -1;
    __syncthreads();
    bool first = false;
    if (si < S) {
        first = (my_id >= 0 && my_id < a.E);
        if (!first && blockIdx.x == 0 && blockIdx.y == 0 && z == 0)
            raise_device_error(a.err, W4A16_DEVERR_EXPERT_ID);
        for (int j = 0; j < si && first; ++j) first = (s_ids[j] != my_id);
    }
    const unsigned lt = (1u << lane) - 1u;
    unsigned fm = __ballot_sync(0xFFFFFFFFu, first);
    if (lane == 0) s_mask[warp] = fm;
    __syncthreads();
    if (first) {
        int ord = __popc(fm & lt);
        for (int w = 0; w < warp; ++w) ord += __popc(s_mask[w]);
        if (ord == static_cast<int>(blockIdx.y)) s_expert = my_id;
    }
    __syncthreads();
    const int e = s_expert;

    // invalid ids produce zero rows in the per-slot output
    if (a.ws == nullptr && blockIdx.y == 0) {
        if (a.early) grid_dependency_wait();
        for (int i = 0; i < S; ++i) {
            if (s_ids[i] >= 0 && s_ids[i] < a.E) continue;
            for (int row = blockIdx.x * cta_rows + threadIdx.x;
                 row < min(a.N, (blockIdx.x + 1) * cta_rows); row += blockDim.x)
                bank.y[static_cast<size_t>(i) * a.N + row] = 0;
        }
    }
    if (e < 0) {
        grid_dependents_launch();
        if (a.chunk_count) {
            grid_dependency_wait();  // the counters were zeroed by the preceding launch
            moe_chunk_done(a, s_ids, cta_rows);
        }
        return;
    }

    // the slots routed to e, in slot order
    const bool mine = (si < S) && my_id == e;
    fm = __ballot_sync(0xFFFFFFFFu, mine);
    if (lane == 0) s_mask[warp] = fm;  // its earlier reads all precede the last barrier

    const MoeLayout lay = moe_layout(Mpad, nblk, G, kTiles, a.tpw);
    unsigned char* xs = smem_raw;
    float* xsum = reinterpret_cast<float*>(smem_raw + lay.xsum);
    float* red = reinterpret_cast<float*>(smem_raw + lay.red);
    unsigned char* tab = smem_raw + lay.tab;
    const uint32_t raw_addr = smem_addr(smem_raw);
    const int a_off = static_cast<int>(((raw_addr + lay.base + 1023u) & ~1023u) - raw_addr);
    unsigned char* ring = smem_raw + a_off + warp * NS * kStageA;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem_raw + a_off + kWarps * NS * kStageA) + warp * NS;

    // warp (tl, kp) takes tiles tile0 + tp * kTiles, tp < ntl, of expert e
    // (kp: its K part when kWpt warps share a tile)
    const int tl = warp / kWpt;
    const int kp = warp - tl * kWpt;
    const int tile0 = blockIdx.x * kTiles * a.tpw + tl;
    const int ntiles_all = (a.N + 15) >> 4;
    const int ntl = tile0 < ntiles_all ? min(a.tpw, (ntiles_all - tile0 + kTiles - 1) / kTiles) : 0;
    const int ms = (nsteps > kp) ? (nsteps - kp + kWpt - 1) / kWpt : 0;  // steps per tile
    const int per_pass = ntl * ms;

    if (lane == 0) {
        for (int i = 0; i < NS; ++i) mbar_init(bars + i, 1);
        mbar_init_fence();
    }
    __syncthreads();  // s_mask, barriers
    int nslots = 0;
    if (mine) {
        int pos = __popc(fm & lt);
        for (int w = 0; w < warp; ++w) pos += __popc(s_mask[w]);
        s_slots[pos] = static_cast<unsigned char>(si);
    }
    for (int w = 0; w < kWarps; ++w) nslots += __popc(s_mask[w]);
    __syncthreads();  // s_slots
    const int npass = (nslots + Mpad - 1) / Mpad;
    const int total = npass * per_pass;  // every pass streams the same weights

    // 2. The CTA's scales and zero points and, when they are plain inputs,
    // the first pass's activation rows are requested before any weight copy
    // is issued: issued after, they would wait behind every CTA's weight
    // stream (several microseconds at launch, when all CTAs fill their rings
    // at once), and compute cannot start without them.  The table moves as
    // two contiguous byte spans (this CTA's rows are consecutive), so a few
    // hundred 16-byte copies replace a load per (row, group).
    const uint16_t* escale = bank.scale + static_cast<size_t>(e) * a.N * G;
    const uint8_t* ezero = bank.zero + static_cast<size_t>(e) * a.N * G;
    const int n_base = blockIdx.x * cta_rows;
    const int rows_valid = min(cta_rows, a.N - n_base);
    const unsigned char* src_s = reinterpret_cast<const unsigned char*>(escale + static_cast<size_t>(n_base) * G);
    const unsigned char* src_z = ezero + static_cast<size_t>(n_base) * G;
    const unsigned char* tab_s = tab + (reinterpret_cast<uintptr_t>(src_s) & 15);
    const unsigned char* tab_z =
        tab + moe_table_scale_bytes(kTiles * a.tpw, G) + (reinterpret_cast<uintptr_t>(src_z) & 15);
    if (use_table) {
        copy_span_async(const_cast<unsigned char*>(tab_s), src_s, rows_valid * G * 2);
        copy_span_async(const_cast<unsigned char*>(tab_z), src_z, rows_valid * G);
    }
    // activation rows of slots [base, base + m) to xs (natural order)
    auto stage_x_async = [&](int base, int m) {
        const int pieces = m * nblk * 16;  // 16-byte pieces of 8 values
        for (int i = threadIdx.x; i < pieces; i += blockDim.x) {
            const int n = i / (nblk * 16);
            const int p = i - n * nblk * 16;
            const int slot = s_slots[base + n];
            const int row = a.x_per_slot ? slot : slot / a.topk;
            cp_async_16(xs + n * tok_stride + p * 16, a.x + static_cast<size_t>(row) * a.K + p * 8);
        }
    };
    const bool x_first = !a.sw_gate && !a.early;  // first pass's rows may be read now
    if (x_first) stage_x_async(0, min(Mpad, nslots));

    // producer cursor over (pass, tile, step); the weights do not depend on
    // the pass
    int w_i = 0;
    auto issue = [&]() {
        const int stg = w_i % NS;
        uint64_t* bar = bars + stg;
        unsigned char* dst = ring + stg * kStageA;
        const int rr = w_i % per_pass;
        const int tp = rr / ms;
        const int ks = kp + (rr - tp * ms) * kWpt;
        const int row0 = e * a.N + (tile0 + tp * kTiles) * 16;  // first row in the stacked bank
        const int blk0 = ks * kSB;
        const int nbs = min(kSB, nblk - blk0);
        const int nh = (nbs + 1) >> 1;
        if (lane == 0) {
            if (w_i >= NS) fence_proxy_async_smem();
            mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nh * kHalfBytes));
            tma_load_2d(dst, wmap, blk0 * 16, row0, bar);
            if (nh > 1) tma_load_2d(dst + kHalfBytes, wmap, blk0 * 16 + 32, row0, bar);
        }
        ++w_i;
    };
    while (w_i < NS && w_i < total) issue();

    if (a.early) grid_dependency_wait();
    // dependents may start now: everything this grid reads is complete
    grid_dependents_launch();

    const int r = lane >> 2;
    const int c = lane & 3;
    const int lrow = (lane & 7) + (((lane >> 3) & 1) << 3);
    const uint32_t lbase = static_cast<uint32_t>(lrow * 128);
    const int lsw = lane & 7;
    const int lch = lane >> 4;
    bool timed_out = false;
    int c_i = 0;  // consumer cursor

    for (int base = 0; base < nslots; base += Mpad) {
        const int m = min(Mpad, nslots - base);
        // activations of the pass's slots, natural order, then paired in place
        if (a.sw_gate) {
            // h = bf16(silu(gate) * up) of each slot; a batch's gate/up pieces
            // are loaded before any is converted
            const int pieces = m * nblk * 16;
            for (int i0 = 0; i0 < pieces; i0 += kSwBatch * kThreads) {
                uint4 gv[kSwBatch], uv[kSwBatch];
#pragma unroll
                for (int j = 0; j < kSwBatch; ++j) {
                    const int i = i0 + j * kThreads + static_cast<int>(threadIdx.x);
                    if (i < pieces) {
                        const int n = i / (nblk * 16);
                        const int p = i - n * nblk * 16;
                        const size_t src = static_cast<size_t>(s_slots[base + n]) * a.K + p * 8;
                        gv[j] = __ldg(reinterpret_cast<const uint4*>(a.sw_gate + src));
                        uv[j] = __ldg(reinterpret_cast<const uint4*>(a.sw_up + src));
                    }
                }
#pragma unroll
                for (int j = 0; j < kSwBatch; ++j) {
                    const int i = i0 + j * kThreads + static_cast<int>(threadIdx.x);
                    if (i >= pieces) continue;
                    const int n = i / (nblk * 16);
                    const int p = i - n * nblk * 16;
                    const uint32_t gw[4] = {gv[j].x, gv[j].y, gv[j].z, gv[j].w};
                    const uint32_t uw[4] = {uv[j].x, uv[j].y, uv[j].z, uv[j].w};
                    uint32_t hw[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float h0 = silu_mul(bf16_to_f32(gw[q] & 0xFFFFu), bf16_to_f32(uw[q] & 0xFFFFu));
                        const float h1 = silu_mul(bf16_to_f32(gw[q] >> 16), bf16_to_f32(uw[q] >> 16));
                        hw[q] = f32_to_bf16_rn(h0) | (static_cast<uint32_t>(f32_to_bf16_rn(h1)) << 16);
                    }
                    *reinterpret_cast<uint4*>(xs + n * tok_stride + p * 16) =
                        make_uint4(hw[0], hw[1], hw[2], hw[3]);
                }
            }
            cp_async_wait_all();  // the scale table's copies
        } else {
            if (!(x_first && base == 0)) stage_x_async(base, m);
            cp_async_wait_all();
        }
        __syncthreads();
        pair_x_in_place<NT>(m, nblk, xs, xsum, tok_stride);
        __syncthreads();

        // 3. stream this warp's K part of its tiles against the pass's slots
        for (int tp = 0; tp < ntl; ++tp) {
        const int tile = tile0 + tp * kTiles;  // 16-row tile of expert e
        const int trow = (tp * kTiles + tl) * 16;  // its first row in the CTA's table
        const int n0 = tile * 16 + r;
        float acc[NT][4];
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[t][i] = 0.f;
        for (int s = 0; s < ms; ++s) {
            const int stg = c_i % NS;
            if (!mbar_wait_bounded(bars + stg, (c_i / NS) & 1)) timed_out = true;
            const uint32_t sa = smem_addr(ring + stg * kStageA);
            const int lb0 = (kp + s * kWpt) * kSB;
            const int nbs = min(kSB, nblk - lb0);
#pragma unroll
            for (int bb = 0; bb < kSB; ++bb) {
                if (bb < nbs) {
                    const uint32_t hb = sa + (bb >> 1) * kHalfBytes + lbase;
                    const int cb = (bb & 1) * 4 + lch;
                    uint32_t q0[4], q1[4];
                    ldmatrix_x4(q0, hb + (static_cast<uint32_t>(cb ^ lsw) << 4));
                    ldmatrix_x4(q1, hb + (static_cast<uint32_t>((cb + 2) ^ lsw) << 4));
                    MmaBlockLoad L;
                    L.w0 = make_uint4(q0[0], q0[2], q1[0], q1[2]);
                    L.w1 = make_uint4(q0[1], q0[3], q1[1], q1[3]);
                    const int blk = lb0 + bb;
                    const int grp = (blk << 7) / a.g;
                    if (use_table) {
                        const int i0 = (trow + r) * G + grp;
                        const int i1 = i0 + 8 * G;
                        L.sz0 = *reinterpret_cast<const uint16_t*>(tab_s + 2 * i0) |
                                (static_cast<uint32_t>(tab_z[i0]) << 16);
                        L.sz1 = *reinterpret_cast<const uint16_t*>(tab_s + 2 * i1) |
                                (static_cast<uint32_t>(tab_z[i1]) << 16);
                    } else {
                        L.sz0 = 0u;
                        L.sz1 = 0u;
                        if (n0 < a.N) {
                            const size_t gi = static_cast<size_t>(n0) * G + grp;
                            L.sz0 = ldg_nc_u16(escale + gi) | (ldg_nc_u8(ezero + gi) << 16);
                        }
                        if (n0 + 8 < a.N) {
                            const size_t gi = static_cast<size_t>(n0 + 8) * G + grp;
                            L.sz1 = ldg_nc_u16(escale + gi) | (ldg_nc_u8(ezero + gi) << 16);
                        }
                    }
                    mma_block<NT>(acc, L, xs + blk * 256, xsum + blk * Mpad, tok_stride, m, lane);
                }
            }
            __syncwarp();  // every lane is done with the stage
            ++c_i;
            if (w_i < total) issue();
        }

        // 4. add the K parts (fixed order) and store per-slot outputs
        float* rb = red + tl * 16 * Mpad;
        if constexpr (kWpt > 1) {
            if (kp == 1) {
#pragma unroll
                for (int t = 0; t < NT; ++t)
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        rb[(r + ((i >> 1) << 3)) * Mpad + t * 8 + 2 * c + (i & 1)] = acc[t][i];
            }
            named_barrier_sync(1 + tl, kWpt * 32);
        }
        if (kp == 0) {
#pragma unroll
            for (int t = 0; t < NT; ++t)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int row = r + ((i >> 1) << 3);
                    const int tok = t * 8 + 2 * c + (i & 1);
                    const int n = tile * 16 + row;
                    if (tok < m && n < a.N) {
                        const float v = (kWpt > 1) ? acc[t][i] + rb[row * Mpad + tok] : acc[t][i];
                        const size_t o = static_cast<size_t>(s_slots[base + tok]) * a.N + n;
                        if (a.ws) a.ws[o] = v;
                        else bank.y[o] = f32_to_bf16_rn(v);
                    }
                }
        }
        if constexpr (kWpt > 1) named_barrier_sync(1 + tl, kWpt * 32);  // rb is free again
        }
        __syncthreads();  // xs is rewritten by the next pass
    }
    if (timed_out && lane == 0) raise_device_error(a.err, W4A16_DEVERR_TIMEOUT);
    moe_chunk_done(a, s_ids, cta_rows);
}

// y[t][n] = sum_j r[t][j] * ws[t][j][n] over slots with a valid expert id.
__global__ void k_moe_route_sum(const float* __restrict__ ws, const float* __restrict__ route_w,
                                const int32_t* __restrict__ ids, uint16_t* __restrict__ y,
                                int M, int topk, int E, int N) {
    const int total = M * N;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
        const int t = i / N;
        const int n = i - t * N;
        float v = 0.f;
        for (int j = 0; j < topk; ++j) {
            const int e = ids[t * topk + j];
            if (e < 0 || e >= E) continue;
            v = fmaf(route_w[t * topk + j], ws[(static_cast<size_t>(t) * topk + j) * N + n], v);
        }
        y[i] = f32_to_bf16_rn(v);
    }
}

using MoeKernel = void (*)(MoeKernelArgs, CUtensorMap, CUtensorMap);

MoeKernel pick_moe_kernel(int Mpad, int tiles) {
    if (Mpad == 8) return tiles == 4 ? k_moe_tma<1, 4> : k_moe_tma<1, 8>;
    return tiles == 4 ? k_moe_tma<2, 4> : k_moe_tma<2, 8>;
}

// static shared memory of a kernel instance (queried once per instance)
int moe_static_smem(MoeKernel k) {
    static std::atomic<int> cached[4] = {{-1}, {-1}, {-1}, {-1}};
    const int i = (k == k_moe_tma<1, 4>) ? 0 : (k == k_moe_tma<1, 8>) ? 1 : (k == k_moe_tma<2, 4>) ? 2 : 3;
    int v = cached[i].load(std::memory_order_relaxed);
    if (v < 0) {
        cudaFuncAttributes fa{};
        v = (cudaFuncGetAttributes(&fa, k) == cudaSuccess) ? static_cast<int>(fa.sharedSizeBytes) : 4096;
        cached[i].store(v, std::memory_order_relaxed);
    }
    return v;
}

}  // namespace

int moe_row_chunks(int N) { return (N + 63) / 64; }

int moe_smem_need(int M, int K, int g) {
    const int Mpad = M <= 8 ? 8 : 16;
    return moe_smem_bytes(Mpad, K / 128, K / g, 8, 1, 2);
}

cudaError_t launch_moe(const MoeArgs& a, const DeviceInfo& dev, cudaStream_t s) {
    MoeKernelArgs k{};
    k.x = a.x;
    k.x_per_slot = a.x_per_slot;
    k.sw_gate = a.sw_gate;
    k.sw_up = a.sw_up;
    k.ids = a.ids;
    k.bank[0] = a.bank[0];
    k.bank[1] = a.nbanks > 1 ? a.bank[1] : a.bank[0];
    k.ws = a.route_w ? a.ws : nullptr;
    k.M = a.M;
    k.topk = a.topk;
    k.E = a.E;
    k.N = a.N;
    k.K = a.K;
    k.g = a.g;
    k.err = a.err;
    const int S = a.M * a.topk;
    const int nblk = a.K / 128;
    const int G = a.K / a.g;
    // slots per pass: 8 for up to 8 tokens (a token's slots normally name
    // distinct experts, so an expert then has at most M slots), else 16;
    // more slots on one expert take more passes
    const int Mpad = (a.M <= 8) ? 8 : 16;
    const int dmax = S < a.E ? S : a.E;
    const int nz = a.nbanks > 1 ? 2 : 1;
    // 64-row CTAs unless that takes more than one wave of two CTAs per SM;
    // then 128-row CTAs, and a warp takes two or four tiles in turn while the
    // grid would still need more than one wave
    const int tiles = (((a.N + 63) / 64) * dmax * nz > 2 * dev.sms) ? 8 : 4;
    MoeKernel kern = pick_moe_kernel(Mpad, tiles);
    // stages: as many as leave room for two CTAs per SM (8-slot passes),
    // counting the kernel's static shared memory and the 1 KB the SM keeps
    // per CTA
    const int per_cta = dev.smem_per_sm / (Mpad == 8 ? 2 : 1) - 1024 - moe_static_smem(kern);
    int tpw = 1;
    if (tiles == 8)
        while (tpw < 4 && ((a.N + tiles * 16 * tpw - 1) / (tiles * 16 * tpw)) * dmax * nz > 2 * dev.sms &&
               moe_smem_bytes(Mpad, nblk, G, tiles, tpw * 2, 2) <= per_cta)
            tpw *= 2;
    const int rows = tiles * 16 * tpw;
    int ns = 2;
    while (ns < kMaxStages && moe_smem_bytes(Mpad, nblk, G, tiles, tpw, ns + 1) <= per_cta &&
           moe_smem_bytes(Mpad, nblk, G, tiles, tpw, ns + 1) <= dev.max_smem_optin)
        ++ns;
    k.stages = ns;
    k.tpw = tpw;
    k.early = a.early;
    k.chunk_count = a.chunk_count;
    k.route_w = a.route_w;
    k.y_routed = a.y_routed;
    k.zero_count = a.zero_count;
    k.zero_n = a.zero_n;
    const int smem = moe_smem_bytes(Mpad, nblk, G, tiles, tpw, ns);
    if (smem > dev.max_smem_optin) return cudaErrorInvalidValue;
    CUtensorMap maps[2];
    for (int b = 0; b < 2; ++b) {
        const MoeBank& bk = k.bank[b];
        if (!encode_weight_map(&maps[b], bk.wq, a.E * a.N, a.K, kBoxRows)) return cudaErrorInvalidValue;
    }
    cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((a.N + rows - 1) / rows, dmax, nz);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, k, maps[0], maps[1]);
    if (e != cudaSuccess) return e;
    e = cudaGetLastError();
    if (e != cudaSuccess || !a.route_w || a.chunk_count) return e;  // routed sum done in-launch
    const int total = a.M * a.N;
    int blocks = (total + 255) / 256;
    if (blocks > 4 * dev.sms) blocks = 4 * dev.sms;
    k_moe_route_sum<<<blocks, 256, 0, s>>>(a.ws, a.route_w, a.ids, a.y_routed, a.M, a.topk, a.E,
                                          a.N);
    return cudaGetLastError();
}

}  // namespace w4a16
