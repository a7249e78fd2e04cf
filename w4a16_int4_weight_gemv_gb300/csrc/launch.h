// Host-side launcher interface between the C-ABI layer (api.cu) and the
// kernel translation units.  Internal to the library.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>  // CUtensorMap
#include <cuda_runtime.h>

namespace w4a16 {

// Boxes of the packed-weight tensor maps: 32 words (128 bytes, 256 k) x
// box_rows rows, 128-byte swizzle.
constexpr unsigned kWeightBoxWords = 32;

// Tensor map of a packed weight matrix [N][K/8] words (host; false on failure).
bool encode_weight_map(CUtensorMap* map, const void* wq, int N, int K, unsigned box_rows);

struct GemvArgs {
    const uint16_t* x;
    const uint32_t* wq;
    const uint16_t* scale;
    const uint8_t* zero;
    void* y;
    int out_f32;
    int M;
    int N;
    int K;
    int g;
    uint32_t* err;
    int weights_static;  // wq/scale/zero may be read before the preceding grid completes
    int swiglu_out;      // rows are 8-row gate/up blocks; y is bf16(silu(gate) * up) [M][N/2]
};

struct GemvPlan {
    int kernel_id;  // 1 = CUDA-core kernel, 2 = warp-MMA kernel, 3 = tensor-core (tcgen05) kernel,
                    // 4 = fp16 warp-MMA kernel with a producer warp
    int ctas;
    int threads;
    int k_split;     // cluster size along K (1 = no split)
    int smem_bytes;  // dynamic shared memory per CTA
    int units_per_cta;  // 32-chunk spans (kernel 1) or 128-k blocks (kernel 2) per CTA
    int tiles_per_cluster;  // upper bound of tiles one tile group processes
    int wpt;                // warps sharing one tile (K split inside the CTA)
    int stages;             // shared-memory stages per warp
    int tile_rows;          // rows per warp tile (CUDA-core kernel)
    int nclusters;          // kernel 4: clusters (tile ranges)
    int max_tiles;          // kernel 4: most tiles one cluster owns
};

struct DeviceInfo {
    int sms;
    int max_smem_optin;  // per CTA
    int smem_per_sm;     // per SM
};

// Choose the K split of a GEMV launch: total factor f = wpt * S (wpt warps of
// a CTA share a tile, S CTAs of a cluster share it), minimising the critical
// path -- tiles per warp group times K units per warp -- at full residency,
// then the busiest CTA's work (tiles per CTA times K units of its slice).
// max_clusters(S, smem) is how many clusters of S CTAs with that much shared
// memory the device can hold at once (clusters are co-scheduled inside a GPC,
// so it can be less than SMs / S); the persistent grid never exceeds it.
struct SplitChoice {
    int wpt, S, ctas, tiles_per_group, units_per_cta, smem_bytes;
};
// split_cost_q: what a split's per-tile partial-sum reduction costs, in
// quarters of a K unit (0: negligible next to a unit).
template <class SmemFn, class ClusterFn>
SplitChoice choose_split(const DeviceInfo& dev, int ntiles, int units_all, int warps_per_cta,
                         int max_ctas_per_sm, int forced_f, int split_cost_q, SmemFn smem_fn,
                         ClusterFn max_clusters) {
    SplitChoice best{};
    long best_cost = -1, best_work = 0;
    for (int f = 1; f <= 32; f *= 2) {
        if (forced_f > 0 && f != forced_f) continue;
        if (forced_f == 0 && f > units_all) break;
        // largest in-CTA share first: on equal cost the fewest CTAs per cluster
        // (wpt runs over the powers of two <= min(f, warps per CTA))
        int wpt0 = 1;
        while (wpt0 * 2 <= f && wpt0 * 2 <= warps_per_cta) wpt0 *= 2;
        for (int wpt = wpt0; wpt >= 1; wpt /= 2) {
            const int S = f / wpt;
            if (S > 8 || wpt * S != f || warps_per_cta % wpt) continue;
            const int upc = (units_all + S - 1) / S;
            const int tg = warps_per_cta / wpt;
            // residency with tiles_per_group unknown: size with one tile first
            int smem = smem_fn(upc, tg, wpt, 1, S);
            if (smem > dev.max_smem_optin) continue;
            int per_sm = dev.smem_per_sm / (smem + 1024);
            if (per_sm > max_ctas_per_sm) per_sm = max_ctas_per_sm;
            if (per_sm < 1) continue;
            int clusters = (per_sm * dev.sms) / S;
            if (S > 1) {
                const int mc = max_clusters(S, smem);
                if (mc < 1) continue;
                if (clusters > mc) clusters = mc;
            }
            // tiles are dealt round-robin over the clusters, so every cluster
            // up to one per tile does useful work
            if (clusters > ntiles) clusters = ntiles;
            if (clusters < 1) clusters = 1;
            const int tpg = (ntiles + clusters * tg - 1) / (clusters * tg);
            smem = smem_fn(upc, tg, wpt, tpg, S);
            if (smem > dev.max_smem_optin) continue;
            // first the longest warp's steps (plus its tiles' reductions when
            // the tiles are split), then the busiest CTA's steps; in quarter units
            const long cost = static_cast<long>(tpg) *
                              (4L * ((upc + wpt - 1) / wpt) + (f > 1 ? split_cost_q : 0));
            const long cta_work = static_cast<long>((ntiles + clusters - 1) / clusters) * upc;
            if (best_cost < 0 || cost < best_cost || (cost == best_cost && cta_work < best_work)) {
                best_cost = cost;
                best_work = cta_work;
                best = SplitChoice{wpt, S, clusters * S, tpg, upc, smem};
            }
        }
    }
    return best;
}

// ---------------------------------------------------------------------------
// fp16 warp-MMA GEMV (kernel 4): 1..16 tokens, g == 128, K % 512 == 0.
// A unit is one 16-row tile x 512 k: 16 rows of 256 packed bytes (16-byte
// chunks XOR-swizzled by row), plus the tile's 16 x 4 zero points and 16 x 4
// scales.  Every warp streams its own units through its own ring of
// `depth` stages (cp.async); WPT warps of a CTA may share a tile (K steps
// dealt round-robin, partials handed to part 0 through shared memory), and
// K may be split over the S CTAs of a cluster (S | K/512).
// ---------------------------------------------------------------------------
// warps per CTA: 8 (two CTAs per SM, so the next launch's CTA can be
// resident beside this one) or 16 (one CTA per SM, twice the warps to hide
// the arithmetic's latencies on long runs)
constexpr int kHmmaWarpsPaired = 8;
constexpr int kHmmaWarpsWide = 16;
constexpr int kHmmaRowPitch = 256;                   // a row's 256 bytes, chunks XOR-swizzled
constexpr int kHmmaUnitBytes = 16 * kHmmaRowPitch;   // 4096
constexpr int kHmmaUnitSZ = 192;   // zero points 16 x 4 bytes, then scales 16 x 8 bytes
constexpr int kHmmaStage = kHmmaUnitBytes + kHmmaUnitSZ;
constexpr int kHmmaMaxDepth = 6;

struct HmmaLayout {
    int ring, bfrag, csum, red, bars, cpart, total;
};
// Byte offsets inside the CTA's shared memory (from a 128-aligned base; the
// total includes the alignment slack) for `warps` warps per CTA, M tokens
// (the count the B fragments are stored for: 1, 2, 4, 8 or 16 -- 16 tokens
// are two 8-column MMA tiles, which double the partials), `steps` 512-k
// steps per K slice, S CTAs per cluster, at most max_tiles tiles per
// cluster, `depth` stages per warp.
__host__ __device__ inline HmmaLayout hmma_layout(int warps, int M, int steps, int S,
                                                  int max_tiles, int depth) {
    const int nt = M > 8 ? 2 : 1;            // 8-token MMA tiles
    const int pairs = M > 8 ? M / 2 : 4;     // token pairs per block in the sums
    HmmaLayout L;
    int off = 0;
    L.ring = off;  // [warp][depth] stages
    off += warps * depth * kHmmaStage;
    L.bfrag = off;  // activation fragments: [block][piece][token][lane % 4] x 16 bytes
    off += steps * 4 * 4 * M * 4 * 16;
    L.csum = off;  // per block and token pair: {c1[2i], c1[2i+1], c2[2i], c2[2i+1]},
    off += steps * 4 * pairs * 32;  // then the block's 2^-shift of tokens 2i, 2i + 1
    L.red = off;  // in-CTA K split: [tile][2][warp][lane] float4 partials
    off += nt * 2 * warps * 32 * 16;
    L.bars = off;  // their mbarriers: [tile group][buffer] {full, empty}
    off += warps * 2 * 2 * 8;
    L.cpart = off;  // K split over the cluster: [tile][tile][rank][lane] float4 pushed to the owner
    off += (S > 1) ? nt * max_tiles * S * 32 * 16 : 0;
    L.total = off + 128;
    return L;
}

struct HmmaChoice {
    int warps, S, nclusters, steps_per_rank, max_tiles, wpt, depth, smem_bytes, per_sm;
};
// Launch shape of kernel 4 with W warps per CTA: the K split S over a
// cluster (a power of two dividing K/512; forced_S > 0 forces it) and WPT
// warps per tile inside the CTA, minimising a cost -- the longest warp's
// units (tiles of its group x K steps of its part) plus what the splits add
// -- then preferring two CTAs per SM (so the next launch's CTA can be
// resident beside this one: a warp with at most 8 units needs only two
// stages to qualify, a longer one three), then the smallest S and WPT; then
// as many stages per warp as fit that residency.
// max_clusters(S, smem) is how many clusters of S CTAs the device holds at
// once.  nclusters == 0: no plan.
// pair_only: consider only shapes with two CTAs per SM.
template <class ClusterFn>
HmmaChoice plan_hmma_split(const DeviceInfo& dev, int W, int M, int N, int K, int forced_S,
                           bool pair_only, ClusterFn max_clusters, int max_sps = 0) {
    HmmaChoice best{};
    long best_t = -1;
    const int ntiles = (N + 15) / 16;
    const int nsteps = K / 512;
    const int half = dev.smem_per_sm / 2 - 1024;
    for (int S = 1; S <= 8; S *= 2) {
        if (forced_S > 0 && S != forced_S) continue;
        if (nsteps % S != 0) continue;
        const int sps = nsteps / S;
        if (max_sps > 0 && sps > max_sps) continue;
        int cap = dev.sms / S;
        const int need_min = hmma_layout(W, M, sps, S, (ntiles + cap - 1) / cap, 2).total;
        if (need_min > dev.max_smem_optin) continue;
        if (S > 1) {
            const int mc = max_clusters(S, need_min <= half ? half : dev.max_smem_optin);
            if (mc < 1) continue;
            if (cap > mc) cap = mc;
        }
        const int ncl = cap < ntiles ? cap : ntiles;
        const int max_tiles = (ntiles + ncl - 1) / ncl;
        for (int wpt = 1; wpt <= W; wpt *= 2) {
            const int ng = W / wpt;
            const int tpg = (max_tiles + ng - 1) / ng;  // tiles of the busiest group
            const int units = tpg * ((sps + wpt - 1) / wpt);
            // cost in eighths of a unit: the busiest warp's units, plus one
            // eighth per partial part 0 of a split tile adds, plus a quarter
            // per tile and extra rank of a cluster split (DSMEM push and
            // cluster barrier) -- fitted to GB300 timings of one token
            const long t = 8L * units + static_cast<long>(tpg) * (wpt - 1) +
                           2L * (S - 1) * max_tiles;
            // short runs (a few units per warp) gain most from the next
            // launch's CTA being resident early: two stages per warp there;
            // long runs want three to keep the stream deep
            const int want = units <= 8 ? 2 : 3;
            // 16 tokens: the kernel takes more than half the register file
            const int per_sm = M <= 8 && hmma_layout(W, M, sps, S, max_tiles, want).total <= half ? 2 : 1;
            if (pair_only && per_sm != 2) continue;
            // clusters of four or more CTAs that could pair up on an SM were
            // placed unevenly (measured 30-60 % slower than S <= 2)
            if (per_sm == 2 && S > 2 && forced_S == 0) continue;
            if (best_t >= 0 && (t > best_t || (t == best_t && per_sm <= best.per_sm))) continue;
            const int budget = per_sm == 2 ? half : dev.max_smem_optin;
            int depth = 2;
            while (depth < kHmmaMaxDepth && depth < units &&
                   hmma_layout(W, M, sps, S, max_tiles, depth + 1).total <= budget)
                ++depth;
            const int smem = hmma_layout(W, M, sps, S, max_tiles, depth).total;
            if (smem > dev.max_smem_optin) continue;
            best_t = t;
            best = HmmaChoice{W, S, ncl, sps, max_tiles, wpt, depth, smem, per_sm};
        }
    }
    return best;
}

// The best 8-warp plan with two CTAs on an SM, where there is one (short
// runs: the next launch's CTA is resident early); otherwise the 16-warp
// plan, which has twice the warps of an SM working (the register file holds
// 16 warps of this kernel, so a 16-warp CTA is alone on its SM).  Measured on GB300 for
// one token: 8 warps is ahead by 2-5 % on 4096 x 4096 .. 14336 x 4096 and
// 4096 x 14336, 16 warps by 4-14 % from 28672 x 4096 up to the vocabulary
// projection.
template <class ClusterFn8, class ClusterFn16>
HmmaChoice choose_hmma_plan_sps(const DeviceInfo& dev, int M, int N, int K, int forced_S,
                                ClusterFn8 max_clusters8, ClusterFn16 max_clusters16, int max_sps) {
    const HmmaChoice paired =
        plan_hmma_split(dev, kHmmaWarpsPaired, M, N, K, forced_S, true, max_clusters8, max_sps);
    if (paired.nclusters > 0) return paired;
    const HmmaChoice wide =
        plan_hmma_split(dev, kHmmaWarpsWide, M, N, K, forced_S, false, max_clusters16, max_sps);
    if (wide.nclusters > 0) return wide;
    return plan_hmma_split(dev, kHmmaWarpsPaired, M, N, K, forced_S, false, max_clusters8, max_sps);
}
// 9..16 tokens prefer K slices of at most 2048 k (measured on GB300, 12 and
// 16 tokens: 14336 x 4096 and 28672 x 4096 5-12 % faster than the bf16
// warp-MMA kernel with clusters of two, 8192 x 8192 14-40 % with clusters of
// four; with an unsplit 4096-k slice 10 % slower than it); any slice that
// fits otherwise
template <class ClusterFn8, class ClusterFn16>
HmmaChoice choose_hmma_plan(const DeviceInfo& dev, int M, int N, int K, int forced_S,
                            ClusterFn8 max_clusters8, ClusterFn16 max_clusters16) {
    if (M > 8 && forced_S == 0) {
        const HmmaChoice c = choose_hmma_plan_sps(dev, M, N, K, 0, max_clusters8, max_clusters16, 4);
        if (c.nclusters > 0) return c;
    }
    return choose_hmma_plan_sps(dev, M, N, K, forced_S, max_clusters8, max_clusters16, 0);
}

// Lets `kernel` run with `bytes` of dynamic shared memory on the current
// device.  The limit persists per function and device, so it is raised only
// when a launch needs more than every earlier one did (a host-side table
// spares the driver call -- about a microsecond -- on every launch).
cudaError_t ensure_dynamic_smem(const void* kernel, int bytes);

// Number of clusters of S CTAs (threads each, smem bytes of dynamic shared
// memory) of `kernel` the current device can run at once; cached.
int max_active_clusters(const void* kernel, int threads, int smem, int S);

// Launch-shape choices (host arithmetic plus cached occupancy queries).
GemvPlan plan_gemv_simt(const DeviceInfo& dev, int M, int N, int K, int g, int k_split_req);
GemvPlan plan_gemv_mma(const DeviceInfo& dev, int M, int N, int K, int g, int k_split_req);
GemvPlan plan_gemv_tc(const DeviceInfo& dev, int M, int N, int K, int g, int k_split_req);
GemvPlan plan_gemv_hmma(const DeviceInfo& dev, int M, int N, int K, int g, int k_split_req);
// True when kernel 4 serves this shape (1..16 tokens, g == 128, K % 512 == 0).
inline bool hmma_supports(int M, int K, int g) { return M >= 1 && M <= 16 && g == 128 && K % 512 == 0; }

cudaError_t launch_gemv_simt(const GemvArgs& a, const GemvPlan& p, cudaStream_t s);
cudaError_t launch_gemv_mma(const GemvArgs& a, const GemvPlan& p, cudaStream_t s);
cudaError_t launch_gemv_tc(const GemvArgs& a, const GemvPlan& p, cudaStream_t s);
cudaError_t launch_gemv_hmma(const GemvArgs& a, const GemvPlan& p, cudaStream_t s);

// Routed SwiGLU expert FFN on the fp16 warp-MMA path (moe_hmma.cu): 1..8
// tokens, M * topk <= 32 slots, g == 128, H and F multiples of 128.  h is
// the bf16 [M*topk][F] intermediate.  bits: 4 (INT4 banks, K/8 words per
// row) or 3 (INT3 banks, 3K/32 words per row).
constexpr int kMoeHmmaMaxSlots = 32;
struct MoeHmmaArgs {
    const uint16_t* x;
    const int32_t* ids;
    const float* route_w;
    const uint32_t* gate_wq;
    const uint16_t* gate_scale;
    const uint8_t* gate_zero;
    const uint32_t* up_wq;
    const uint16_t* up_scale;
    const uint8_t* up_zero;
    const uint32_t* down_wq;
    const uint16_t* down_scale;
    const uint8_t* down_zero;
    uint16_t* h;
    uint16_t* y;
    int M, topk, E;
    int64_t H, F;
    uint32_t* err;
    int bits;
};
bool moe_hmma_supports(int M, int topk, int64_t H, int64_t F, int64_t g);
bool moe_hmma_fits(const DeviceInfo& dev, int M, int topk, int E, int64_t H, int64_t F, int bits);
cudaError_t launch_moe_hmma(const MoeHmmaArgs& a, const DeviceInfo& dev, cudaStream_t s);

// One stacked expert bank: wq [E][N][K/8], scale and zero [E][N][K/g], and
// its bf16 per-slot output [M*topk][N] (used when there is no routed sum).
struct MoeBank {
    const uint32_t* wq;
    const uint16_t* scale;
    const uint8_t* zero;
    uint16_t* y;
};
struct MoeArgs {
    const uint16_t* x;        // [M][K], or [M][topk][K] with x_per_slot
    int x_per_slot;
    const uint16_t* sw_gate;  // non-null: activations bf16(silu(gate) * up), [M*topk][K]
    const uint16_t* sw_up;
    const int32_t* ids;
    const float* route_w;     // non-null: routed sum into y_routed through ws
    MoeBank bank[2];
    int nbanks;               // 1, or 2 banks of one shape against the same activations
    int early;                // inputs other than the activations may be read before the
                              // grid dependency wait (the predecessor is this chain's own)
    uint16_t* y_routed;       // bf16 [M][N]
    float* ws;                // fp32 [M*topk][N] partials of the routed sum
    unsigned* chunk_count;    // non-null: the routed sum is formed inside the launch, per
                              // 64/128-row chunk, by its last CTA (counters zero on entry)
    unsigned* zero_count;     // counters this launch zeroes first (for the next launch)
    int zero_n;
    int M;
    int topk;
    int E;
    int N;
    int K;
    int g;
    uint32_t* err;
};
// Dynamic shared memory the expert kernel needs at least (two stages).
int moe_smem_need(int M, int K, int g);
// Number of row chunks (CTAs along x) of an expert launch for N rows.
int moe_row_chunks(int N);
cudaError_t launch_moe(const MoeArgs& a, const DeviceInfo& dev, cudaStream_t s);

cudaError_t launch_pack(const uint8_t* codes, uint32_t* wq, int64_t N, int64_t K, int sms,
                        cudaStream_t s);
cudaError_t launch_dequant(const uint32_t* wq, const uint16_t* scale, const uint8_t* zero,
                           void* w, int out_f32, int64_t N, int64_t K, int64_t g, int sms,
                           cudaStream_t s);
cudaError_t launch_swiglu(const uint16_t* gate, const uint16_t* up, int64_t ld_in, uint16_t* h,
                          int64_t ld_out, int64_t rows, int64_t N, int sms, cudaStream_t s);
// INT3 codes <-> words (K % 128 == 0; 3K/32 words per row) and dequant
cudaError_t launch_pack3(const uint8_t* codes, uint32_t* wq3, int64_t N, int64_t K, int sms,
                         cudaStream_t s);
cudaError_t launch_dequant3(const uint32_t* wq3, const uint16_t* scale, const uint8_t* zero,
                            void* w, int out_f32, int64_t N, int64_t K, int64_t g, int sms,
                            cudaStream_t s);

}  // namespace w4a16
