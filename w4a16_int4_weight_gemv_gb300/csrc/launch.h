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
};

struct GemvPlan {
    int kernel_id;  // 1 = CUDA-core kernel, 2 = warp-MMA kernel, 3 = tensor-core (tcgen05) kernel
    int ctas;
    int threads;
    int k_split;     // cluster size along K (1 = no split)
    int smem_bytes;  // dynamic shared memory per CTA
    int units_per_cta;  // 32-chunk spans (kernel 1) or 128-k blocks (kernel 2) per CTA
    int tiles_per_cluster;  // upper bound of tiles one tile group processes
    int wpt;                // warps sharing one tile (K split inside the CTA)
    int stages;             // shared-memory stages per warp
    int tile_rows;          // rows per warp tile (CUDA-core kernel)
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

cudaError_t launch_gemv_simt(const GemvArgs& a, const GemvPlan& p, cudaStream_t s);
cudaError_t launch_gemv_mma(const GemvArgs& a, const GemvPlan& p, cudaStream_t s);
cudaError_t launch_gemv_tc(const GemvArgs& a, const GemvPlan& p, cudaStream_t s);

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

}  // namespace w4a16
