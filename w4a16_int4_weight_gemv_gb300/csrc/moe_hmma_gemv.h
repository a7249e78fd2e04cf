// The down launch of the fp16 warp-MMA expert FFN (moe_hmma.cu) on its own:
// an expert-indexed GEMV of M*topk <= 32 slots, x a row per token or per
// slot, routed sums or per-slot outputs, 16-row output tiles (N % 16 == 0),
// g == 128, INT4 or INT3 expert banks.
#pragma once

#include "launch.h"

namespace w4a16 {

struct MoeHmmaGemvArgs {
    const uint16_t* x;     // [M][K], or [M][topk][K] with x_per_slot
    int x_per_slot;
    const int32_t* ids;    // [M][topk]
    const float* route_w;  // [M][topk]: y [M][N] routed sums; null: y [M*topk][N] per slot
    const uint32_t* wq;    // [E][N][K/8] (INT4) or [E][N][3K/32] (INT3)
    const uint16_t* scale; // [E][N][K/128]
    const uint8_t* zero;   // [E][N][K/128]
    uint16_t* y;
    int M, topk, E;
    int64_t N, K;
    uint32_t* err;
    int bits;  // 4 or 3
};
bool moe_hmma_gemv_supports(int M, int topk, int64_t N, int64_t K, int64_t g);
bool moe_hmma_gemv_fits(const DeviceInfo& dev, int M, int topk, int E, int64_t N, int64_t K, int bits,
                        int x_per_slot, int routed);
cudaError_t launch_moe_hmma_gemv(const MoeHmmaGemvArgs& a, const DeviceInfo& dev, cudaStream_t s);

}  // namespace w4a16
