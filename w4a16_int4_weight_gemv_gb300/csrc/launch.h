// Host-side launcher interface between the C-ABI layer (api.cu) and the
// kernel translation units.  Internal to the library.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace w4a16 {

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
};

struct GemvPlan {
    int kernel_id;  // 1 = CUDA-core M=1 kernel, 2 = warp-MMA kernel
    int ctas;
    int threads;
    int k_split;     // cluster size along K (1 = no split)
    int smem_bytes;  // dynamic shared memory per CTA
    int units_per_cta;  // 32-chunk spans (kernel 1) or 128-k blocks (kernel 2) per CTA
    int tiles_per_cluster;
};

struct DeviceInfo {
    int sms;
    int max_smem_optin;
};

// Launch-shape choices (pure host arithmetic, no CUDA calls).
GemvPlan plan_gemv_simt(const DeviceInfo& dev, int N, int K, int k_split_req);
GemvPlan plan_gemv_mma(const DeviceInfo& dev, int M, int N, int K, int k_split_req);

cudaError_t launch_gemv_simt(const GemvArgs& a, const GemvPlan& p, cudaStream_t s);
cudaError_t launch_gemv_mma(const GemvArgs& a, const GemvPlan& p, cudaStream_t s);

struct MoeArgs {
    const uint16_t* x;
    int x_per_slot;
    const int32_t* ids;
    const float* route_w;
    const uint32_t* wq;
    const uint16_t* scale;
    const uint8_t* zero;
    uint16_t* y;
    float* ws;  // fp32 [M][topk][N] partials when route_w != nullptr
    int M;
    int topk;
    int E;
    int N;
    int K;
    int g;
    uint32_t* err;
};
cudaError_t launch_moe(const MoeArgs& a, const DeviceInfo& dev, cudaStream_t s);

cudaError_t launch_pack(const uint8_t* codes, uint32_t* wq, int64_t N, int64_t K, int sms,
                        cudaStream_t s);
cudaError_t launch_dequant(const uint32_t* wq, const uint16_t* scale, const uint8_t* zero,
                           void* w, int out_f32, int64_t N, int64_t K, int64_t g, int sms,
                           cudaStream_t s);
cudaError_t launch_swiglu(const uint16_t* gate, const uint16_t* up, int64_t ld_in, uint16_t* h,
                          int64_t ld_out, int64_t rows, int64_t N, int sms, cudaStream_t s);

}  // namespace w4a16
