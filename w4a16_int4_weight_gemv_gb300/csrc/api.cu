// C ABI of the W4A16 library: argument validation, launch planning and
// dispatch.  Declarations and the contract of each call are in w4a16.h.
//
// Every entry point validates all arguments before it enqueues anything, so
// an invalid call has no effect on the device.  The library allocates no
// device memory: the only device state it owns is one 32-bit error word per
// device (a __device__ variable), where kernels record data-dependent
// problems instead of trapping.
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda_runtime.h>

#include "launch.h"
#include "moe_hmma_gemv.h"
#include "w4a16.h"

namespace w4a16 {
namespace {

__device__ uint32_t g_error_word;

constexpr int kMaxDevices = 64;

struct DeviceCache {
    bool ready = false;
    DeviceInfo info{};
    uint32_t* err = nullptr;
};

std::mutex g_mu;
DeviceCache g_dev[kMaxDevices];

// Properties and the error word's address for the current device (once per device).
w4a16_status current_device(DeviceCache** out) {
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return W4A16_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceCache& c = g_dev[d];
    if (!c.ready) {
        int sms = 0, smem = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, d) != cudaSuccess)
            return W4A16_ERR_CUDA;
        if (cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, d) !=
            cudaSuccess)
            return W4A16_ERR_CUDA;
        int smem_sm = 0;
        if (cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, d) !=
            cudaSuccess)
            return W4A16_ERR_CUDA;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return W4A16_ERR_CUDA;
        c.info.sms = sms;
        c.info.max_smem_optin = smem;
        c.info.smem_per_sm = smem_sm;
        c.err = static_cast<uint32_t*>(p);
        c.ready = true;
    }
    *out = &c;
    return W4A16_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

w4a16_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return W4A16_OK;
    (void)cudaGetLastError();  // clear a sticky launch-configuration error
    return W4A16_ERR_CUDA;
}

// Shape rules shared by the GEMV entry points.
w4a16_status check_gemv_shape(int M, int64_t N, int64_t K, int64_t g) {
    if (M < 1 || N < 1 || K < 32 || g < 32) return W4A16_ERR_SHAPE;
    if (K % 32 != 0 || g % 32 != 0 || K % g != 0) return W4A16_ERR_SHAPE;
    if (M > 16) return W4A16_ERR_UNSUPPORTED;
    if (K > 65536) return W4A16_ERR_UNSUPPORTED;
    if (N > (int64_t(1) << 31) / (K / 8) - 1) return W4A16_ERR_UNSUPPORTED;
    return W4A16_OK;
}

w4a16_status make_plan(int M, int64_t N, int64_t K, int64_t g, int kernel_id, int k_split,
                       GemvPlan* plan, DeviceCache** dev) {
    // default: the fp16 warp-MMA kernel where it applies (g == 128,
    // K % 512 == 0) -- for one or two tokens always, for three or four
    // tokens on matrices of at least 2^24 weights, for 3..16 tokens on
    // matrices of at least 2^25 weights; otherwise the bf16 warp-MMA kernel
    // where the groups are multiples of 128 k; the CUDA-core kernel for one
    // or two tokens with finer groups.  (Measured on GB300: kernel 4 ahead
    // at one and two tokens by 0-37 % on the MLP, square and 8192 x 8192
    // shapes; at 3..8 tokens ahead by 5-32 % from 14336 x 4096 up, and behind
    // by up to 20 % on 4096 x 4096 and smaller matrices; at 9..16 tokens
    // (two MMA tiles, K slices of at most 2048 k) ahead by 5-40 % from
    // 14336 x 4096 up where a plan exists, falling back to kernel 2 where
    // none does, e.g. 4096 x 14336.  Between 2^24 and 2^25 weights, over
    // nine shapes from 4096 x 4096 to 8192 x 2048: at three and four tokens
    // 12 % ahead on average, at most 2 % behind; at 8 and 16 tokens from
    // 46 % ahead to 23 % behind, so kernel 2 stays there.)
    const int requested = kernel_id;
    const bool automatic = kernel_id == 0;
    if (automatic) {
        const bool k4 = hmma_supports(M, static_cast<int>(K), static_cast<int>(g)) &&
                        (M <= 2 || N * K >= (int64_t(1) << 25) ||
                         (M <= 4 && N * K >= (int64_t(1) << 24)));
        kernel_id = k4 ? 4 : (g % 128 == 0) ? 2 : 1;
    }
    if (kernel_id == 1 && M > 2) return W4A16_ERR_UNSUPPORTED;
    if ((kernel_id == 2 || kernel_id == 3) && g % 128 != 0) return W4A16_ERR_UNSUPPORTED;
    if (kernel_id == 4 && !hmma_supports(M, static_cast<int>(K), static_cast<int>(g)))
        return W4A16_ERR_UNSUPPORTED;
    if (kernel_id < 1 || kernel_id > 4) return W4A16_ERR_UNSUPPORTED;
    if ((kernel_id == 3 || kernel_id == 4) && k_split > 8) return W4A16_ERR_UNSUPPORTED;
    if (k_split < 0 || k_split > 32 || (k_split & (k_split - 1))) return W4A16_ERR_UNSUPPORTED;
    w4a16_status st = current_device(dev);
    if (st != W4A16_OK) return st;
    const int n = static_cast<int>(N), k = static_cast<int>(K);
    const int gg = static_cast<int>(g);
    // plans depend only on the shape and the device: computed once each
    struct Entry {
        int device, kernel_id, M, N, K, g, k_split;
        GemvPlan plan;
    };
    static std::mutex mu;
    static Entry cache[256];
    static int used = 0, next = 0;
    const int d = static_cast<int>(*dev - g_dev);
    {
        std::lock_guard<std::mutex> lock(mu);
        for (int i = 0; i < used; ++i) {
            const Entry& c = cache[i];
            if (c.device == d && c.kernel_id == requested && c.M == M && c.N == n && c.K == k &&
                c.g == gg && c.k_split == k_split) {
                *plan = c.plan;
                return W4A16_OK;
            }
        }
    }
    *plan = (kernel_id == 1)   ? plan_gemv_simt((*dev)->info, M, n, k, gg, k_split)
            : (kernel_id == 2) ? plan_gemv_mma((*dev)->info, M, n, k, gg, k_split)
            : (kernel_id == 3) ? plan_gemv_tc((*dev)->info, M, n, k, gg, k_split)
                               : plan_gemv_hmma((*dev)->info, M, n, k, gg, k_split);
    if (automatic && kernel_id == 4 && plan->ctas < 1) {
        // no fp16-MMA plan for this shape (activations too large for shared memory)
        kernel_id = 2;
        *plan = plan_gemv_mma((*dev)->info, M, n, k, gg, k_split);
    }
    if (plan->ctas < 1 || plan->smem_bytes > (*dev)->info.max_smem_optin)
        return W4A16_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(mu);
    Entry& slot = (used < 256) ? cache[used++] : cache[next++ & 255];
    slot = Entry{d, requested, M, n, k, gg, k_split, *plan};
    return W4A16_OK;
}

w4a16_status gemv_impl(const uint16_t* x, const uint32_t* wq, const uint16_t* scale,
                       const uint8_t* zero, void* y, w4a16_out_dtype out_dtype, int M, int64_t N,
                       int64_t K, int64_t g, int kernel_id, int k_split, unsigned flags,
                       void* stream) {
    if (flags & ~static_cast<unsigned>(W4A16_FLAG_WEIGHTS_STATIC | W4A16_FLAG_SWIGLU_OUTPUT |
                                       W4A16_FLAG_NO_CLUSTER))
        return W4A16_ERR_UNSUPPORTED;
    if (!x || !wq || !scale || !zero || !y) return W4A16_ERR_NULL;
    w4a16_status st = check_gemv_shape(M, N, K, g);
    if (st != W4A16_OK) return st;
    if (out_dtype != W4A16_OUT_BF16 && out_dtype != W4A16_OUT_F32) return W4A16_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(wq) || !aligned16(scale) || !aligned16(zero) || !aligned16(y))
        return W4A16_ERR_ALIGN;
    GemvPlan plan{};
    DeviceCache* dev = nullptr;
    st = make_plan(M, N, K, g, kernel_id, k_split, &plan, &dev);
    if (st != W4A16_OK) return st;
    if ((flags & W4A16_FLAG_NO_CLUSTER) && plan.k_split > 1 && k_split == 0 && plan.kernel_id != 3) {
        // the same kernel with its K split kept inside the CTA (kernel 4:
        // no cluster, warps per tile chosen anew; kernels 1 and 2: the
        // plan's warps per tile), where such a plan exists
        GemvPlan inner{};
        if (make_plan(M, N, K, g, plan.kernel_id, plan.kernel_id == 4 ? 1 : plan.wpt, &inner, &dev) ==
                W4A16_OK &&
            inner.k_split == 1)
            plan = inner;
    }
    const int swiglu = (flags & W4A16_FLAG_SWIGLU_OUTPUT) ? 1 : 0;
    // the fused SwiGLU lives in the epilogues of the two warp-MMA kernels,
    // whose lanes hold rows r and r + 8 of a tile (a gate and its up row)
    if (swiglu && ((plan.kernel_id != 2 && plan.kernel_id != 4) || N % 16 != 0 ||
                   out_dtype != W4A16_OUT_BF16))
        return W4A16_ERR_UNSUPPORTED;
    GemvArgs a{x, wq, scale, zero, y, out_dtype == W4A16_OUT_F32 ? 1 : 0, M,
               static_cast<int>(N), static_cast<int>(K), static_cast<int>(g), dev->err,
               (flags & W4A16_FLAG_WEIGHTS_STATIC) ? 1 : 0, swiglu};
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return from_cuda(plan.kernel_id == 1   ? launch_gemv_simt(a, plan, s)
                     : plan.kernel_id == 2 ? launch_gemv_mma(a, plan, s)
                     : plan.kernel_id == 3 ? launch_gemv_tc(a, plan, s)
                                           : launch_gemv_hmma(a, plan, s));
}

}  // namespace

cudaError_t ensure_dynamic_smem(const void* kernel, int bytes) {
    struct Entry {
        const void* kernel;
        int device, bytes;
    };
    static std::mutex mu;
    static Entry table[512];
    static int used = 0;
    int d = 0;
    cudaError_t e = cudaGetDevice(&d);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    Entry* hit = nullptr;
    for (int i = 0; i < used && !hit; ++i)
        if (table[i].kernel == kernel && table[i].device == d) hit = &table[i];
    if (hit && hit->bytes >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    if (hit) hit->bytes = bytes;
    else if (used < 512) table[used++] = Entry{kernel, d, bytes};
    return cudaSuccess;
}

int max_active_clusters(const void* kernel, int threads, int smem, int S) {
    struct Entry {
        const void* kernel;
        int device, threads, smem, S, value;
    };
    static std::mutex mu;
    static Entry cache[256];
    static int used = 0;
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess) return 0;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i) {
        const Entry& e = cache[i];
        if (e.kernel == kernel && e.device == d && e.threads == threads && e.smem == smem &&
            e.S == S)
            return e.value;
    }
    int n = 0;
    if (ensure_dynamic_smem(kernel, smem) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(S * 64);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        n = 0;
    }
    if (used < 256) cache[used++] = Entry{kernel, d, threads, smem, S, n};
    return n;
}

}  // namespace w4a16

using namespace w4a16;

extern "C" {

int w4a16_abi_version(void) { return 1; }

const char* w4a16_status_string(w4a16_status status) {
    switch (status) {
        case W4A16_OK: return "ok";
        case W4A16_ERR_NULL: return "a required pointer is NULL";
        case W4A16_ERR_SHAPE: return "a size is out of range or inconsistent";
        case W4A16_ERR_ALIGN: return "a pointer is not 16-byte aligned";
        case W4A16_ERR_UNSUPPORTED: return "request outside what is implemented";
        case W4A16_ERR_WORKSPACE: return "workspace missing or too small";
        case W4A16_ERR_CUDA: return "the CUDA runtime refused a launch or query";
    }
    return "unknown status";
}

w4a16_status int4_pack(const uint8_t* codes, uint32_t* wq, int64_t N, int64_t K, void* stream) {
    if (!codes || !wq) return W4A16_ERR_NULL;
    if (N < 0 || K < 0 || K % 8 != 0) return W4A16_ERR_SHAPE;
    if (!aligned16(codes) || !aligned16(wq)) return W4A16_ERR_ALIGN;
    if (N == 0 || K == 0) return W4A16_OK;
    DeviceCache* dev = nullptr;
    w4a16_status st = current_device(&dev);
    if (st != W4A16_OK) return st;
    return from_cuda(launch_pack(codes, wq, N, K, dev->info.sms, static_cast<cudaStream_t>(stream)));
}

w4a16_status int4_dequant(const uint32_t* wq, const uint16_t* scale, const uint8_t* zero, void* w,
                          w4a16_out_dtype out_dtype, int64_t N, int64_t K, int64_t g,
                          void* stream) {
    if (!wq || !scale || !zero || !w) return W4A16_ERR_NULL;
    if (N < 0 || K < 0 || g < 32 || K % 32 != 0 || g % 32 != 0 || K % g != 0)
        return W4A16_ERR_SHAPE;
    if (out_dtype != W4A16_OUT_BF16 && out_dtype != W4A16_OUT_F32) return W4A16_ERR_UNSUPPORTED;
    if (!aligned16(wq) || !aligned16(scale) || !aligned16(zero) || !aligned16(w))
        return W4A16_ERR_ALIGN;
    if (N == 0 || K == 0) return W4A16_OK;
    DeviceCache* dev = nullptr;
    w4a16_status st = current_device(&dev);
    if (st != W4A16_OK) return st;
    return from_cuda(launch_dequant(wq, scale, zero, w, out_dtype == W4A16_OUT_F32 ? 1 : 0, N, K,
                                    g, dev->info.sms, static_cast<cudaStream_t>(stream)));
}

w4a16_status int3_pack(const uint8_t* codes, uint32_t* wq3, int64_t N, int64_t K, void* stream) {
    if (!codes || !wq3) return W4A16_ERR_NULL;
    if (N < 0 || K < 0 || K % 128 != 0) return W4A16_ERR_SHAPE;
    if (!aligned16(codes) || !aligned16(wq3)) return W4A16_ERR_ALIGN;
    if (N == 0 || K == 0) return W4A16_OK;
    DeviceCache* dev = nullptr;
    w4a16_status st = current_device(&dev);
    if (st != W4A16_OK) return st;
    return from_cuda(launch_pack3(codes, wq3, N, K, dev->info.sms, static_cast<cudaStream_t>(stream)));
}

w4a16_status int3_dequant(const uint32_t* wq3, const uint16_t* scale, const uint8_t* zero, void* w,
                          w4a16_out_dtype out_dtype, int64_t N, int64_t K, int64_t g,
                          void* stream) {
    if (!wq3 || !scale || !zero || !w) return W4A16_ERR_NULL;
    if (N < 0 || K < 0 || g < 32 || K % 128 != 0 || g % 32 != 0 || K % g != 0)
        return W4A16_ERR_SHAPE;
    if (out_dtype != W4A16_OUT_BF16 && out_dtype != W4A16_OUT_F32) return W4A16_ERR_UNSUPPORTED;
    if (!aligned16(wq3) || !aligned16(scale) || !aligned16(zero) || !aligned16(w))
        return W4A16_ERR_ALIGN;
    if (N == 0 || K == 0) return W4A16_OK;
    DeviceCache* dev = nullptr;
    w4a16_status st = current_device(&dev);
    if (st != W4A16_OK) return st;
    return from_cuda(launch_dequant3(wq3, scale, zero, w, out_dtype == W4A16_OUT_F32 ? 1 : 0, N, K,
                                     g, dev->info.sms, static_cast<cudaStream_t>(stream)));
}

size_t w4a16_gemv_workspace_bytes(int M, int64_t N, int64_t K, int64_t g) {
    (void)M;
    (void)N;
    (void)K;
    (void)g;
    return 0;
}

w4a16_status w4a16_gemv(const uint16_t* x, const uint32_t* wq, const uint16_t* scale,
                        const uint8_t* zero, void* y, w4a16_out_dtype out_dtype, int M, int64_t N,
                        int64_t K, int64_t g, void* workspace, size_t workspace_bytes,
                        void* stream) {
    (void)workspace;
    (void)workspace_bytes;
    return gemv_impl(x, wq, scale, zero, y, out_dtype, M, N, K, g, 0, 0, 0u, stream);
}

w4a16_status w4a16_gemv_ex(const uint16_t* x, const uint32_t* wq, const uint16_t* scale,
                           const uint8_t* zero, void* y, w4a16_out_dtype out_dtype, int M,
                           int64_t N, int64_t K, int64_t g, unsigned flags, void* stream) {
    return gemv_impl(x, wq, scale, zero, y, out_dtype, M, N, K, g, 0, 0, flags, stream);
}

w4a16_status w4a16_gemv_variant(const uint16_t* x, const uint32_t* wq, const uint16_t* scale,
                                const uint8_t* zero, void* y, w4a16_out_dtype out_dtype, int M,
                                int64_t N, int64_t K, int64_t g, int kernel_id, int k_split,
                                void* stream) {
    if (kernel_id < 1 || kernel_id > 4) return W4A16_ERR_UNSUPPORTED;
    return gemv_impl(x, wq, scale, zero, y, out_dtype, M, N, K, g, kernel_id, k_split, 0u,
                     stream);
}

w4a16_status w4a16_gemv_plan(int M, int64_t N, int64_t K, int64_t g, int* kernel_id, int* ctas,
                             int* threads, int* k_split, int* smem_bytes) {
    w4a16_status st = check_gemv_shape(M, N, K, g);
    if (st != W4A16_OK) return st;
    GemvPlan plan{};
    DeviceCache* dev = nullptr;
    st = make_plan(M, N, K, g, 0, 0, &plan, &dev);
    if (st != W4A16_OK) return st;
    if (kernel_id) *kernel_id = plan.kernel_id;
    if (ctas) *ctas = plan.ctas;
    if (threads) *threads = plan.threads;
    if (k_split) *k_split = plan.k_split * plan.wpt;
    if (smem_bytes) *smem_bytes = plan.smem_bytes;
    return W4A16_OK;
}

size_t w4a16_moe_workspace_bytes(int M, int topk, int64_t N, int route) {
    if (!route || M < 1 || topk < 1 || N < 1) return 0;
    return static_cast<size_t>(M) * static_cast<size_t>(topk) * static_cast<size_t>(N) *
           sizeof(float);
}

w4a16_status w4a16_moe_gemv(const uint16_t* x, int x_per_slot, const int32_t* expert_ids,
                            const float* route_w, const uint32_t* wq, const uint16_t* scale,
                            const uint8_t* zero, uint16_t* y, int M, int topk, int E, int64_t N,
                            int64_t K, int64_t g, void* workspace, size_t workspace_bytes,
                            void* stream) {
    return w4a16_moe_gemv_variant(x, x_per_slot, expert_ids, route_w, wq, scale, zero, y, M, topk,
                                  E, N, K, g, 0, workspace, workspace_bytes, stream);
}

w4a16_status w4a16_moe_gemv_variant(const uint16_t* x, int x_per_slot, const int32_t* expert_ids,
                                    const float* route_w, const uint32_t* wq, const uint16_t* scale,
                                    const uint8_t* zero, uint16_t* y, int M, int topk, int E,
                                    int64_t N, int64_t K, int64_t g, int kernel_id,
                                    void* workspace, size_t workspace_bytes, void* stream) {
    if (!x || !expert_ids || !wq || !scale || !zero || !y) return W4A16_ERR_NULL;
    if (M < 1 || topk < 1 || E < 1 || N < 1 || K < 32 || g < 32) return W4A16_ERR_SHAPE;
    if (K % 32 != 0 || g % 32 != 0 || K % g != 0) return W4A16_ERR_SHAPE;
    if (kernel_id != 0 && kernel_id != 2 && kernel_id != 4) return W4A16_ERR_UNSUPPORTED;
    if (g % 128 != 0 || M * topk > 256 || K > 65536) return W4A16_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(E) * N > (int64_t(1) << 31) / (K / 8) - 1)
        return W4A16_ERR_UNSUPPORTED;
    if (kernel_id == 4 && !moe_hmma_gemv_supports(M, topk, N, K, g)) return W4A16_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(expert_ids) || !aligned16(wq) || !aligned16(scale) ||
        !aligned16(zero) || !aligned16(y) || (route_w && !aligned16(route_w)))
        return W4A16_ERR_ALIGN;
    // the routed sum's workspace is part of the call's contract whichever
    // kernel the library picks (kernel 4 alone does without it)
    if (route_w && kernel_id != 4) {
        const size_t need = w4a16_moe_workspace_bytes(M, topk, N, 1);
        if (!workspace || workspace_bytes < need) return W4A16_ERR_WORKSPACE;
        if (!aligned16(workspace)) return W4A16_ERR_ALIGN;
    }
    DeviceCache* dev = nullptr;
    w4a16_status st = current_device(&dev);
    if (st != W4A16_OK) return st;
    // the library's choice: the fp16 warp-MMA expert kernel wherever it
    // applies (faster on every expert shape measured), else kernel 2
    const bool k4 = (kernel_id == 4 || kernel_id == 0) && moe_hmma_gemv_supports(M, topk, N, K, g) &&
                    moe_hmma_gemv_fits(dev->info, M, topk, E, N, K, 4, x_per_slot, route_w != nullptr);
    if (kernel_id == 4 && !k4) return W4A16_ERR_UNSUPPORTED;
    if (k4) {
        // routed sums in shared memory: the workspace is not used
        MoeHmmaGemvArgs a{x, x_per_slot ? 1 : 0, expert_ids, route_w, wq, scale, zero, y,
                          M, topk, E, N, K, dev->err, 4};
        return from_cuda(launch_moe_hmma_gemv(a, dev->info, static_cast<cudaStream_t>(stream)));
    }
    // the whole activation set of one expert pass must fit in shared memory
    if (moe_smem_need(M, static_cast<int>(K), static_cast<int>(g)) > dev->info.max_smem_optin)
        return W4A16_ERR_UNSUPPORTED;
    MoeArgs a{};
    a.x = x;
    a.x_per_slot = x_per_slot ? 1 : 0;
    a.ids = expert_ids;
    a.route_w = route_w;
    a.bank[0] = MoeBank{wq, scale, zero, route_w ? nullptr : y};
    a.nbanks = 1;
    a.y_routed = route_w ? y : nullptr;
    a.ws = static_cast<float*>(workspace);
    a.M = M;
    a.topk = topk;
    a.E = E;
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    a.g = static_cast<int>(g);
    a.err = dev->err;
    return from_cuda(launch_moe(a, dev->info, static_cast<cudaStream_t>(stream)));
}

namespace {
size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }
}  // namespace

size_t w4a16_moe_ffn_workspace_bytes(int M, int topk, int64_t H, int64_t F) {
    if (M < 1 || topk < 1 || H < 1 || F < 1) return 0;
    const size_t S = static_cast<size_t>(M) * static_cast<size_t>(topk);
    const size_t chunks = static_cast<size_t>((H + 63) / 64);
    return 2 * align256(S * static_cast<size_t>(F) * 2) + align256(S * static_cast<size_t>(H) * 4) +
           align256(chunks * sizeof(unsigned));
}

w4a16_status w4a16_moe_ffn(const uint16_t* x, const int32_t* expert_ids, const float* route_w,
                           const uint32_t* gate_wq, const uint16_t* gate_scale,
                           const uint8_t* gate_zero, const uint32_t* up_wq,
                           const uint16_t* up_scale, const uint8_t* up_zero,
                           const uint32_t* down_wq, const uint16_t* down_scale,
                           const uint8_t* down_zero, uint16_t* y, int M, int topk, int E,
                           int64_t H, int64_t F, int64_t g, void* workspace,
                           size_t workspace_bytes, void* stream) {
    if (!x || !expert_ids || !route_w || !gate_wq || !gate_scale || !gate_zero || !up_wq ||
        !up_scale || !up_zero || !down_wq || !down_scale || !down_zero || !y)
        return W4A16_ERR_NULL;
    if (M < 1 || topk < 1 || E < 1 || H < 32 || F < 32 || g < 32) return W4A16_ERR_SHAPE;
    if (g % 32 != 0 || H % g != 0 || F % g != 0) return W4A16_ERR_SHAPE;
    if (g % 128 != 0 || M * topk > 256 || H > 65536 || F > 65536) return W4A16_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(E) * F > (int64_t(1) << 31) / (H / 8) - 1 ||
        static_cast<int64_t>(E) * H > (int64_t(1) << 31) / (F / 8) - 1)
        return W4A16_ERR_UNSUPPORTED;
    const void* ptrs[] = {x,      expert_ids, route_w,  gate_wq,    gate_scale, gate_zero, up_wq,
                          up_scale, up_zero,  down_wq, down_scale, down_zero,  y};
    for (const void* p : ptrs)
        if (!aligned16(p)) return W4A16_ERR_ALIGN;
    const size_t need = w4a16_moe_ffn_workspace_bytes(M, topk, H, F);
    if (!workspace || workspace_bytes < need) return W4A16_ERR_WORKSPACE;
    if (!aligned16(workspace)) return W4A16_ERR_ALIGN;
    DeviceCache* dev = nullptr;
    w4a16_status st = current_device(&dev);
    if (st != W4A16_OK) return st;
    if (moe_smem_need(M, static_cast<int>(H), static_cast<int>(g)) > dev->info.max_smem_optin ||
        moe_smem_need(M, static_cast<int>(F), static_cast<int>(g)) > dev->info.max_smem_optin)
        return W4A16_ERR_UNSUPPORTED;
    const size_t S = static_cast<size_t>(M) * static_cast<size_t>(topk);
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    uint16_t* g_out = reinterpret_cast<uint16_t*>(ws);
    uint16_t* u_out = reinterpret_cast<uint16_t*>(ws + align256(S * F * 2));
    float* part = reinterpret_cast<float*>(ws + 2 * align256(S * F * 2));
    unsigned* counters = reinterpret_cast<unsigned*>(ws + 2 * align256(S * F * 2) + align256(S * H * 4));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (moe_hmma_supports(M, topk, H, F, g) && moe_hmma_fits(dev->info, M, topk, E, H, F, 4)) {
        // the fp16 warp-MMA path: h = SwiGLU of the gate/up products in the
        // first launch's epilogue (into the gate-output part of the
        // workspace), the down products and routed sums in the second (in
        // shared memory: the rest of the workspace is not used)
        MoeHmmaArgs m{x,     expert_ids, route_w, gate_wq, gate_scale, gate_zero,
                      up_wq, up_scale,   up_zero, down_wq, down_scale, down_zero,
                      g_out, y,          M,       topk,    E,          H,
                      F,     dev->err,   4};
        return from_cuda(launch_moe_hmma(m, dev->info, s));
    }
    // gate and up products of every slot: one launch over both banks
    MoeArgs a{};
    a.x = x;
    a.ids = expert_ids;
    a.bank[0] = MoeBank{gate_wq, gate_scale, gate_zero, g_out};
    a.bank[1] = MoeBank{up_wq, up_scale, up_zero, u_out};
    a.nbanks = 2;
    a.zero_count = counters;  // for the down launch's in-launch routed sum
    a.zero_n = moe_row_chunks(static_cast<int>(H));
    a.M = M;
    a.topk = topk;
    a.E = E;
    a.N = static_cast<int>(F);
    a.K = static_cast<int>(H);
    a.g = static_cast<int>(g);
    a.err = dev->err;
    cudaError_t e = launch_moe(a, dev->info, s);
    if (e != cudaSuccess) return from_cuda(e);
    // down products of h = silu(gate) * up (formed while staging); the last
    // CTA of each row chunk forms that chunk's routed sums
    MoeArgs d{};
    d.sw_gate = g_out;
    d.sw_up = u_out;
    d.ids = expert_ids;
    d.route_w = route_w;
    d.bank[0] = MoeBank{down_wq, down_scale, down_zero, nullptr};
    d.nbanks = 1;
    d.early = 1;  // the gate/up launch signals its dependents only after its own wait
    d.y_routed = y;
    d.ws = part;
    d.chunk_count = counters;  // routed sum by the last CTA of each row chunk
    d.M = M;
    d.topk = topk;
    d.E = E;
    d.N = static_cast<int>(H);
    d.K = static_cast<int>(F);
    d.g = static_cast<int>(g);
    d.err = dev->err;
    return from_cuda(launch_moe(d, dev->info, s));
}

size_t w3a16_moe_ffn_workspace_bytes(int M, int topk, int64_t H, int64_t F) {
    (void)H;
    if (M < 1 || topk < 1 || F < 1) return 0;
    return align256(static_cast<size_t>(M) * static_cast<size_t>(topk) * static_cast<size_t>(F) * 2);
}

w4a16_status w3a16_moe_ffn(const uint16_t* x, const int32_t* expert_ids, const float* route_w,
                           const uint32_t* gate_wq3, const uint16_t* gate_scale,
                           const uint8_t* gate_zero, const uint32_t* up_wq3,
                           const uint16_t* up_scale, const uint8_t* up_zero,
                           const uint32_t* down_wq3, const uint16_t* down_scale,
                           const uint8_t* down_zero, uint16_t* y, int M, int topk, int E,
                           int64_t H, int64_t F, int64_t g, void* workspace,
                           size_t workspace_bytes, void* stream) {
    if (!x || !expert_ids || !route_w || !gate_wq3 || !gate_scale || !gate_zero || !up_wq3 ||
        !up_scale || !up_zero || !down_wq3 || !down_scale || !down_zero || !y)
        return W4A16_ERR_NULL;
    if (M < 1 || topk < 1 || E < 1 || H < 128 || F < 128 || g < 32) return W4A16_ERR_SHAPE;
    if (g % 32 != 0 || H % 128 != 0 || F % 128 != 0 || H % g != 0 || F % g != 0) return W4A16_ERR_SHAPE;
    if (!moe_hmma_supports(M, topk, H, F, g) || H > 65536 || F > 65536) return W4A16_ERR_UNSUPPORTED;
    const void* ptrs[] = {x,        expert_ids, route_w,  gate_wq3,   gate_scale, gate_zero, up_wq3,
                          up_scale, up_zero,    down_wq3, down_scale, down_zero,  y};
    for (const void* p : ptrs)
        if (!aligned16(p)) return W4A16_ERR_ALIGN;
    const size_t need = w3a16_moe_ffn_workspace_bytes(M, topk, H, F);
    if (!workspace || workspace_bytes < need) return W4A16_ERR_WORKSPACE;
    if (!aligned16(workspace)) return W4A16_ERR_ALIGN;
    DeviceCache* dev = nullptr;
    w4a16_status st = current_device(&dev);
    if (st != W4A16_OK) return st;
    if (!moe_hmma_fits(dev->info, M, topk, E, H, F, 3)) return W4A16_ERR_UNSUPPORTED;
    MoeHmmaArgs m{x,      expert_ids, route_w, gate_wq3, gate_scale, gate_zero,
                  up_wq3, up_scale,   up_zero, down_wq3, down_scale, down_zero,
                  static_cast<uint16_t*>(workspace), y, M, topk, E, H,
                  F,      dev->err,   3};
    return from_cuda(launch_moe_hmma(m, dev->info, static_cast<cudaStream_t>(stream)));
}

w4a16_status w3a16_moe_gemv(const uint16_t* x, int x_per_slot, const int32_t* expert_ids,
                            const float* route_w, const uint32_t* wq3, const uint16_t* scale,
                            const uint8_t* zero, uint16_t* y, int M, int topk, int E, int64_t N,
                            int64_t K, int64_t g, void* stream) {
    if (!x || !expert_ids || !wq3 || !scale || !zero || !y) return W4A16_ERR_NULL;
    if (M < 1 || topk < 1 || E < 1 || N < 1 || K < 128 || g < 32) return W4A16_ERR_SHAPE;
    if (K % 128 != 0 || g % 32 != 0 || K % g != 0) return W4A16_ERR_SHAPE;
    if (!moe_hmma_gemv_supports(M, topk, N, K, g)) return W4A16_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(expert_ids) || !aligned16(wq3) || !aligned16(scale) ||
        !aligned16(zero) || !aligned16(y) || (route_w && !aligned16(route_w)))
        return W4A16_ERR_ALIGN;
    DeviceCache* dev = nullptr;
    w4a16_status st = current_device(&dev);
    if (st != W4A16_OK) return st;
    if (!moe_hmma_gemv_fits(dev->info, M, topk, E, N, K, 3, x_per_slot, route_w != nullptr))
        return W4A16_ERR_UNSUPPORTED;
    MoeHmmaGemvArgs a{x, x_per_slot ? 1 : 0, expert_ids, route_w, wq3, scale, zero, y,
                      M, topk, E, N, K, dev->err, 3};
    return from_cuda(launch_moe_hmma_gemv(a, dev->info, static_cast<cudaStream_t>(stream)));
}

w4a16_status w4a16_swiglu(const uint16_t* gate, const uint16_t* up, int64_t ld_in, uint16_t* h,
                          int64_t ld_out, int64_t rows, int64_t N, void* stream) {
    if (!gate || !up || !h) return W4A16_ERR_NULL;
    if (rows < 0 || N < 0 || N % 2 != 0 || ld_in < N || ld_out < N || ld_in % 2 != 0 ||
        ld_out % 2 != 0)
        return W4A16_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(gate) & 3u) || (reinterpret_cast<uintptr_t>(up) & 3u) ||
        (reinterpret_cast<uintptr_t>(h) & 3u))
        return W4A16_ERR_ALIGN;
    if (rows == 0 || N == 0) return W4A16_OK;
    DeviceCache* dev = nullptr;
    w4a16_status st = current_device(&dev);
    if (st != W4A16_OK) return st;
    return from_cuda(launch_swiglu(gate, up, ld_in, h, ld_out, rows, N, dev->info.sms,
                                   static_cast<cudaStream_t>(stream)));
}

int w4a16_host_memory_mapped(const void* p) {
    if (!p) return 0;
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return (at.type == cudaMemoryTypeHost && at.devicePointer == p) ? 1 : 0;
}

}  // extern "C"

namespace w4a16 {
// elementwise.cu: one bounded mbarrier wait that completes (arrive != 0) or expires
cudaError_t launch_wait_selftest(uint32_t max_iters, int arrive, uint32_t* err, cudaStream_t s);
}  // namespace w4a16

extern "C" {

w4a16_status w4a16_wait_selftest(unsigned max_iters, int arrive, void* stream) {
    if (max_iters < 1 || max_iters > 8192) return W4A16_ERR_SHAPE;
    DeviceCache* dev = nullptr;
    w4a16_status st = current_device(&dev);
    if (st != W4A16_OK) return st;
    return from_cuda(launch_wait_selftest(max_iters, arrive ? 1 : 0, dev->err,
                                          static_cast<cudaStream_t>(stream)));
}

w4a16_status w4a16_device_error(uint32_t* bits_out, int clear, void* stream) {
    if (!bits_out) return W4A16_ERR_NULL;
    DeviceCache* dev = nullptr;
    w4a16_status st = current_device(&dev);
    if (st != W4A16_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return from_cuda(cudaErrorUnknown);
    uint32_t v = 0;
    if (cudaMemcpy(&v, dev->err, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess)
        return from_cuda(cudaErrorUnknown);
    const uint32_t zero_word = 0;
    if (clear && cudaMemcpy(dev->err, &zero_word, sizeof zero_word, cudaMemcpyHostToDevice) !=
                     cudaSuccess)
        return from_cuda(cudaErrorUnknown);
    *bits_out = v;
    return W4A16_OK;
}

}  // extern "C"
