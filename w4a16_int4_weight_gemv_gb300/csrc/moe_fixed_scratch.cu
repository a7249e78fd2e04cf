// Routed expert GEMV that allocates nothing: its fp32 partials live in a
// fixed device array compiled into the library.
//
// Who needs it.  Some callers cannot call cudaMalloc, or cannot hand the
// library a workspace: engines whose device memory is pre-partitioned into
// fixed pools with nothing spare to lend, and plug-ins loaded by a host
// runtime that owns the allocator and exposes none of it.  For them the
// library keeps one statically sized scratch buffer per device.
//
// Costs and rules.  The buffer is kFixedScratchBytes per GPU that loads the
// library and is held until the process exits.  Only routed calls (route_w
// given) use it; the first one on each device looks its address up
// (cudaGetSymbolAddress, with that device current) and caches it for the
// life of the process, so the call must not be used after cudaDeviceReset.
// Every call on a device shares the one buffer: calls whose kernels may
// overlap on the GPU (different streams without ordering between them) race
// on it and give wrong results; calls in one stream, or otherwise ordered,
// are safe.  The contents left by the previous call are never read: each
// routed slot's partials are written before the reduction reads them, and
// slots with an invalid expert id are skipped by both kernels.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "w4a16.h"

namespace w4a16 {
namespace {

constexpr size_t kFixedScratchBytes = W4A16_FIXED_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_fixed_scratch[kFixedScratchBytes];

constexpr int kMaxScratchDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxScratchDevices] = {};

// Device address of g_fixed_scratch on the current device (looked up once).
w4a16_status fixed_scratch(void** out) {
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxScratchDevices)
        return W4A16_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[d]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_fixed_scratch) != cudaSuccess || !p) {
            (void)cudaGetLastError();
            return W4A16_ERR_CUDA;
        }
        g_scratch_ptr[d] = p;
    }
    *out = g_scratch_ptr[d];
    return W4A16_OK;
}

}  // namespace
}  // namespace w4a16

extern "C" W4A16_API w4a16_status w4a16_moe_gemv_fixed_scratch(
    const uint16_t* x, int x_per_slot, const int32_t* expert_ids, const float* route_w,
    const uint32_t* wq, const uint16_t* scale, const uint8_t* zero, uint16_t* y, int M, int topk,
    int E, int64_t N, int64_t K, int64_t g, void* stream) {
    if (!route_w)  // no routed sum: no partials, no buffer
        return w4a16_moe_gemv(x, x_per_slot, expert_ids, route_w, wq, scale, zero, y, M, topk, E,
                              N, K, g, nullptr, 0, stream);
    if (M >= 1 && topk >= 1 && N >= 1) {
        // reject oversized requests before touching the device
        const size_t need = w4a16_moe_workspace_bytes(M, topk, N, 1);
        if (need > w4a16::kFixedScratchBytes) return W4A16_ERR_WORKSPACE;
    }
    void* scratch = nullptr;
    const w4a16_status st = w4a16::fixed_scratch(&scratch);
    if (st != W4A16_OK) return st;
    return w4a16_moe_gemv(x, x_per_slot, expert_ids, route_w, wq, scale, zero, y, M, topk, E, N,
                          K, g, scratch, w4a16::kFixedScratchBytes, stream);
}
