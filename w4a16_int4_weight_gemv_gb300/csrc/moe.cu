// Expert-indexed W4A16 GEMV (sm_103a): the grouped expert kernel of the
// local-kimi README, technical-detail section, as a true GEMV.
//
// For token t and routed slot j, expert e = ids[t][j] multiplies its own INT4
// matrix W_e by the slot's activation row.  Tokens that route to the same
// expert share one pass over that expert's weights: CTA (chunk, d) finds the
// d-th distinct expert among the routed slots (in order of first
// appearance), gathers the activation rows of every slot routed to it into
// shared memory (the same permuted layout the dense warp-MMA kernel uses)
// and streams 16 * warps rows of W_e against all of them at once.  The
// routed ids live on the device, so the grid is sized for the worst case
// (min(E, M*topk) distinct experts) and CTAs beyond the actual count exit at
// once.
//
// With route weights the per-slot results go to an fp32 workspace and a
// second kernel forms y[t] = sum_j r[t][j] d[t][j] in slot order -- a fixed
// order, so the result is deterministic (no floating-point atomics).
#include "common.cuh"
#include "launch.h"
#include "mma_core.cuh"

namespace w4a16 {
namespace {

constexpr int kWarps = 4;
constexpr int kPD = 4;
constexpr int kMaxSlots = 256;

struct MoeKernelArgs {
    const uint16_t* x;
    int x_per_slot;
    const int32_t* ids;
    const uint4* wq;
    const uint16_t* scale;
    const uint8_t* zero;
    uint16_t* y;  // per-slot bf16 output (no route weights)
    float* ws;    // per-slot fp32 output (route weights given)
    int M;
    int topk;
    int E;
    int N;
    int K;
    int g;
    uint32_t* err;
};

template <int NT>
__global__ void __launch_bounds__(kWarps * 32)
k_moe_mma(const MoeKernelArgs a) {
    constexpr int Mpad = 8 * NT;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __shared__ int s_ids[kMaxSlots];
    __shared__ unsigned char s_first[kMaxSlots];
    __shared__ int s_expert;
    __shared__ int s_nslots;
    __shared__ int s_slots[kMaxSlots];
    __shared__ int s_rowsel[Mpad];

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int S = a.M * a.topk;
    const int nblk = a.K >> 7;
    const int Q = a.K >> 5;
    const int G = a.K / a.g;
    const int tok_stride = mma_token_stride(nblk);
    unsigned char* xs = smem_raw;
    float* xsum = reinterpret_cast<float*>(smem_raw + Mpad * tok_stride);

    // 1. which expert does this CTA serve?
    for (int i = threadIdx.x; i < S; i += blockDim.x) s_ids[i] = a.ids[i];
    if (threadIdx.x == 0) s_expert = -1;
    __syncthreads();
    for (int i = threadIdx.x; i < S; i += blockDim.x) {
        const int e = s_ids[i];
        bool first = (e >= 0 && e < a.E);
        if (!first && blockIdx.x == 0 && blockIdx.y == 0)
            raise_device_error(a.err, W4A16_DEVERR_EXPERT_ID);
        for (int j = 0; j < i && first; ++j) first = (s_ids[j] != e);
        s_first[i] = first ? 1 : 0;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < S; i += blockDim.x) {
        if (!s_first[i]) continue;
        int ord = 0;
        for (int j = 0; j < i; ++j) ord += s_first[j];
        if (ord == static_cast<int>(blockIdx.y)) s_expert = s_ids[i];
    }
    __syncthreads();
    const int e = s_expert;

    // invalid ids produce zero rows in the per-slot output
    if (a.ws == nullptr && blockIdx.y == 0) {
        for (int i = 0; i < S; ++i) {
            if (s_ids[i] >= 0 && s_ids[i] < a.E) continue;
            for (int row = blockIdx.x * kWarps * 16 + threadIdx.x;
                 row < min(a.N, (blockIdx.x + 1) * kWarps * 16); row += blockDim.x)
                a.y[static_cast<size_t>(i) * a.N + row] = 0;
        }
    }
    if (e < 0) return;

    if (threadIdx.x == 0) {
        int n = 0;
        for (int i = 0; i < S; ++i)
            if (s_ids[i] == e) s_slots[n++] = i;
        s_nslots = n;
    }
    __syncthreads();
    const int nslots = s_nslots;

    const uint4* wq = a.wq + static_cast<size_t>(e) * a.N * Q;
    const uint16_t* scale = a.scale + static_cast<size_t>(e) * a.N * G;
    const uint8_t* zero = a.zero + static_cast<size_t>(e) * a.N * G;
    const int r = lane >> 2;
    const int c = lane & 3;
    const int n0 = (blockIdx.x * kWarps + warp) * 16 + r;
    const int n1 = n0 + 8;

    const int tile = blockIdx.x * kWarps + warp;  // 16-row tile of expert e
    auto issue = [&](int blk, MmaBlockLoad& L) {
        mma_block_issue(L, wq, scale, zero, a.N, Q, G, a.g, tile, blk, lane);
    };

    // 2. passes of up to Mpad slots routed to expert e (normally one)
    for (int base = 0; base < nslots; base += Mpad) {
        const int m = min(Mpad, nslots - base);
        MmaBlockLoad ring[kPD];
#pragma unroll
        for (int p = 0; p < kPD; ++p)
            if (p < nblk) issue(p, ring[p]);
        if (threadIdx.x < Mpad) {
            int rs = -1;
            if (static_cast<int>(threadIdx.x) < m) {
                const int slot = s_slots[base + threadIdx.x];
                rs = a.x_per_slot ? slot : slot / a.topk;
            }
            s_rowsel[threadIdx.x] = rs;
        }
        __syncthreads();
        stage_x_permuted<NT>(a.x, s_rowsel, m, a.K, 0, nblk, xs, xsum, tok_stride);
        __syncthreads();

        float acc[NT][4];
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[t][i] = 0.f;
        for (int b0 = 0; b0 < nblk; b0 += kPD) {
#pragma unroll
            for (int p = 0; p < kPD; ++p) {
                const int b = b0 + p;
                if (b < nblk) {
                    mma_block<NT>(acc, ring[p], xs + b * 256, xsum + b * Mpad, tok_stride, m,
                                  lane);
                    if (b + kPD < nblk) issue(b + kPD, ring[p]);
                }
            }
        }
        // outputs: C fragment rows r / r + 8, tokens 2c, 2c + 1 (+ 8 t)
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int tok = t * 8 + 2 * c + (i & 1);
                const int n = (i < 2) ? n0 : n1;
                if (tok < m && n < a.N) {
                    const size_t o = static_cast<size_t>(s_slots[base + tok]) * a.N + n;
                    if (a.ws) a.ws[o] = acc[t][i];
                    else a.y[o] = f32_to_bf16_rn(acc[t][i]);
                }
            }
        __syncthreads();  // s_rowsel / xs are rewritten by the next pass
    }
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

}  // namespace

cudaError_t launch_moe(const MoeArgs& a, const DeviceInfo& dev, cudaStream_t s) {
    MoeKernelArgs k{};
    k.x = a.x;
    k.x_per_slot = a.x_per_slot;
    k.ids = a.ids;
    k.wq = reinterpret_cast<const uint4*>(a.wq);
    k.scale = a.scale;
    k.zero = a.zero;
    k.y = a.route_w ? nullptr : a.y;
    k.ws = a.route_w ? a.ws : nullptr;
    k.M = a.M;
    k.topk = a.topk;
    k.E = a.E;
    k.N = a.N;
    k.K = a.K;
    k.g = a.g;
    k.err = a.err;
    const int S = a.M * a.topk;
    const int dmax = S < a.E ? S : a.E;
    const int chunks = (a.N + kWarps * 16 - 1) / (kWarps * 16);
    const int nblk = a.K / 128;
    const dim3 grid(chunks, dmax);
    cudaError_t e;
    if (a.M <= 8) {
        const int smem = 8 * mma_token_stride(nblk) + nblk * 8 * 4;
        e = cudaFuncSetAttribute(k_moe_mma<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        k_moe_mma<1><<<grid, kWarps * 32, smem, s>>>(k);
    } else {
        const int smem = 16 * mma_token_stride(nblk) + nblk * 16 * 4;
        e = cudaFuncSetAttribute(k_moe_mma<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        k_moe_mma<2><<<grid, kWarps * 32, smem, s>>>(k);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess || !a.route_w) return e;
    const int total = a.M * a.N;
    int blocks = (total + 255) / 256;
    if (blocks > 4 * dev.sms) blocks = 4 * dev.sms;
    k_moe_route_sum<<<blocks, 256, 0, s>>>(a.ws, a.route_w, a.ids, a.y, a.M, a.topk, a.E, a.N);
    return cudaGetLastError();
}

}  // namespace w4a16
