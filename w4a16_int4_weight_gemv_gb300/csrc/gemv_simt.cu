// M = 1 or 2 W4A16 GEMV on CUDA cores (sm_103a).
//
// The decode-time product of the local-kimi README, technical-detail section:
// one (or two) activation rows against a group-quantised INT4 matrix, done as
// a true GEMV -- every lane walks the reduction axis K of its rows with
// 128-bit coalesced loads and keeps one fp32 accumulator per output.
//
// Arithmetic.  For one 16-byte chunk (32 consecutive k of one row, all in one
// quantisation group because g % 32 == 0) the kernel forms
//     acc = sum_k code_k * x_k
// with every product exact in fp32, then applies the group's zero point and
// scale once:  partial += s * (acc - z * sum_k x_k),  which equals
// sum_k (code_k - z) * s * x_k.
//
// Nibble -> float without conversion instructions: the bit pattern
// (word & (0xF << p)) read as a binary32 is code * 2^(p - 149) (a subnormal,
// or for p = 20 and code >= 8 one of the smallest normals, whose value is
// still the integer pattern times 2^-149).  Multiplying it by x * 2^(85 - p)
// gives code * x * 2^-64 exactly, so a weight costs one LOP3 and half a packed
// FFMA (fma.rn.f32x2 multiplies two codes by their two x' at once) per token,
// plus one shift per word that brings the top two nibbles down by 8 bits.
// The kernel is issue-bound: everything other than the masks and the packed
// FMAs is kept off the issue ports as far as possible or amortised over a span
// of rows.  The 2^(85 - p) factors are
// folded into the staged activations and the 2^64 is restored on the output.
// The FMAs keep subnormal operands (the library is built without
// flush-to-zero); the exact product of a bf16 x and a 4-bit code stays normal
// unless |code * x| < 2^-62.  Inputs need |x| < 2^43 so x * 2^85 stays finite;
// a larger (or non-finite) activation sets W4A16_DEVERR_RANGE.
//
// Work split.  One persistent CTA of 16 warps per SM.  Warps own tiles of TR
// rows (4, or 8 when rows are plentiful); a step of a warp is one span of its
// tile (32 consecutive chunks = 512 contiguous bytes of each row, one chunk
// per lane).  Everything a step reads from memory lands in a per-warp ring of
// shared-memory stages and completes on the stage's mbarrier: the packed words
// by bulk copies (the TMA engine, one 512-byte copy per row, issued by one
// lane) and the step's scales and zero points by cp.async pieces from a few
// lanes.  So the bytes in flight are bounded by shared memory rather than by
// registers or by the L1's outstanding-request tracking, and the step loop is
// a small non-unrolled loop that stays in the instruction cache.  When rows
// are few, the K range of a tile is split over WPT warps of the CTA (partials
// added in shared memory behind a named barrier, once per tile) and over the
// CTAs of a thread-block cluster (added through distributed shared memory,
// once per kernel), always in a fixed order, so results are deterministic.
//
// Activations.  The CTA's K slice of x is read once with 16-byte loads --
// issued before any weight copy, so they are not queued behind the weight
// stream -- scaled per nibble position into fp32 x' and stored in shared
// memory lane-major ([span][piece][lane][4 floats]) so that a warp's 16-byte
// reads of one piece are consecutive (conflict-free) at immediate offsets;
// per-chunk sums are reduced with warp shuffles in the same pass.
//
// Launch.  Kernels are launched with programmatic stream serialisation: the
// next launch on the stream may start its CTAs as this grid drains, and every
// CTA waits (griddepcontrol.wait) for the preceding grid before it reads or
// writes global memory -- or, when the caller declares the weights constant,
// only before it reads x or writes y, so its first weight loads overlap the
// previous kernel.
#include "common.cuh"
#include "launch.h"

namespace w4a16 {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kCtasPerSm = 1;  // CTAs of this kernel resident per SM
constexpr int kMaxStages = 8;

// Shared-memory stage of one warp step for tiles of TR rows: the rows' 512-byte
// spans of packed words, then their scales (up to 64 bytes a row) and zero
// points (up to 32 bytes a row).
template <int TR>
struct Stage {
    static constexpr int kWords = 0;
    static constexpr int kScales = TR * 512;
    static constexpr int kZeros = TR * 512 + TR * 64;
    static constexpr int kBytes = TR * 608;
};

struct SimtKernelArgs {
    const uint16_t* x;
    const uint4* wq;
    const uint16_t* scale;
    const uint8_t* zero;
    void* y;
    int out_f32;
    int N;
    int K;
    int g;
    int wpt;              // warps per tile (K split inside the CTA)
    int ksplit;           // CTAs per cluster (K split across the cluster)
    int spans_per_cta;    // 32-chunk spans in one CTA's K slice
    int tiles_per_group;  // upper bound of tiles any tile group processes
    int stages;           // shared-memory stages per warp
    int weights_static;   // weights may be read before the preceding grid completes
    uint32_t* err;
};

// x'[k] = x[k] * 2^(85 - p), p the bit offset the code of k sits at after the
// masking: nibbles 0..5 at 4*i, nibbles 6 and 7 (shifted down by 8) at 16, 20.
__device__ __forceinline__ float position_factor(int i) {
    const int p = (i < 6) ? 4 * i : 4 * i - 8;
    return exp2i(85 - p);
}

// acc += sum over the 16 codes of two words of code * x'.  The products of
// codes (k, k+1) go through one packed fp32 FMA (fma.rn.f32x2: two IEEE fmas
// per instruction, subnormal operands kept), so a word costs 8 masks, 4 packed
// FMAs and one shift.  The shift by 8 is a high multiply, which issues on the
// FMA pipe instead of the ALU pipe.
__device__ __forceinline__ void dot_words(float& a0, float& a1, uint32_t v0, uint32_t v1,
                                          const float* xr) {
    const uint32_t vs[2] = {v0, v1};
    float2 acc = make_float2(a0, a1);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const uint32_t v = vs[j];
        const uint32_t t = __umulhi(v, 0x01000000u);  // v >> 8
        acc = __ffma2_rn(make_float2(__uint_as_float(v & 0x0000000Fu), __uint_as_float(v & 0x000000F0u)),
                         make_float2(xr[8 * j + 0], xr[8 * j + 1]), acc);
        acc = __ffma2_rn(make_float2(__uint_as_float(v & 0x00000F00u), __uint_as_float(v & 0x0000F000u)),
                         make_float2(xr[8 * j + 2], xr[8 * j + 3]), acc);
        acc = __ffma2_rn(make_float2(__uint_as_float(v & 0x000F0000u), __uint_as_float(v & 0x00F00000u)),
                         make_float2(xr[8 * j + 4], xr[8 * j + 5]), acc);
        acc = __ffma2_rn(make_float2(__uint_as_float(t & 0x000F0000u), __uint_as_float(t & 0x00F00000u)),
                         make_float2(xr[8 * j + 6], xr[8 * j + 7]), acc);
    }
    a0 = acc.x;
    a1 = acc.y;
}

__device__ __forceinline__ void store_y(void* y, int out_f32, size_t i, float v) {
    v *= exp2i(64);
    if (out_f32) static_cast<float*>(y)[i] = v;
    else static_cast<uint16_t*>(y)[i] = f32_to_bf16_rn(v);
}

__host__ __device__ inline int simt_base_bytes(int MT, int TR, int spans, int tg, int wpt,
                                               int tpg, int S) {
    const int b = MT * spans * (4096 + 128) + 2 * tg * wpt * TR * MT * 4 +
                  (S > 1 ? tpg * S * tg * TR * MT * 4 : 0);
    return (b + 127) & ~127;
}

// CPG > 0: g = 32 * CPG with CPG in {1, 2, 4}; the step's scales and zero
// points are copied into its stage with cp.async (needs K % 1024 == 0 and
// 16-byte aligned row pieces).  CPG == 0: any g; every lane loads the pair of
// its own chunk for each row.
template <int MT, int TR, int CPG>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
k_gemv_simt(const SimtKernelArgs a) {
    using St = Stage<TR>;
    constexpr bool kAsyncSZ = CPG > 0;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int WPT = a.wpt;
    const int TG = kWarps / WPT;     // tile groups per CTA
    const int tg = warp / WPT;
    const int kp = warp - tg * WPT;  // this warp's part of the K slice
    const int Q = a.K >> 5;          // 16-byte chunks per row
    const int nspan_all = (Q + 31) >> 5;
    const int S = a.ksplit;
    const int rank = (S > 1) ? static_cast<int>(cluster_rank()) : 0;
    const int cid = blockIdx.x / S;
    const int ncl = gridDim.x / S;
    const int SP = a.spans_per_cta;
    const int span0 = rank * SP;
    const int nspan = max(0, min(nspan_all, span0 + SP) - span0);
    const int ntiles = (a.N + TR - 1) / TR;
    const int G = a.K / a.g;
    const int cpg = a.g >> 5;  // chunks per quantisation group
    const int NS = a.stages;
    // async scale/zero pieces per row: scales GS * 2 bytes in 16-byte pieces,
    // zeros GS bytes in 16-byte pieces (one 8-byte piece when GS == 8)
    constexpr int GS = kAsyncSZ ? 32 / CPG : 1;
    constexpr int kSPR = kAsyncSZ ? (GS * 2) / 16 : 0;
    constexpr int kZPR = kAsyncSZ ? (GS >= 16 ? GS / 16 : 1) : 0;
    constexpr int kPPR = kSPR + kZPR;
    constexpr int kPieces = TR * kPPR;
    constexpr int n_arrive = kPieces < 32 ? kPieces : 32;

    float* xs = reinterpret_cast<float*>(smem_raw);  // [MT][SP * 1024] swizzled x'
    float* xsum = xs + MT * SP * 1024;              // [MT][SP * 32] chunk sums * 2^-64
    float* red = xsum + MT * SP * 32;               // [2][TG][WPT][TR * MT]
    float* part = red + 2 * TG * WPT * TR * MT;     // [tpg][S][TG][TR * MT] (S > 1)
    const int base = simt_base_bytes(MT, TR, SP, TG, WPT, a.tiles_per_group, S);
    unsigned char* ring = smem_raw + base + warp * NS * St::kBytes;
    uint64_t* bars =
        reinterpret_cast<uint64_t*>(smem_raw + base + kWarps * NS * St::kBytes) + warp * NS;

    // tile groups are dealt round-robin over the CTAs (group tg of CTA cid is
    // tg * ncl + cid), so with more CTAs than a full group layout needs the
    // tiles spread over all of them instead of filling the first ones
    const int gid = tg * ncl + cid;
    const int NG = ncl * TG;
    const int my_tiles = (ntiles > gid) ? (ntiles - gid + NG - 1) / NG : 0;
    const int my_spans = (nspan > kp) ? (nspan - kp + WPT - 1) / WPT : 0;
    const int nss = my_tiles * my_spans;  // (tile, span) steps of this warp

    grid_dependents_launch();
    if (lane == 0) {
        for (int i = 0; i < NS; ++i) mbar_init(bars + i, 1 + (kAsyncSZ ? n_arrive : 0));
        mbar_init_fence();
    }
    __syncwarp();
    // K split over a cluster: this CTA is running; the matching wait comes
    // before the first store into a peer's shared memory
    if (S > 1) cluster_arrive_relaxed();

    // producer cursor: step (w_tile, w_span) goes to stage w_stage
    int w_tile = gid, w_span = kp, w_stage = 0, w_issued = 0;
    auto issue = [&]() {
        uint64_t* bar = bars + w_stage;
        unsigned char* dst = ring + w_stage * St::kBytes;
        const int c0 = (span0 + w_span) << 5;
        const int rows = min(TR, a.N - w_tile * TR);
        const size_t row0 = static_cast<size_t>(w_tile) * TR;
        // lane 0 announces the bytes; lanes r < rows copy row r (the copies may
        // land before the announcement: the phase needs both)
        const uint32_t row_bytes = static_cast<uint32_t>(min(32, Q - c0)) * 16u;
        if (lane == 0) {
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(bar, row_bytes * static_cast<uint32_t>(rows));
        }
        if (lane < rows)
            bulk_copy_g2s(dst + St::kWords + lane * 512, a.wq + (row0 + lane) * Q + c0, row_bytes,
                          bar);
        if constexpr (kAsyncSZ) {
            const int first = c0 / CPG;  // first group of the span
#pragma unroll
            for (int pc0 = 0; pc0 < kPieces; pc0 += 32) {
                const int pc = pc0 + lane;
                const int r = pc / kPPR;
                const int j = pc - r * kPPR;
                if (pc < kPieces && r < rows) {
                    const size_t gi = (row0 + r) * G + first;
                    if (j < kSPR)
                        cp_async_16(dst + St::kScales + r * 64 + j * 16, a.scale + gi + j * 8);
                    else if (GS >= 16)
                        cp_async_16(dst + St::kZeros + r * 32 + (j - kSPR) * 16,
                                    a.zero + gi + (j - kSPR) * 16);
                    else
                        cp_async_8(dst + St::kZeros + r * 32, a.zero + gi);
                }
            }
            if (lane < n_arrive) cp_async_arrive_noinc(bar);
        }
        if (++w_stage == NS) w_stage = 0;
        ++w_issued;
        w_span += WPT;
        if (w_span >= nspan) {
            w_span = kp;
            w_tile += NG;
        }
    };

    // stage x' and the chunk sums of this CTA's K slice (one pass)
    const int kbeg = span0 << 10;
    const int kend = min(a.K, (span0 + nspan) << 10);
    const int npieces = nspan << 7;  // 8 consecutive k per piece, 4 pieces per chunk
    auto load_piece = [&](int m, int i) {
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (i < npieces && kbeg + (i << 3) < kend)
            v = __ldg(reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(m) * a.K + kbeg +
                                                     (i << 3)));
        return v;
    };
    // all lanes of the warp take part (chunk sums are 4-lane shuffles)
    bool out_of_range = false;  // some |x| >= 2^43: x' would overflow
    auto store_piece = [&](int m, int i, const uint4 v) {
        const int k0 = i << 3;   // local k
        const int cl = k0 >> 5;  // local chunk
        const int q0 = (k0 >> 2) & 7;
        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
        float f[8];
        float sum = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            // bf16 magnitude bits >= those of 2^43 (biased exponent 170)
            out_of_range |= (wv[e] & 0x7FFFu) >= 0x5500u || (wv[e] & 0x7FFF0000u) >= 0x55000000u;
            const float lo = bf16_to_f32(wv[e] & 0xFFFFu);
            const float hi = bf16_to_f32(wv[e] >> 16);
            sum += lo + hi;
            f[2 * e] = lo * position_factor(2 * e);
            f[2 * e + 1] = hi * position_factor(2 * e + 1);
        }
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        if (i < npieces) {
            float4* bp = reinterpret_cast<float4*>(xs + m * SP * 1024) + (cl >> 5) * 256 + (cl & 31);
            bp[q0 * 32] = make_float4(f[0], f[1], f[2], f[3]);
            bp[(q0 + 1) * 32] = make_float4(f[4], f[5], f[6], f[7]);
            if ((i & 3) == 0) xsum[m * SP * 32 + cl] = sum * exp2i(-64);
        }
    };

    // The activations gate all arithmetic: their loads are issued before the
    // weight rings so they are not queued behind the weight stream, and only
    // one stage per warp is requested before they are converted -- issuing a
    // whole ring per warp here (tens of MB over the GPU) stalls the warps on
    // memory back-pressure before they reach the conversion.  The rings are
    // topped up once x' is staged.  With static weights that one stage is
    // requested while the preceding grid finishes.
    if (a.weights_static && nss > 0) issue();
    grid_dependency_wait();
    constexpr int kXPre = 4;  // pieces per thread and token loaded ahead
    uint4 xpre[MT][kXPre];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int j = 0; j < kXPre; ++j) xpre[m][j] = load_piece(m, threadIdx.x + j * blockDim.x);
    __syncthreads();
    if (w_issued == 0 && nss > 0) issue();
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int j = 0; j < kXPre; ++j)
            if (j * static_cast<int>(blockDim.x) < npieces)
                store_piece(m, threadIdx.x + j * blockDim.x, xpre[m][j]);
    for (int m = 0; m < MT; ++m)
        for (int b = kXPre * blockDim.x; b < npieces; b += blockDim.x)
            store_piece(m, b + threadIdx.x, load_piece(m, b + threadIdx.x));
    if (__syncthreads_or(out_of_range) && threadIdx.x == 0)
        raise_device_error(a.err, W4A16_DEVERR_RANGE);
    while (w_issued < NS && w_issued < nss) issue();
    if (S > 1) cluster_wait();  // every peer CTA has started

    float acc[TR][MT];
#pragma unroll
    for (int r = 0; r < TR; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[r][m] = 0.f;
    int c_tile = gid, c_span = kp, ti = 0, c_stage = 0;
    uint32_t c_phase = 0;
    bool timed_out = false;

    // Reduce the TR * MT partials of every lane across the warp.  Halving
    // exchanges first (each lane keeps the half of the values its partner
    // does not), then a butterfly on the last value: lane l ends with the sum
    // of value v(l) = its low log2(TR * MT) bits read in reverse order.
    constexpr int NV = TR * MT;
    constexpr int LV = NV == 16 ? 4 : (NV == 8 ? 3 : (NV == 4 ? 2 : (NV == 2 ? 1 : 0)));
    auto warp_reduce_scatter = [&](float (&v)[NV]) -> float {
#pragma unroll
        for (int lvl = 0; lvl < LV; ++lvl) {
            const int half = NV >> (lvl + 1);
            const bool upper = (lane >> lvl) & 1;
#pragma unroll
            for (int i = 0; i < half; ++i) {
                const float send = upper ? v[i] : v[i + half];
                const float keep = upper ? v[i + half] : v[i];
                v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 1 << lvl);
            }
        }
        float s = v[0];
#pragma unroll
        for (int o = 1 << LV; o < 32; o <<= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        return s;
    };
    // value index held by this lane after the reduce-scatter
    int vid = 0;
#pragma unroll
    for (int lvl = 0; lvl < LV; ++lvl) vid |= ((lane >> lvl) & 1) << (LV - 1 - lvl);

    // lane l < NV owns output value vid (row vid / MT, token vid % MT)
    auto tile_end = [&]() {
        float v[NV];
#pragma unroll
        for (int r = 0; r < TR; ++r)
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                v[r * MT + m] = acc[r][m];
                acc[r][m] = 0.f;
            }
        float mine = warp_reduce_scatter(v);
        const int orow = vid / MT;
        const int otok = vid - orow * MT;
        if (WPT > 1) {
            float* rb = red + ((ti & 1) * TG + tg) * WPT * NV;
            if (lane < NV) rb[kp * NV + vid] = mine;
            named_barrier_sync(1 + tg, WPT * 32);
            if (kp == 0 && lane < NV) {
                mine = 0.f;
                for (int q = 0; q < WPT; ++q) mine += rb[q * NV + vid];
            }
        }
        if (kp == 0 && lane < NV) {
            if (S == 1) {
                const int n = c_tile * TR + orow;
                if (n < a.N) store_y(a.y, a.out_f32, static_cast<size_t>(otok) * a.N + n, mine);
            } else {
                // into the owner's shared memory (CTA ti % S of the cluster)
                st_dsmem_f32(part + ((ti * S + rank) * TG + tg) * NV + vid,
                             static_cast<uint32_t>(ti % S), mine);
            }
        }
    };

#pragma unroll 1
    for (int ss = 0; ss < nss; ++ss) {
        if (!mbar_wait_bounded(bars + c_stage, c_phase)) timed_out = true;
        const unsigned char* stg = ring + c_stage * St::kBytes;
        const int cl = (c_span << 5) + lane;  // chunk within the slice
        const int c = (span0 << 5) + cl;      // global chunk
        if (c < Q) {
            uint32_t sz[TR];
            if constexpr (kAsyncSZ) {
                const int lg = lane / CPG;  // group within the span
#pragma unroll
                for (int r = 0; r < TR; ++r)
                    sz[r] = *reinterpret_cast<const uint16_t*>(stg + St::kScales + r * 64 + lg * 2) |
                            (static_cast<uint32_t>(stg[St::kZeros + r * 32 + lg]) << 16);
            } else {
                const int grp = c / cpg;
#pragma unroll
                for (int r = 0; r < TR; ++r) {
                    const int n = c_tile * TR + r;
                    sz[r] = 0u;
                    if (n < a.N) {
                        const size_t gi = static_cast<size_t>(n) * G + grp;
                        sz[r] = ldg_nc_u16(a.scale + gi) | (ldg_nc_u8(a.zero + gi) << 16);
                    }
                }
            }
            uint4 wv[TR];
#pragma unroll
            for (int r = 0; r < TR; ++r)
                wv[r] = *reinterpret_cast<const uint4*>(stg + St::kWords + r * 512 + lane * 16);
            float d0[TR][MT], d1[TR][MT];
#pragma unroll
            for (int r = 0; r < TR; ++r)
#pragma unroll
                for (int m = 0; m < MT; ++m) d0[r][m] = d1[r][m] = 0.f;
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                const float4* xb = reinterpret_cast<const float4*>(xs + m * SP * 1024) +
                                   c_span * 256 + lane;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float xr[16];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float4 t = xb[(4 * h + q) * 32];
                        xr[4 * q + 0] = t.x;
                        xr[4 * q + 1] = t.y;
                        xr[4 * q + 2] = t.z;
                        xr[4 * q + 3] = t.w;
                    }
#pragma unroll
                    for (int r = 0; r < TR; ++r) {
                        if (h == 0) dot_words(d0[r][m], d1[r][m], wv[r].x, wv[r].y, xr);
                        else dot_words(d0[r][m], d1[r][m], wv[r].z, wv[r].w, xr);
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < TR; ++r) {
                const float sc = __uint_as_float(sz[r] << 16);
                const float zf =
                    __uint_as_float(__byte_perm(sz[r], 0x4B000000u, 0x7542)) - 8388608.f;
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    const float xc = xsum[m * SP * 32 + cl];
                    acc[r][m] = fmaf(sc, fmaf(-zf, xc, d0[r][m] + d1[r][m]), acc[r][m]);
                }
            }
        }
        __syncwarp();  // every lane is done with stage c_stage
        if (w_issued < nss) issue();
        if (++c_stage == NS) {
            c_stage = 0;
            c_phase ^= 1u;
        }
        c_span += WPT;
        if (c_span >= nspan) {
            tile_end();
            c_span = kp;
            c_tile += NG;
            ++ti;
        }
    }
    if (timed_out && lane == 0) raise_device_error(a.err, W4A16_DEVERR_TIMEOUT);
    // a warp with no span in the slice still joins its group's reductions
    if (my_spans == 0)
        for (; ti < my_tiles; ++ti) {
            tile_end();
            c_tile += NG;
        }

    // cluster K split: every rank stored its partials of tile t into the
    // shared memory of the owner, rank t % S; after one cluster barrier the
    // owner adds them in rank order (deterministic) and stores y
    if (S > 1) {
        cluster_barrier();
        const int per_t = TG * TR * MT;
        const int tot = a.tiles_per_group * per_t;
        for (int idx = threadIdx.x; idx < tot; idx += blockDim.x) {
            const int t = idx / per_t;
            const int rem = idx - t * per_t;
            const int g2 = rem / (TR * MT);
            const int l = rem - g2 * TR * MT;
            const int gid2 = g2 * ncl + cid;
            const int mt = (ntiles > gid2) ? (ntiles - gid2 + NG - 1) / NG : 0;
            if (t >= mt || (t % S) != rank) continue;
            float v = 0.f;
            for (int q = 0; q < S; ++q) v += part[((t * S + q) * TG + g2) * (TR * MT) + l];
            const int orow = l / MT;
            const int n = (gid2 + t * NG) * TR + orow;
            if (n < a.N) store_y(a.y, a.out_f32, static_cast<size_t>(l - orow * MT) * a.N + n, v);
        }
    }
}

// rows per warp tile: 8 when there are rows enough to keep every warp busy
int tile_rows_for(const DeviceInfo& dev, int N) { return (N / 8 >= dev.sms * kWarps) ? 8 : 4; }

bool async_sz_ok(int K, int g) {
    const int G = K / g;
    if (K % 1024 != 0) return false;
    if (g == 128) return G % 8 == 0;
    if (g == 64 || g == 32) return G % 16 == 0;
    return false;
}


using SimtKernel = void (*)(SimtKernelArgs);

SimtKernel pick_simt_kernel(int M, int tile_rows, int K, int g) {
    const int cpg = async_sz_ok(K, g) ? g / 32 : 0;
    SimtKernel kern = nullptr;
#define W4A16_SIMT_PICK(MT_, TR_)                                                   \
    kern = cpg == 1   ? k_gemv_simt<MT_, TR_, 1>                                   \
           : cpg == 2 ? k_gemv_simt<MT_, TR_, 2>                                   \
           : cpg == 4 ? k_gemv_simt<MT_, TR_, 4>                                   \
                      : k_gemv_simt<MT_, TR_, 0>;
    if (M == 1) {
        if (tile_rows == 8) { W4A16_SIMT_PICK(1, 8) } else { W4A16_SIMT_PICK(1, 4) }
    } else {
        if (tile_rows == 8) { W4A16_SIMT_PICK(2, 8) } else { W4A16_SIMT_PICK(2, 4) }
    }
#undef W4A16_SIMT_PICK
    return kern;
}

}  // namespace

GemvPlan plan_gemv_simt(const DeviceInfo& dev, int M, int N, int K, int g, int k_split_req) {
    const int nspan_all = (K / 32 + 31) / 32;
    const int TR = tile_rows_for(dev, N);
    const int ntiles = (N + TR - 1) / TR;
    const int stage = TR * 608;
    const void* kern = reinterpret_cast<const void*>(pick_simt_kernel(M, TR, K, g));
    int budget = dev.smem_per_sm / kCtasPerSm - 1024;
    if (budget > dev.max_smem_optin) budget = dev.max_smem_optin;
    // feasibility and residency with the minimum two stages per warp; the
    // launch fills the budget with stages, so cluster co-residency is queried
    // at the budget
    // a split tile's reduction costs about a quarter of a 1024-k span: with
    // tiles to spare (the vocabulary head) the unsplit plan wins (82 vs 85 us)
    const SplitChoice c = choose_split(
        dev, ntiles, nspan_all, kWarps, kCtasPerSm, k_split_req, 1,
        [M, TR, stage](int upc, int tg, int wpt, int tpg, int S) {
            return simt_base_bytes(M, TR, upc, tg, wpt, tpg, S) + kWarps * 2 * (stage + 8);
        },
        [kern, budget](int S, int) { return max_active_clusters(kern, kThreads, budget, S); });
    GemvPlan p{};
    p.kernel_id = 1;
    p.k_split = c.S;
    p.wpt = c.wpt;
    p.units_per_cta = c.units_per_cta;
    p.threads = kThreads;
    p.ctas = c.ctas;
    p.tiles_per_cluster = c.tiles_per_group;
    p.tile_rows = TR;
    if (c.ctas > 0) {
        const int base = simt_base_bytes(M, TR, c.units_per_cta, kWarps / c.wpt, c.wpt,
                                         c.tiles_per_group, c.S);
        // a warp runs at most tiles_per_group * ceil(units / wpt) steps; more
        // stages than that only occupy shared memory the next launch could use
        const int max_steps = c.tiles_per_group * ((c.units_per_cta + c.wpt - 1) / c.wpt);
        int ns = (budget - base) / (kWarps * (stage + 8));
        if (ns > kMaxStages) ns = kMaxStages;
        if (ns > max_steps) ns = max_steps < 2 ? 2 : max_steps;
        p.stages = ns;
        p.smem_bytes = base + kWarps * ns * (stage + 8);
    }
    return p;
}

cudaError_t launch_gemv_simt(const GemvArgs& a, const GemvPlan& p, cudaStream_t s) {
    SimtKernelArgs k{};
    k.x = a.x;
    k.wq = reinterpret_cast<const uint4*>(a.wq);
    k.scale = a.scale;
    k.zero = a.zero;
    k.y = a.y;
    k.out_f32 = a.out_f32;
    k.N = a.N;
    k.K = a.K;
    k.g = a.g;
    k.wpt = p.wpt;
    k.ksplit = p.k_split;
    k.spans_per_cta = p.units_per_cta;
    k.tiles_per_group = p.tiles_per_cluster;
    k.stages = p.stages;
    k.weights_static = a.weights_static;
    k.err = a.err;
    SimtKernel kern = pick_simt_kernel(a.M, p.tile_rows, a.K, a.g);
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
    return cudaLaunchKernelEx(&cfg, kern, k);
}

}  // namespace w4a16
