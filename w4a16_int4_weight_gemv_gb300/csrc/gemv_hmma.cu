// Dense W4A16 GEMV for 1..16 tokens on warp MMA with fp16 operands (sm_103a).
//
// The decode-time product of the local-kimi README, technical-detail section:
// a true GEMV with K contiguous, every output row one fp32 accumulation.
//
// Why the tensor pipe for a GEMV.  On sm_103a the integer/logic pipe issues
// at half rate (16 lanes per SMSP and clock): turning a packed word into
// operands costs one LOP3 per code on the CUDA cores (each fp32 operand holds
// one code), which alone needs ~85 % of that pipe at HBM speed.  An fp16 pair
// holds two codes, so feeding the codes to the tensor pipe as the A operand of
// mma.sync.m16n8k16 halves that work, and the multiply-adds leave the CUDA
// cores altogether; the tokens are the B operand (8 columns, 1..8 used;
// 9..16 tokens are two such tiles sharing every A operand).
//
// Dequantisation.  (w & 0x000F000F) | 0x64006400 is the fp16 pair
// {1024 + q0, 1024 + q4} and (w & 0x00F000F0) | 0x64006400 the pair
// {1024 + 16 q1, 1024 + 16 q5}; the same two LOP3s on w >> 8 give codes 2, 6
// and 3, 7 -- five logic instructions per word of eight codes.  The factor 16
// of the odd codes is taken out of the activations (their B entries are x/16),
// so every product A*B is 1024 B + q x' exactly, and for each 128-k block (one
// quantisation group, g == 128)
//     sum_k (q_k - z) x'_k = D - 1024 sum_k B_k - z sum_k x'_k,
// with D the block's MMA sum; the scale multiplies that once per block.
//
// Activations.  Each CTA converts its K slice of x once, after the
// grid-dependency wait, in one pass: every 128-k block of every token gets
// its own power of two, x' = x * 2^sh with the block's largest |x| landing in
// [2^14, 2^15) (fp16 holds it and every element within 2^24 of it exactly),
// is rounded to fp16 and stored in the order the B fragments are read: one
// 16-byte load per lane and chunk gives the four B registers of two MMAs.
// Beside the fragments go the block sums of the rounded values (c1 = 1024
// sum B, c2 = sum x') and 2^-sh, which multiplies the scale in the epilogue.
//
// Memory path.  A unit is one 16-row tile x 512 k.  Every warp streams its
// own units through its own ring of `depth` stages with 16-byte cp.async
// copies -- the 256 packed bytes of each row as one aligned 256-byte block,
// its 16-byte chunks XOR-swizzled by the row so that ldmatrix reads the
// eight rows of a chunk from eight bank groups (measured 3-8 % faster than
// a padded 272-byte pitch, whose rows split every copied line across two
// lines of shared memory), then the tile's zero points and scales -- one
// commit group per unit, waited for with cp.async.wait_group.  The whole
// ring is filled before the loop and a stage is refilled as soon as it is
// consumed, so a warp with at most `depth` units has them all in flight at
// once and a longer one keeps depth - 1 in flight while it computes.  (The
// copy engine is not used: a bulk or tensor copy costs its issuing warp tens
// of nanoseconds on sm_103a, and with the weights split over many such
// copies the issue time outweighs the arithmetic.)
//
// Work split.  The CTAs of a cluster share a range of 16-row tiles, rank r
// taking the r-th K slice; inside the CTA, WPT warps share a tile, warp part
// p taking K steps p, p + WPT, ...; tile groups take the CTA's tiles in turn.
// The other parts hand their partials to part 0 through double-buffered
// shared memory guarded by mbarriers (every wait bounded), and part 0 adds
// them in part order; ranks push their tile sums into the owner's shared
// memory and the owner adds them in rank order after a cluster barrier --
// fixed orders, so results are deterministic.
//
// Launch.  The rings are sized so that two CTAs fit on an SM where possible:
// with programmatic dependent launch the next GEMV's CTA becomes resident
// while this one runs, and with W4A16_FLAG_WEIGHTS_STATIC it requests its
// first units before the grid-dependency wait.
#include <cuda_fp16.h>

#include "common.cuh"
#include "hmma_core.cuh"
#include "launch.h"

namespace w4a16 {
namespace {

constexpr int kSZScales = 64;

struct HmmaKernelArgs {
    const uint16_t* x;
    const unsigned char* wq;  // packed words as bytes, row pitch K / 2
    const uint16_t* scale;
    const uint8_t* zero;
    void* y;
    int out_f32;
    int M;
    int N;
    int K;
    int S;               // CTAs per cluster (K split)
    int nclusters;       // tile ranges
    int steps_per_rank;  // 512-k steps per K slice
    int max_tiles;       // most tiles one cluster owns
    int wpt;             // warps per tile
    int depth;           // stages per warp
    int weights_static;
    int swiglu_out;      // rows 16t..+7 gate, 16t+8..+15 up: y = bf16 SwiGLU [M][N/2]
    uint32_t* err;       // device error word (W4A16_DEVERR_TIMEOUT)
};


// Store the C-fragment values of lane l for 16-row tile `tile`: rows
// 16 tile + l / 4 (x, y) and + 8 (z, w), tokens 2 (l % 4) (x, z) and + 1 (y, w).
// The SwiGLU form: rows g and g + 8 of the tile are gate and up row
// 8 tile + g (every tile is whole: N % 16 == 0).  Kept out of line so that
// its exponentials do not add to the main loop's register pressure.
__device__ __noinline__ void store_swiglu_fragment(uint16_t* y, int M, int N, int tile, int l,
                                                   float4 v, int tok0) {
    const int g = l >> 2, c = tok0 + 2 * (l & 3);
    const size_t nh = static_cast<size_t>(N >> 1);
    const size_t hr = static_cast<size_t>(tile) * 8 + g;
    if (c < M) y[c * nh + hr] = swiglu_of_sums(v.x, v.z);
    if (c + 1 < M) y[(c + 1) * nh + hr] = swiglu_of_sums(v.y, v.w);
}

// tok0: the first token of the 8-token MMA tile the fragment belongs to
__device__ __forceinline__ void store_fragment(const HmmaKernelArgs& a, int tile, int l, float4 v,
                                               int tok0) {
    if (a.swiglu_out) {
        store_swiglu_fragment(static_cast<uint16_t*>(a.y), a.M, a.N, tile, l, v, tok0);
        return;
    }
    const int g = l >> 2, c = tok0 + 2 * (l & 3);
    const int ra = (tile << 4) + g;
    const int rb = ra + 8;
    if (c < a.M) {
        const size_t o = static_cast<size_t>(c) * a.N;
        if (ra < a.N) store_out(a.y, a.out_f32, o + ra, v.x);
        if (rb < a.N) store_out(a.y, a.out_f32, o + rb, v.z);
    }
    if (c + 1 < a.M) {
        const size_t o = static_cast<size_t>(c + 1) * a.N;
        if (ra < a.N) store_out(a.y, a.out_f32, o + ra, v.y);
        if (rb < a.N) store_out(a.y, a.out_f32, o + rb, v.w);
    }
}


// MP: the token count rounded up to 1, 2, 4, 8 or 16 -- the B fragments are
// stored for MP tokens (the columns of tokens M..MP-1 are never stored, so
// their contents do not matter); 16 tokens are two 8-column MMA tiles that
// share every A operand.  W warps per CTA
template <int MP, int W>
__global__ void __launch_bounds__(32 * W, W == kHmmaWarpsPaired && MP <= 8 ? 2 : 1)
    k_gemv_hmma(const HmmaKernelArgs a) {
    constexpr int kThreads = 32 * W;
    constexpr int NT = MP > 8 ? 2 : 1;       // 8-token MMA tiles
    constexpr int CSP = MP > 8 ? MP / 2 : 4;  // token pairs per block in the sums
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int S = a.S;
    const int rank = (S > 1) ? static_cast<int>(cluster_rank()) : 0;
    const int cid = blockIdx.x / S;
    const int ntiles = (a.N + 15) >> 4;
    const int t0 = static_cast<int>(static_cast<long long>(ntiles) * cid / a.nclusters);
    const int t1 = static_cast<int>(static_cast<long long>(ntiles) * (cid + 1) / a.nclusters);
    const int nt = t1 - t0;
    const int nsr = a.steps_per_rank;  // S divides K / 512: every rank has them all
    const int s0 = rank * nsr;
    const int M = a.M;
    const int G = a.K >> 7;
    const int WPT = a.wpt;
    const int NG = W / WPT;
    const int grp = warp / WPT;
    const int part = warp - grp * WPT;
    const int D = a.depth;

    const uint32_t raw = smem_addr(smem_raw);
    unsigned char* base = smem_raw + (((raw + 127u) & ~127u) - raw);
    const HmmaLayout L = hmma_layout(W, MP, nsr, S, a.max_tiles, D);
    unsigned char* ring = base + L.ring + warp * D * kHmmaStage;
    uint4* bfrag = reinterpret_cast<uint4*>(base + L.bfrag);
    float* csum = reinterpret_cast<float*>(base + L.csum);
    float4* red = reinterpret_cast<float4*>(base + L.red);
    float4* cpart = reinterpret_cast<float4*>(base + L.cpart);
    uint64_t* gbar = reinterpret_cast<uint64_t*>(base + L.bars);
    if (WPT > 1 && threadIdx.x < NG * 2) {
        // buffer b of group g: `full` completes when the group's other parts
        // have written their partials, `empty` when part 0 has read them
        mbar_init(gbar + threadIdx.x * 2, (WPT - 1) * 32);
        mbar_init(gbar + threadIdx.x * 2 + 1, 32);
    }

    // this warp's units: tiles grp, grp + NG, ... of the CTA, K steps part,
    // part + WPT, ... of the slice
    const int my_tiles = (nt > grp) ? (nt - grp + NG - 1) / NG : 0;
    const int my_steps = (nsr > part) ? (nsr - part + WPT - 1) / WPT : 0;
    const int nu = my_tiles * my_steps;

    grid_dependents_launch();
    if (S > 1) cluster_arrive_relaxed();

    // Producer side of this warp's ring: unit (i_tile, i_step) into stage
    // i_slot as one commit group.  Lane l copies the 16-byte chunks
    // (row 2 i + l / 16, chunk l % 16), i = 0..7, so each copy instruction
    // reads two whole 256-byte row pieces; lanes 0..15 then copy the 4 zero
    // points of row l, lanes 16..31 its 4 scales.  In the stage, chunk c of
    // row r sits at chunk c ^ (r & 7) of the row's 256 bytes: every row is
    // one aligned 256-byte block (a copy instruction fills two of them, with
    // no line of the copy split across two lines of shared memory), and the
    // eight rows an ldmatrix phase reads for one chunk fall in eight bank
    // groups.  For row 2 i + h the swizzle is (c ^ h) ^ 2 (i & 3), so four
    // lane offsets serve the eight copies.
    const size_t row_bytes = static_cast<size_t>(a.K) >> 1;
    const size_t src_lane = static_cast<size_t>(lane >> 4) * row_bytes + (lane & 15) * 16;
    const int sw_h = lane >> 4, sw_c = ((lane & 15) ^ sw_h) << 4;
    const int dl0 = sw_h * kHmmaRowPitch + sw_c, dl1 = sw_h * kHmmaRowPitch + (sw_c ^ 32);
    const int dl2 = sw_h * kHmmaRowPitch + (sw_c ^ 64), dl3 = sw_h * kHmmaRowPitch + (sw_c ^ 96);
    auto dst_off = [&](int i) {  // copy i (compile-time): row 2 i + h
        return ((i & 3) == 0 ? dl0 : (i & 3) == 1 ? dl1 : (i & 3) == 2 ? dl2 : dl3) +
               i * 2 * kHmmaRowPitch;
    };
    const int rr = lane & 15;
    int i_u = 0, i_slot = 0, i_tile = t0 + grp, i_step = part;
    auto issue_next = [&]() {
        if (i_u < nu) {
            const int row0 = i_tile << 4;
            const int rows = min(16, a.N - row0);
            const int step = s0 + i_step;
            unsigned char* stage = ring + i_slot * kHmmaStage;
            const unsigned char* src = a.wq + static_cast<size_t>(row0) * row_bytes + step * 256 + src_lane;
            if (rows == 16) {
#pragma unroll
                for (int i = 0; i < 8; ++i) cp_async_16(stage + dst_off(i), src + i * 2 * row_bytes);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (2 * i + (lane >> 4) < rows) cp_async_16(stage + dst_off(i), src + i * 2 * row_bytes);
            }
            if (rr < rows) {
                const size_t gi = static_cast<size_t>(row0 + rr) * G + step * 4;
                if (lane < 16) cp_async_4(stage + kHmmaUnitBytes + rr * 4, a.zero + gi);
                else cp_async_8(stage + kHmmaUnitBytes + kSZScales + rr * 8, a.scale + gi);
            }
            ++i_u;
            if (++i_slot == D) i_slot = 0;
            i_step += WPT;
            if (i_step >= nsr) {
                i_step = part;
                i_tile += NG;
            }
        }
        cp_async_commit();  // one group per call, empty past the end
    };
    // the ring is filled whole before the loop (a warp with few units has
    // them all in flight at once); with static weights this happens before
    // the preceding grid completes
    if (a.weights_static)
        for (int k = 0; k < D; ++k) issue_next();
    grid_dependency_wait();

    {
        if constexpr (MP == 1) {
            // Activations of one token (measured 2 % faster on the 4096 x 4096
            // GEMV than the 16-k items below): every (token, round) item of
            // this thread is one 8-k piece; the loads of
            // up to four items are issued before any is converted, so the latency
            // is paid once per four -- and the first four are issued before the
            // weight copies.  The 16 pieces of a block are 16 consecutive lanes
            // (block max and sums by shuffles).
            const int tid = threadIdx.x;
            constexpr int T = kThreads;
            const int nblk = nsr * 4;       // 128-k blocks of the slice
            const int npieces = nblk * 16;  // 8-k pieces per token
            const int nrounds = (npieces + T - 1) / T;
            const int items = M * nrounds;
            const uint16_t* xs = a.x + static_cast<size_t>(s0) * 512;
            auto load_items = [&](int it0, uint4 (&v)[4]) {
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    const int it = it0 + b;
                    const int m = it / nrounds;
                    const int p = (it - m * nrounds) * T + tid;
                    v[b] = make_uint4(0u, 0u, 0u, 0u);
                    if (it < items && p < npieces)
                        v[b] = __ldg(reinterpret_cast<const uint4*>(xs + static_cast<size_t>(m) * a.K + p * 8));
                }
            };
            uint4 v[4];
            load_items(0, v);
            if (!a.weights_static)
                for (int k = 0; k < D; ++k) issue_next();
            for (int it0 = 0; it0 < items; it0 += 4) {
                if (it0 > 0) load_items(it0, v);
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    const int it = it0 + b;
                    if (it >= items) break;  // the same for the whole CTA
                    const int m = it / nrounds;
                    const int p = (it - m * nrounds) * T + tid;
                    const uint32_t w[4] = {v[b].x, v[b].y, v[b].z, v[b].w};
                    uint32_t mx = 0u;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        mx = max(mx, w[e] & 0x7FFFu);
                        mx = max(mx, (w[e] >> 16) & 0x7FFFu);
                    }
#pragma unroll
                    for (int o = 1; o < 16; o <<= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                    const int sh = block_shift(mx);
                    float fa, fb;
                    pow2_pair(sh, fa, fb);
                    const float fo = fb * 0.0625f;  // odd codes: B = x' / 16
                    uint32_t h[8];
                    float c1 = 0.f, c2 = 0.f;
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const uint32_t bits = (e & 1) ? (w[e >> 1] & 0xFFFF0000u) : (w[e >> 1] << 16);
                        const float xv = __uint_as_float(bits) * fa;
                        const __half hv = __float2half_rn((e & 1) ? xv * fo : xv * fb);
                        h[e] = __half_as_ushort(hv);
                        const float bv = __half2float(hv);
                        c1 += bv;
                        c2 += (e & 1) ? 16.f * bv : bv;
                    }
#pragma unroll
                    for (int o = 1; o < 16; o <<= 1) {
                        c1 += __shfl_xor_sync(0xffffffffu, c1, o);
                        c2 += __shfl_xor_sync(0xffffffffu, c2, o);
                    }
                    if (p < npieces) {
                        const int blk = p >> 4, j = (p >> 2) & 3, q = p & 3;
                        uint4 o4;
                        o4.x = h[0] | (h[4] << 16);  // MMA 1, b0: codes 0, 4
                        o4.y = h[1] | (h[5] << 16);  // MMA 1, b1: codes 1, 5 (x/16)
                        o4.z = h[2] | (h[6] << 16);  // MMA 2, b0: codes 2, 6
                        o4.w = h[3] | (h[7] << 16);  // MMA 2, b1: codes 3, 7 (x/16)
                        bfrag[((blk * 4 + j) * MP + m) * 4 + q] = o4;
                        if ((p & 15) == 0) {
                            float* cs = csum + (blk * CSP + (m >> 1)) * 8;
                            cs[m & 1] = 1024.f * c1;
                            cs[2 + (m & 1)] = c2;
                            cs[4 + (m & 1)] = exp2i(-sh);
                        }
                    }
                }
            }
        } else {
            // Activations: one item is two 8-k pieces (16 k) of one token's K
            // slice (pieces l and l + 8 of a 128-k block, l = 0..7); the 8 items
            // of a block are 8 consecutive lanes, which share the block's maximum
            // and sums by shuffles.  Four items per
            // thread are in flight: the first four are loaded before the weight
            // copies are issued (loads issued after them wait behind the weight
            // stream), and each item's slot is refilled four items ahead as soon
            // as it is converted.
            const int tid = threadIdx.x;
            constexpr int T = kThreads;
            const int nit = nsr * 32;  // items per token of the slice
            const int nflat = M * nit;
            const int items = (nflat + T - 1) / T;
            const uint16_t* xs = a.x + static_cast<size_t>(s0) * 512;
            auto load_item = [&](int it, uint4 (&v)[2]) {
                const int f = it * T + tid;
                v[0] = v[1] = make_uint4(0u, 0u, 0u, 0u);
                if (it < items && f < nflat) {
                    const int m = f / nit, r = f - m * nit;
                    // pieces l and l + 8 of block r / 8 (l = r % 8)
                    const uint4* src = reinterpret_cast<const uint4*>(xs + static_cast<size_t>(m) * a.K) +
                                       (r >> 3) * 16 + (r & 7);
                    v[0] = __ldg(src);
                    v[1] = __ldg(src + 8);
                }
            };
            uint4 v[4][2];
#pragma unroll
            for (int b = 0; b < 4; ++b) load_item(b, v[b]);
            if (!a.weights_static)
                for (int k = 0; k < D; ++k) issue_next();
            for (int it0 = 0; it0 < items; it0 += 4) {
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    const int it = it0 + b;
                    if (it >= items) break;  // the same for the whole CTA
                    const int f = it * T + tid;
                    uint32_t mx = pieces_absmax<2>(v[b]);
#pragma unroll
                    for (int o = 1; o < 8; o <<= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                    const int sh = block_shift(mx);
                    float fa, fb;
                    pow2_pair(sh, fa, fb);
                    uint4 o2[2];
                    float c1 = 0.f, c2 = 0.f;
                    int4_piece_fragments<2>(v[b], fa, fb, o2, c1, c2);
                    load_item(it + 4, v[b]);
#pragma unroll
                    for (int o = 1; o < 8; o <<= 1) {
                        c1 += __shfl_xor_sync(0xffffffffu, c1, o);
                        c2 += __shfl_xor_sync(0xffffffffu, c2, o);
                    }
                    if (f < nflat) {
                        const int m = f / nit, r = f - m * nit;
                        // piece p = 16 blk + l: chunk l / 4 of the block, word l % 4
                        const int blk = r >> 3, l = r & 7;
                        bfrag[((blk * 4 + (l >> 2)) * MP + m) * 4 + (l & 3)] = o2[0];
                        bfrag[((blk * 4 + (l >> 2) + 2) * MP + m) * 4 + (l & 3)] = o2[1];
                        if (l == 0) {
                            float* cs = csum + (blk * CSP + (m >> 1)) * 8;
                            cs[m & 1] = 1024.f * c1;
                            cs[2 + (m & 1)] = c2;
                            cs[4 + (m & 1)] = exp2i(-sh);
                        }
                    }
                }
            }
        }
    }
    __syncthreads();
    if (S > 1) cluster_wait();  // every peer CTA has started: remote stores are safe

    const int g = lane >> 2, c = lane & 3;
    // ldmatrix addressing: lane l supplies row (l & 7) + 8 ((l >> 3) & 1) of
    // chunk 4 bb + t + (l >> 4) (t = 0, then 2 for the second load); with
    // s = l & 7 (the row's swizzle), bits 0..2 of that chunk index flip with
    // those of s and bit 3 (bb >> 1) is left alone, so four lane offsets
    // lv[t / 2 + 2 (bb & 1)] plus 128 (bb >> 1) cover the eight loads
    const int lrow = (lane & 7) + (((lane >> 3) & 1) << 3);
    const int lch = lane >> 4;
    const int sw_s = lane & 7;
    const uint32_t ring_addr = smem_addr(ring) + static_cast<uint32_t>(lrow * kHmmaRowPitch);
    const uint32_t lve = (lch ^ (sw_s & 1)) << 4;
    const uint32_t lv0 = lve + ((0 ^ (sw_s & 2)) << 4) + ((0 ^ (sw_s & 4)) << 4);
    const uint32_t lv1 = lve + ((2 ^ (sw_s & 2)) << 4) + ((0 ^ (sw_s & 4)) << 4);
    const uint32_t lv2 = lve + ((0 ^ (sw_s & 2)) << 4) + ((4 ^ (sw_s & 4)) << 4);
    const uint32_t lv3 = lve + ((2 ^ (sw_s & 2)) << 4) + ((4 ^ (sw_s & 4)) << 4);
    // B fragments of token g (+ 8 t for MMA tile t; padding-token lanes read
    // token 0's: their output columns are never stored) and the block sums of
    // tokens 2c, 2c + 1 (+ 8 t)
    const uint4* bq_lane[NT];
    const float* cs_lane[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        bq_lane[t] = bfrag + (g + 8 * t < M ? g + 8 * t : 0) * 4 + c;
        cs_lane[t] = csum + (c + 4 * t) * 8;
    }

    float4 tacc[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) tacc[t] = make_float4(0.f, 0.f, 0.f, 0.f);
    bool timed_out = false;  // a bounded wait for a partner's partials expired
    int c_slot = 0, c_step = part, c_tile = 0, ti = 0;  // c_tile: local tile of the group
#pragma unroll 1
    for (int k = 0; k < nu; ++k) {
        cp_async_wait_pending(D - 1);  // units k + 1 .. k + D - 1 may be in flight
        __syncwarp();  // every lane's copies of unit k have landed
        const int slot = c_slot;
        const int lstep = c_step;
        if (++c_slot == D) c_slot = 0;
        const uint32_t wst = ring_addr + static_cast<uint32_t>(slot * kHmmaStage);
        const unsigned char* sz = ring + slot * kHmmaStage + kHmmaUnitBytes;
        const uint32_t za = *reinterpret_cast<const uint32_t*>(sz + g * 4);
        const uint32_t zb = *reinterpret_cast<const uint32_t*>(sz + (g + 8) * 4);
        const uint2 sa = *reinterpret_cast<const uint2*>(sz + kSZScales + g * 8);
        const uint2 sb = *reinterpret_cast<const uint2*>(sz + kSZScales + (g + 8) * 8);
        float acc[NT][4];
#pragma unroll
        for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
#pragma unroll
        for (int bb = 0; bb < 4; ++bb) {
            const uint32_t hb = wst + static_cast<uint32_t>((bb >> 1) * 128);
            uint32_t q0[4], q1[4];
            ldmatrix_x4(q0, hb + ((bb & 1) ? lv2 : lv0));
            ldmatrix_x4(q1, hb + ((bb & 1) ? lv3 : lv1));
            const uint32_t wa[4] = {q0[0], q0[2], q1[0], q1[2]};  // row g, chunks 0..3
            const uint32_t wb[4] = {q0[1], q0[3], q1[1], q1[3]};  // row g + 8
            // two accumulator chains per MMA tile: codes 0/4 + 1/5 and codes
            // 2/6 + 3/7; the A operands of a chunk serve every tile
            float d0[NT][4], d1[NT][4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t ta = wa[j] >> 8, tb = wb[j] >> 8;
                const uint32_t a0 = f16_codes_lo(wa[j]), a1 = f16_codes_lo(wb[j]);
                const uint32_t a2 = f16_codes_hi(wa[j]), a3 = f16_codes_hi(wb[j]);
                const uint32_t e0 = f16_codes_lo(ta), e1 = f16_codes_lo(tb);
                const uint32_t e2 = f16_codes_hi(ta), e3 = f16_codes_hi(tb);
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    const uint4 bq = bq_lane[t][((lstep * 16) + bb * 4 + j) * MP * 4];
                    if (j == 0) {
                        mma_f16_16816_zero(d0[t], a0, a1, a2, a3, bq.x, bq.y);
                        mma_f16_16816_zero(d1[t], e0, e1, e2, e3, bq.z, bq.w);
                    } else {
                        mma_f16_16816(d0[t], a0, a1, a2, a3, bq.x, bq.y);
                        mma_f16_16816(d1[t], e0, e1, e2, e3, bq.z, bq.w);
                    }
                }
            }
            const float zfa = zero_point_f32(za, bb), zfb = zero_point_f32(zb, bb);
            const uint32_t swa = (bb < 2) ? sa.x : sa.y, swb = (bb < 2) ? sb.x : sb.y;
            const float sfa = __uint_as_float((bb & 1) ? (swa & 0xFFFF0000u) : (swa << 16));
            const float sfb = __uint_as_float((bb & 1) ? (swb & 0xFFFF0000u) : (swb << 16));
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                const float* csb = cs_lane[t] + (lstep * 4 + bb) * CSP * 8;
                const float4 cs = *reinterpret_cast<const float4*>(csb);
                const float2 fs = *reinterpret_cast<const float2*>(csb + 4);
                // token 2c in x/z, 2c + 1 in y/w; with one token only the former
                acc[t][0] = fmaf(sfa * fs.x, (d0[t][0] + d1[t][0]) - fmaf(zfa, cs.z, cs.x), acc[t][0]);
                acc[t][2] = fmaf(sfb * fs.x, (d0[t][2] + d1[t][2]) - fmaf(zfb, cs.z, cs.x), acc[t][2]);
                if (MP > 1) {
                    acc[t][1] = fmaf(sfa * fs.y, (d0[t][1] + d1[t][1]) - fmaf(zfa, cs.w, cs.y), acc[t][1]);
                    acc[t][3] = fmaf(sfb * fs.y, (d0[t][3] + d1[t][3]) - fmaf(zfb, cs.w, cs.y), acc[t][3]);
                }
            }
        }
        __syncwarp();  // every lane is done with the stage before it is refilled
        issue_next();  // unit k + D into the stage just consumed
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            tacc[t].x += acc[t][0];
            tacc[t].z += acc[t][2];
            if (MP > 1) {
                tacc[t].y += acc[t][1];
                tacc[t].w += acc[t][3];
            }
        }
        c_step += WPT;
        if (c_step < nsr) continue;
        c_step = part;
        // the tile's part is complete: the other parts hand their partials
        // to part 0 and go on (they wait only to reuse a buffer part 0 has not
        // read yet); part 0 adds them in part order, then stores or pushes
        const int tile = t0 + grp + c_tile * NG;
        if (WPT > 1) {
            if (part != 0) {
                timed_out |= !hand_partials<W, NT>(red, gbar, grp, WPT, part, ti, lane, tacc);
            } else {
                const int b = ti & 1;
                uint64_t* full = gbar + (grp * 2 + b) * 2;
                timed_out |= !mbar_wait_bounded(full, (ti >> 1) & 1);
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    const float4* rb = red + t * 2 * W * 32 + (b * W + grp * WPT) * 32;
                    for (int q = 1; q < WPT; ++q) {
                        const float4 v = rb[q * 32 + lane];
                        tacc[t].x += v.x;
                        tacc[t].y += v.y;
                        tacc[t].z += v.z;
                        tacc[t].w += v.w;
                    }
                }
                mbar_arrive(full + 1);
            }
        }
        if (part == 0) {
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                if (S == 1) {
                    store_fragment(a, tile, lane, tacc[t], 8 * t);
                } else {
                    const int tl = tile - t0;
                    st_dsmem_f32x4(reinterpret_cast<float*>(cpart + ((t * a.max_tiles + tl) * S + rank) * 32 + lane),
                                   static_cast<uint32_t>(tl % S), tacc[t]);
                }
            }
        }
#pragma unroll
        for (int t = 0; t < NT; ++t) tacc[t] = make_float4(0.f, 0.f, 0.f, 0.f);
        ++c_tile;
        ++ti;
    }
    // a part with no K step still hands part 0 a (zero) partial per tile
    if (WPT > 1 && my_steps == 0)
        for (; ti < my_tiles; ++ti)
            timed_out |= !hand_partials<W, NT>(red, gbar, grp, WPT, part, ti, lane, tacc);
    cp_async_wait_pending(0);
    if (timed_out && lane == 0) raise_device_error(a.err, W4A16_DEVERR_TIMEOUT);

    // K split over the cluster: every rank pushed its tile sums into the owner
    // (tile % S); after the barrier the owner adds them in rank order
    if (S > 1) {
        cluster_barrier();
        for (int idx = threadIdx.x; idx < NT * nt * 32; idx += blockDim.x) {
            const int t = idx / (nt * 32);
            const int tl = (idx >> 5) - t * nt, l = idx & 31;
            if (tl % S != rank) continue;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int q = 0; q < S; ++q) {
                const float4 pv = cpart[((t * a.max_tiles + tl) * S + q) * 32 + l];
                v.x += pv.x;
                v.y += pv.y;
                v.z += pv.z;
                v.w += pv.w;
            }
            store_fragment(a, t0 + tl, l, v, 8 * t);
        }
    }
}

using HmmaKernel = void (*)(HmmaKernelArgs);
template <int W>
HmmaKernel hmma_kernel_w(int M) {
    return M <= 1 ? k_gemv_hmma<1, W>
           : M <= 2 ? k_gemv_hmma<2, W>
           : M <= 4 ? k_gemv_hmma<4, W>
           : M <= 8 ? k_gemv_hmma<8, W>
                    : k_gemv_hmma<16, W>;
}
HmmaKernel hmma_kernel(int M, int warps) {
    return warps == kHmmaWarpsWide ? hmma_kernel_w<kHmmaWarpsWide>(M) : hmma_kernel_w<kHmmaWarpsPaired>(M);
}
// tokens rounded up to the instantiated count
int hmma_mp(int M) { return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : M <= 8 ? 8 : 16; }

}  // namespace

GemvPlan plan_gemv_hmma(const DeviceInfo& dev, int M, int N, int K, int g, int k_split_req) {
    GemvPlan p{};
    p.kernel_id = 4;
    if (!hmma_supports(M, K, g)) return p;
    const void* k8 = reinterpret_cast<const void*>(hmma_kernel(M, kHmmaWarpsPaired));
    const void* k16 = reinterpret_cast<const void*>(hmma_kernel(M, kHmmaWarpsWide));
    const HmmaChoice c = choose_hmma_plan(
        dev, hmma_mp(M), N, K, k_split_req,
        [k8](int S, int smem) { return max_active_clusters(k8, 32 * kHmmaWarpsPaired, smem, S); },
        [k16](int S, int smem) { return max_active_clusters(k16, 32 * kHmmaWarpsWide, smem, S); });
    if (c.nclusters < 1) return p;
    p.k_split = c.S;
    p.wpt = c.wpt;
    p.units_per_cta = c.steps_per_rank;
    p.threads = 32 * c.warps;
    p.ctas = c.nclusters * c.S;
    p.stages = c.depth;
    p.smem_bytes = c.smem_bytes;
    p.nclusters = c.nclusters;
    p.max_tiles = c.max_tiles;
    p.tiles_per_cluster = c.max_tiles;
    p.tile_rows = 16;
    return p;
}

cudaError_t launch_gemv_hmma(const GemvArgs& a, const GemvPlan& p, cudaStream_t s) {
    HmmaKernelArgs k{};
    k.x = a.x;
    k.wq = reinterpret_cast<const unsigned char*>(a.wq);
    k.scale = a.scale;
    k.zero = a.zero;
    k.y = a.y;
    k.out_f32 = a.out_f32;
    k.M = a.M;
    k.N = a.N;
    k.K = a.K;
    k.S = p.k_split;
    k.nclusters = p.nclusters;
    k.steps_per_rank = p.units_per_cta;
    k.max_tiles = p.max_tiles;
    k.wpt = p.wpt;
    k.depth = p.stages;
    k.weights_static = a.weights_static;
    k.swiglu_out = a.swiglu_out;
    k.err = a.err;
    const HmmaKernel kern = hmma_kernel(a.M, p.threads / 32);
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
