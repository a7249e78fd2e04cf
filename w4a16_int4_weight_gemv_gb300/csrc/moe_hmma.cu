// Routed SwiGLU expert FFN of 1..8 tokens on the fp16 warp-MMA path (g ==
// 128): the grouped expert kernel of the local-kimi README (technical-detail
// section), as two launches; the second also serves alone as the expert-
// indexed GEMV (below).
//
//   1. gate/up: for every distinct routed expert e, the gate and up products
//      of all tokens, h[t][j] = bf16(silu(bf16(W^gate_e x[t])) *
//      bf16(W^up_e x[t])) stored for every slot (t, j) routed to e.
//   2. down: a CTA owns 16-row tiles of the output and computes, for every
//      routed slot, d[t][j] = W^down_e h[t][j] on them (fp32, in shared
//      memory), then y[t] = bf16(sum_j route_w[t][j] d[t][j]) (j ascending,
//      invalid ids skipped) -- no partials leave the CTA.
//
// Both launches share one design with the dense fp16 warp-MMA GEMV: a 16-row
// tile of weights is the A operand of mma.sync m16n8k16, the codes become
// fp16 with one LOP3 per two (1024 + code, the 16x scaling of odd codes
// folded into B), the activations are staged per CTA as fp16 B fragments
// with each 128-k block scaled by a power of two, units of 16 rows x 512 k
// stream through per-warp cp.async rings, and parts of a split tile hand
// their partials to part 0.  What differs:
//
// Tiles.  Warp 0 routes once per CTA: the distinct valid experts in order
// of first appearance among the M * topk slots (<= 32).  A launch-1 tile
// pairs gate rows 8r..8r+7 (tile rows 0..7) with the same up rows (tile rows
// 8..15) of one expert, so a lane holds a gate and its up row and forms h in
// the epilogue; its B columns are the M tokens.  A launch-2 tile is 16 rows
// of one expert's down matrix; its B columns are that expert's routed slots
// (an "entry": up to 8 slots; an expert with more slots has several
// entries), and a CTA's warps take the entries of its row tiles in turn,
// each entry's K steps in one warp.  Every tile column the MMA computes
// beyond the real ones is free.
//
// Partial steps.  K need not be a multiple of 512 (the FFN's H = 2304 is
// 4.5 steps): the last unit of a row carries 1..3 blocks, copied and used
// block by block.  The zero points and scales of a unit are copied from the
// 4-byte-aligned words around them (their rows start at any byte, g = 128
// giving K / 128 groups per row), zero-filled past the end of the arrays,
// and picked out with funnel shifts.
//
// Launch.  Launch 2 reads the routing and its weights before its
// grid-dependency wait; launch 1 signals its dependents only after its own
// wait, so everything launch 2 reads early was complete before launch 1 ran.
//
// Expert GEMV.  Launch 2 alone (template flag ALONE) is an expert-indexed
// GEMV: d[t][j] = W_e x_in for every routed slot, x_in a row per slot or per
// token.  It reads nothing before its wait and flags invalid ids itself.
// Slots that share a token row share one staged B column (tile columns are
// slots, their B and sums are looked up through slot / topk).  With route
// weights the routed sums are formed as in the FFN; per-slot outputs are
// stored from registers as each tile completes, and when N / 16 row tiles
// are fewer than the SMs the (row tile, entry) tiles are dealt evenly over
// all CTAs instead (a 1024-row expert has 64 row tiles).
//
// ~3-bit experts (BITS == 3; the README's hardware-requirements paragraph
// asks for expert weights near three bits, the INT3 format is this
// library's: a chunk of 32 codes in three words, five 3-bit fields in each
// 16-bit half at bits 0, 3, 6, 9, 12, codes 30 and 31 in the spare bits 15
// and 31).  The same kernel with another unit format: a row of a unit is
// 192 bytes (4 groups x 48), staged at a 208-byte pitch so that the 32-bit
// reads of 8 rows x 4 chunks hit 32 different banks; lane (g, c) reads
// chunk c of each 128-k block of rows g and g + 8 (three words each) and
// makes the 16 fp16 pairs of a row with one LOP3 each -- fields at bits 0,
// 3, 6 of a word give 1024 + q, 1024 + 8q, 1024 + 64q, the same masks on
// the word shifted right by 9 give the fields at 9 and 12, and three LOP3s
// gather the spare bits into {1024 + q30, 1024 + q31}: 24 ALU operations per
// 32 codes.  B holds x / 1, x / 8 or x / 64 to match; the eight MMAs of a
// block take pairs (2m, 2m + 1) as their two k halves.
#include <cuda_fp16.h>

#include "common.cuh"
#include "hmma_core.cuh"
#include "launch.h"
#include "moe_hmma_gemv.h"

namespace w4a16 {
namespace {

// warps per CTA: 16, or 8 (two CTAs to an SM) where 16 do not fit
constexpr int kMWPaired = 8;
constexpr int kMWWide = 16;
constexpr int kMMaxDepth = 4;
// A stage holds one unit (16 rows x 512 k): the weight rows at m_pitch
// bytes each, then 16 rows x 8 zero-point bytes and 16 rows x 16 scale
// bytes.  INT4: 256-byte rows, 16-byte chunks XOR-swizzled by the row; INT3:
// 192-byte rows at a 208-byte pitch.
__host__ __device__ constexpr int m_pitch(int bits) { return bits == 4 ? kHmmaRowPitch : 208; }
__host__ __device__ constexpr int m_zero(int bits) { return 16 * m_pitch(bits); }
__host__ __device__ constexpr int m_scale(int bits) { return m_zero(bits) + 128; }
__host__ __device__ constexpr int m_stage(int bits) { return m_zero(bits) + 384; }
static_assert(m_zero(4) == kHmmaUnitBytes && m_stage(3) % 16 == 0, "stage layout");

struct MoeHK {
    int phase;                 // 1: gate/up -> h; 2: down -> routed sums
    const uint16_t* x;         // launch 1: x [M][K]; launch 2: h [M*topk][K]
    const int32_t* ids;        // [M][topk]
    const float* route_w;      // [M][topk] (launch 2)
    const unsigned char* wq_a;  // launch 1: gate bank, launch 2: down bank
    const uint16_t* scale_a;
    const uint8_t* zero_a;
    const unsigned char* wq_b;  // launch 1: up bank
    const uint16_t* scale_b;
    const uint8_t* zero_b;
    uint16_t* h;               // launch 1 output [M*topk][N]
    uint16_t* y;               // launch 2 output [M][N]
    int M, topk, E, N, K;      // N, K: rows and columns of one expert matrix
    int ents;                  // staged B columns: M (launch 1, and launch 2 with a row per
                               // token) or M * topk
    int max_rt;                // launch 2: 16-row output tiles whose products a CTA keeps in
                               // shared memory for the routed sums (0 with slot_out)
    int wpt, depth;
    uint32_t* err;
    // launch 2 as an expert GEMV of its own (the kernel's ALONE instantiation):
    // it reads nothing before its grid-dependency wait and flags invalid ids
    // itself; slot s
    // multiplies staged column s / xdiv (1: x a row per slot, topk: a row per
    // token); slot_out: y is bf16 [M*topk][N] per slot, stored as each tile
    // completes (zero rows for an invalid id), instead of the routed sums
    // [M][N]; split (with slot_out): the (row tile, entry) tiles are spread
    // evenly over all CTAs instead of each CTA owning whole row tiles
    int xdiv, slot_out, split;
};

struct MoeHLayout {
    int ring, bfrag, csum, red, bars, ids, ent_e, ent_n, ent_col, ybuf, nent, total;
};
__host__ __device__ inline MoeHLayout moeh_layout(int W, int ents, int kblocks, int depth, int max_rt,
                                                  int bits, int slots, int wpt) {
    MoeHLayout L;
    int off = 0;
    L.ring = off;  // [warp][depth] stages
    off += W * depth * m_stage(bits);
    L.bfrag = off;  // [block][piece][column entity][lane % 4] x 16 bytes
    off += kblocks * 4 * ents * 4 * 16;
    L.csum = off;  // [block][column entity] {1024 sum B, sum x', 2^-sh, 0}
    off += kblocks * ents * 16;
    L.red = off;  // [2][warp][lane] float4 partials of split tiles (none unsplit)
    off += wpt > 1 ? 2 * W * 32 * 16 : 0;
    L.bars = off;  // [tile group][buffer] {full, empty}
    off += W * 2 * 2 * 8;
    L.ids = off;  // routed expert of each slot (-1: invalid)
    off += kMoeHmmaMaxSlots * 4;
    L.ent_e = off;  // expert of each entry
    off += kMoeHmmaMaxSlots * 4;
    L.ent_n = off;  // slots of each entry (launch 2)
    off += kMoeHmmaMaxSlots * 4;
    L.ent_col = off;  // [entry][8] slots (launch 2)
    off += kMoeHmmaMaxSlots * 8 * 4;
    L.ybuf = off;  // launch 2: [row tile][slot][16 rows] fp32 products
    off += max_rt * slots * 16 * 4;
    L.nent = off;
    off += 16;
    L.total = off + 128;
    return L;
}

// cp.async of the 4 bytes at src, of which only the first n (0..4) are read
// (the rest of the destination is zero-filled)
__device__ __forceinline__ void cp_async_4_fill(void* dst, const void* src, int n) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_addr(dst)), "l"(src),
                 "r"(n)
                 : "memory");
}

__device__ __forceinline__ int clamp4(long long v) { return v < 0 ? 0 : (v > 4 ? 4 : static_cast<int>(v)); }

// 3-bit pairs: (a & MASK) | C by one LOP3
template <uint32_t MASK, uint32_t C>
__device__ __forceinline__ uint32_t and_or(uint32_t a) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "n"(MASK), "n"(C));
    return d;
}
template <uint32_t MASK>
__device__ __forceinline__ uint32_t and_or_r(uint32_t a, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "n"(MASK), "r"(c));
    return d;
}
// The 16 fp16 pairs of one INT3 chunk (words w0, w1, w2).  Pair P < 15:
// word P / 5, field f = P % 5, codes 10 (P / 5) + f (low half) and
// 10 (P / 5) + 5 + f (high half), times 1, 8, 64, 1, 8 for f = 0..4; pair 15:
// codes 30 and 31, times 1.  Each value is 1024 + code * factor.
__device__ __forceinline__ void int3_pairs(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t (&p)[16]) {
    constexpr uint32_t E = 0x64006400u;
    const uint32_t w[3] = {w0, w1, w2};
#pragma unroll
    for (int i = 0; i < 3; ++i) {
        const uint32_t t = w[i] >> 9;
        p[5 * i + 0] = and_or<0x00070007u, E>(w[i]);
        p[5 * i + 1] = and_or<0x00380038u, E>(w[i]);
        p[5 * i + 2] = and_or<0x01C001C0u, E>(w[i]);
        p[5 * i + 3] = and_or<0x00070007u, E>(t);
        p[5 * i + 4] = and_or<0x00380038u, E>(t);
    }
    p[15] = and_or_r<0x00040004u>(w2 >> 13, and_or_r<0x00020002u>(w1 >> 14, and_or<0x00010001u, E>(w0 >> 15)));
}
// x' factor of pair P (the inverse of its code factor) and its two codes
__host__ __device__ constexpr int int3_pair_shift(int P) {  // log2 of the code factor
    return P == 15 ? 0 : ((P % 5) == 1 || (P % 5) == 4) ? 3 : (P % 5) == 2 ? 6 : 0;
}
__host__ __device__ constexpr int int3_pair_lo(int P) { return P == 15 ? 30 : 10 * (P / 5) + P % 5; }

// ALONE: launch 2 as an expert GEMV of its own (the xdiv, slot_out and
// split fields apply); the FFN's two launches are instantiated without them
template <int W, int BITS, bool ALONE>
__global__ void __launch_bounds__(32 * W, W == kMWPaired ? 2 : 1) k_moe_hmma(const MoeHK a) {
    constexpr int T = 32 * W;
    constexpr int kPitch = m_pitch(BITS), kStage = m_stage(BITS);
    constexpr int kZero = m_zero(BITS), kScale = m_scale(BITS);
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int S = a.M * a.topk;
    const int kblocks = a.K >> 7;
    const int nsteps = (kblocks + 3) >> 2;
    const int G = kblocks;  // zero points and scales per row (g == 128)
    const int WPT = a.wpt;
    const int NG = W / WPT;
    const int grp = warp / WPT;
    const int part = warp - grp * WPT;
    const int D = a.depth;
    const int ENTS = a.ents;
    const bool p1 = !ALONE && a.phase == 1;
    const bool slot_out = ALONE && a.slot_out;

    const uint32_t raw = smem_addr(smem_raw);
    unsigned char* base = smem_raw + (((raw + 127u) & ~127u) - raw);
    const MoeHLayout L = moeh_layout(W, ENTS, kblocks, D, a.max_rt, BITS, S, WPT);
    unsigned char* ring = base + L.ring + warp * D * kStage;
    uint4* bfrag = reinterpret_cast<uint4*>(base + L.bfrag);
    float4* csum = reinterpret_cast<float4*>(base + L.csum);
    float4* red = reinterpret_cast<float4*>(base + L.red);
    uint64_t* gbar = reinterpret_cast<uint64_t*>(base + L.bars);
    int* s_ids = reinterpret_cast<int*>(base + L.ids);
    int* ent_e = reinterpret_cast<int*>(base + L.ent_e);
    int* ent_n = reinterpret_cast<int*>(base + L.ent_n);
    int* ent_col = reinterpret_cast<int*>(base + L.ent_col);
    int* s_nent = reinterpret_cast<int*>(base + L.nent);
    float* ybuf = reinterpret_cast<float*>(base + L.ybuf);

    if (WPT > 1 && threadIdx.x < NG * 2) {
        mbar_init(gbar + threadIdx.x * 2, (WPT - 1) * 32);
        mbar_init(gbar + threadIdx.x * 2 + 1, 32);
    }
    if (!p1) grid_dependents_launch();

    // Routing (warp 0): slot s = lane.  Entries: launch 1, one per distinct
    // valid expert; launch 2, one per group of up to 8 of an expert's slots;
    // both in order of the expert's first appearance.
    auto route = [&]() {
        if (warp != 0) return;
        const int e = lane < S ? a.ids[lane] : -1;
        const bool valid = lane < S && e >= 0 && e < a.E;
        if ((p1 || ALONE) && lane < S && !valid) raise_device_error(a.err, W4A16_DEVERR_EXPERT_ID);
        // the lanes routed to this lane's expert (an invalid slot matches none)
        const unsigned peers = __match_any_sync(0xffffffffu, valid ? e : -1 - lane);
        const int first = __ffs(peers) - 1;
        const int pos = __popc(peers & ((1u << lane) - 1u));  // earlier slots of the expert
        const int cnt = __popc(peers);
        const bool is_first = valid && first == lane;
        const int nsub = is_first ? (p1 ? 1 : (cnt + 7) >> 3) : 0;
        int incl = nsub;
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        const int ebase = __shfl_sync(0xffffffffu, incl - nsub, valid ? first : 0);
        if (valid) {
            if (p1) {
                if (is_first) ent_e[ebase] = e;
            } else {
                const int en = ebase + (pos >> 3);
                ent_col[en * 8 + (pos & 7)] = lane;
                if ((pos & 7) == 0) {
                    ent_e[en] = e;
                    ent_n[en] = min(8, cnt - pos);
                }
            }
        }
        if (lane < kMoeHmmaMaxSlots) s_ids[lane] = valid ? e : -1;
        if (lane == 31) *s_nent = incl;
    };
    if (ALONE) grid_dependency_wait();  // no input of this launch is known complete
    // launch 2 in the chain routes now; launch 1 and the INT4 expert GEMV
    // route while their first activation loads are in flight (measured on
    // the expert GEMV, 64 experts, top-8: INT4 1-6 % faster at 1..4 tokens,
    // INT3 -- one staging item in flight, not four -- 1-2 % slower)
    const bool early_route = !p1 && (!ALONE || BITS == 3);
    if (early_route) route();
    __syncthreads();  // barriers initialised, routing of launch 2 published

    // Tiles.  Launch 1: the CTA's range of the (entry, 8-row pair) tiles,
    // entry-major.  Launch 2: for each of the CTA's 16-row output tiles, one
    // tile per entry.  A tile is walked as (outer, inner): launch 1 (entry,
    // pair), launch 2 (output tile of the CTA, entry).
    const int tpe = p1 ? (a.N >> 3) : (a.N >> 4);  // pair / row tiles per expert matrix
    int nent = 0, isz = 1, t0 = 0, nt = 0, rt0 = 0, nrt = 0;
    auto set_range = [&](int ne) {
        nent = ne;
        if (p1) {
            const long long tt = static_cast<long long>(ne) * tpe;
            t0 = static_cast<int>(tt * blockIdx.x / gridDim.x);
            nt = static_cast<int>(tt * (blockIdx.x + 1) / gridDim.x) - t0;
            isz = tpe;
        } else if (ALONE && a.split && ne > 0) {
            // an even share of the (row tile, entry) tiles, row-tile-major;
            // t0 counts from the first entry of the CTA's first row tile
            const long long tt = static_cast<long long>(ne) * tpe;
            const long long ta = tt * blockIdx.x / gridDim.x;
            nt = static_cast<int>(tt * (blockIdx.x + 1) / gridDim.x - ta);
            rt0 = static_cast<int>(ta / ne);
            t0 = static_cast<int>(ta - static_cast<long long>(rt0) * ne);
            nrt = nt > 0 ? (t0 + nt - 1) / ne + 1 : 0;
            isz = ne;
        } else {
            rt0 = static_cast<int>(static_cast<long long>(tpe) * blockIdx.x / gridDim.x);
            nrt = static_cast<int>(static_cast<long long>(tpe) * (blockIdx.x + 1) / gridDim.x) - rt0;
            t0 = 0;
            nt = nrt * ne;
            isz = ne > 0 ? ne : 1;
        }
    };
    if (early_route) set_range(*s_nent);

    const size_t row_bytes = BITS == 4 ? static_cast<size_t>(a.K) >> 1 : static_cast<size_t>(a.K) / 128 * 48;
    const int sw_h = lane >> 4, sw_c = ((lane & 15) ^ sw_h) << 4;
    // INT3 copies: lanes 0..23 copy 16-byte chunk col3 of row 2 i + h3
    const int h3 = lane >= 12 ? 1 : 0;
    const int col3 = lane - 12 * h3;
    const int dl0 = sw_h * kHmmaRowPitch + sw_c, dl1 = sw_h * kHmmaRowPitch + (sw_c ^ 32);
    const int dl2 = sw_h * kHmmaRowPitch + (sw_c ^ 64), dl3 = sw_h * kHmmaRowPitch + (sw_c ^ 96);
    auto dst_off = [&](int i) {
        return ((i & 3) == 0 ? dl0 : (i & 3) == 1 ? dl1 : (i & 3) == 2 ? dl2 : dl3) +
               i * 2 * kHmmaRowPitch;
    };
    const int rr = lane & 15;
    const bool zlane = lane < 16;
    const long long zend = static_cast<long long>(a.E) * a.N * G;  // zero-point bytes per bank
    // tile t of the range -> entry and row block, advanced without division
    int my_tiles = 0, my_steps = 0, nu = 0;
    auto set_units = [&]() {
        my_tiles = (nt > grp) ? (nt - grp + NG - 1) / NG : 0;
        my_steps = (nsteps > part) ? (nsteps - part + WPT - 1) / WPT : 0;
        nu = my_tiles * my_steps;
    };
    if (early_route) set_units();
    int i_u = 0, i_slot = 0, i_step = part, i_o = 0, i_i = 0;
    auto start_cursor = [&](int& o, int& in) {
        const int t = t0 + grp;
        o = t / isz;  // once per warp
        in = t - o * isz;
    };
    auto next_tile = [&](int& o, int& in) {
        in += NG;
        while (in >= isz) {
            in -= isz;
            ++o;
        }
    };
    // entry and row tile of the expert matrix of the tile at (o, in)
    auto tile_of = [&](int o, int in, int& en, int& r) {
        if (p1) {
            en = o;
            r = in;
        } else {
            en = in;
            r = rt0 + o;
        }
    };
    // first weight byte of tile rows 0 and 8, and the global row index of
    // rows 0 and 8 (launch 1: gate rows in bank a, the same up rows in bank b)
    auto tile_rows = [&](int o, int in, const unsigned char*& w0, const unsigned char*& w8,
                         long long& z0, long long& z8) {
        int en, r;
        tile_of(o, in, en, r);
        const long long e = ent_e[en];
        if (p1) {
            z0 = e * a.N + 8LL * r;
            z8 = z0;
            w0 = a.wq_a + z0 * static_cast<long long>(row_bytes);
            w8 = a.wq_b + z8 * static_cast<long long>(row_bytes);
        } else {
            z0 = e * a.N + 16LL * r;
            z8 = z0 + 8;
            w0 = a.wq_a + z0 * static_cast<long long>(row_bytes);
            w8 = w0 + 8 * row_bytes;
        }
    };
    // the producer's tile: this lane's first weight byte of tile rows sw_h
    // and 8 + sw_h, and the first group of its zero-point / scale row
    const bool bank_b = p1 && rr >= 8;  // launch 1: tile rows 8..15 are up rows
    const unsigned char* i_w0 = nullptr;
    const unsigned char* i_w8 = nullptr;
    long long i_zg = 0;
    auto producer_tile = [&]() {
        const unsigned char *w0, *w8;
        long long z0, z8;
        tile_rows(i_o, i_i, w0, w8, z0, z8);
        const size_t lane_b = BITS == 4 ? sw_h * row_bytes + (lane & 15) * 16 : h3 * row_bytes + col3 * 16;
        i_w0 = w0 + lane_b;
        i_w8 = w8 + lane_b;
        i_zg = (rr < 8 ? z0 + rr : z8 + (rr - 8)) * G;
    };
    auto issue_next = [&]() {
        if (i_u < nu) {
            const int step = i_step;
            const int nbs = min(4, kblocks - 4 * step);
            unsigned char* stage = ring + i_slot * kStage;
            if constexpr (BITS == 4) {
                if ((lane & 15) < nbs * 4) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const unsigned char* src =
                            (i < 4 ? i_w0 + 2 * i * row_bytes : i_w8 + (2 * i - 8) * row_bytes) + step * 256;
                        cp_async_16(stage + dst_off(i), src);
                    }
                }
            } else {
                if (lane < 24 && col3 < nbs * 3) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const unsigned char* src =
                            (i < 4 ? i_w0 + 2 * i * row_bytes : i_w8 + (2 * i - 8) * row_bytes) + step * 192;
                        cp_async_16(stage + (2 * i + h3) * kPitch + col3 * 16, src);
                    }
                }
            }
            // zero points (lanes 0..15) or scales (16..31) of tile row rr,
            // from the 4-byte words around them
            const long long gi = i_zg + 4LL * step;  // first group of the unit
            if (zlane) {
                const uint8_t* zb = bank_b ? a.zero_b : a.zero_a;
                const long long w4 = gi & ~3LL;
                unsigned char* dz = stage + kZero + rr * 8;
                if (w4 + 8 <= zend) {
                    cp_async_4(dz, zb + w4);
                    cp_async_4(dz + 4, zb + w4 + 4);
                } else {  // the last bytes of the array: read no further
                    const int n0 = clamp4(zend - w4), n1 = clamp4(zend - w4 - 4);
                    cp_async_4_fill(dz, zb + w4, n0);
                    cp_async_4_fill(dz + 4, zb + (n1 > 0 ? w4 + 4 : w4), n1);
                }
            } else {
                const unsigned char* sb =
                    reinterpret_cast<const unsigned char*>(bank_b ? a.scale_b : a.scale_a);
                const long long b = gi * 2, w4 = b & ~3LL, send = zend * 2;
                unsigned char* ds = stage + kScale + rr * 16;
                if (w4 + 12 <= send) {
                    cp_async_4(ds, sb + w4);
                    cp_async_4(ds + 4, sb + w4 + 4);
                    cp_async_4(ds + 8, sb + w4 + 8);
                } else {
#pragma unroll
                    for (int q = 0; q < 3; ++q) {
                        const int n = clamp4(send - w4 - 4 * q);
                        cp_async_4_fill(ds + 4 * q, sb + (n > 0 ? w4 + 4 * q : w4), n);
                    }
                }
            }
            ++i_u;
            if (++i_slot == D) i_slot = 0;
            i_step += WPT;
            if (i_step >= nsteps) {
                i_step = part;
                next_tile(i_o, i_i);
                if (i_u < nu) producer_tile();
            }
        }
        cp_async_commit();
    };
    // launch 2: routing and weights are inputs of the whole chain
    if (early_route) {
        if (nu > 0) {
            start_cursor(i_o, i_i);
            producer_tile();
        }
        for (int k = 0; k < D; ++k) issue_next();
    }
    grid_dependency_wait();
    if (p1) grid_dependents_launch();

    // launch 1 (and the INT4 expert GEMV) routes while its first activation
    // loads are in flight, then requests its first units
    auto start_launch1 = [&]() {
        if (early_route) return;
        route();
        __syncthreads();
        set_range(*s_nent);
        set_units();
        if (nu > 0) {
            start_cursor(i_o, i_i);
            producer_tile();
        }
        for (int k = 0; k < D; ++k) issue_next();
    };
    if constexpr (BITS == 4) {
        // B columns: the K range of every column entity (token or slot), in
        // fragment order, each 128-k block scaled by a power of two.  One
        // item is two 8-k pieces (16 k) of one column, pieces l and l + 8 of
        // a 128-k block; the 8 items of a block are 8 consecutive lanes (they
        // share the block's maximum and sums by shuffles).  Four items per thread are in flight, each slot
        // refilled four items ahead as soon as it is converted.
        const int tid = threadIdx.x;
        const int ipc = kblocks * 8;    // items per column
        const int cols = ENTS;          // staged B columns: tokens or slots
        const int nflat = cols * ipc;
        const int items = (nflat + T - 1) / T;
        auto load_item = [&](int it, uint4 (&v)[2]) {
            const int f = it * T + tid;
            v[0] = v[1] = make_uint4(0u, 0u, 0u, 0u);
            if (it < items && f < nflat) {
                const int m = f / ipc, r = f - m * ipc;
                // pieces l and l + 8 of block r / 8 (l = r % 8)
                const uint4* src = reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(m) * a.K) +
                                   (r >> 3) * 16 + (r & 7);
                v[0] = __ldg(src);
                v[1] = __ldg(src + 8);
            }
        };
        uint4 v[4][2];
#pragma unroll
        for (int b = 0; b < 4; ++b) load_item(b, v[b]);
        start_launch1();
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
                    const int m = f / ipc, r = f - m * ipc;
                    const int blk = r >> 3, l = r & 7;  // pieces 16 blk + l and 16 blk + l + 8
                    bfrag[((blk * 4 + (l >> 2)) * cols + m) * 4 + (l & 3)] = o2[0];
                    bfrag[((blk * 4 + (l >> 2) + 2) * cols + m) * 4 + (l & 3)] = o2[1];
                    if (l == 0) csum[blk * cols + m] = make_float4(1024.f * c1, c2, exp2i(-sh), 0.f);
                }
            }
        }
    } else {
        // B columns for INT3 units: one item is 32 k (a chunk) of one column
        // entity; the 4 chunks of a 128-k block are 4 consecutive lanes.
        // An item's 16 B registers are the pairs of its chunk (int3_pairs
        // order), x scaled by the block's power of two and divided by the
        // pair's code factor.
        const int tid = threadIdx.x;
        const int cpc = kblocks * 4;    // chunks per column
        const int cols = ENTS;          // staged B columns: tokens or slots
        const int nflat = cols * cpc;
        const int items = (nflat + T - 1) / T;
        auto load_item = [&](int it, uint4 (&v)[4]) {
            const int f = it * T + tid;
#pragma unroll
            for (int b = 0; b < 4; ++b) v[b] = make_uint4(0u, 0u, 0u, 0u);
            if (it < items && f < nflat) {
                const int m = f / cpc, r = f - m * cpc;
                const uint4* src = reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(m) * a.K + r * 32);
#pragma unroll
                for (int b = 0; b < 4; ++b) v[b] = __ldg(src + b);
            }
        };
        uint4 v[4], vn[4];
        load_item(0, v);
        start_launch1();
        for (int it = 0; it < items; ++it) {  // the same count for the whole CTA
            load_item(it + 1, vn);
            const int f = it * T + tid;
            const uint32_t wv[16] = {v[0].x, v[0].y, v[0].z, v[0].w, v[1].x, v[1].y, v[1].z, v[1].w,
                                     v[2].x, v[2].y, v[2].z, v[2].w, v[3].x, v[3].y, v[3].z, v[3].w};
            uint32_t mx2 = 0u;
#pragma unroll
            for (int e = 0; e < 16; ++e) mx2 = __vmaxu2(mx2, wv[e] & 0x7FFF7FFFu);
            uint32_t mx = max(mx2 & 0xFFFFu, mx2 >> 16);
            mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const int sh = block_shift(mx);
            float fa, fb;
            pow2_pair(sh, fa, fb);
            auto xs = [&](int i) {  // x of code i of the chunk, times 2^sh / fb
                const uint32_t w = wv[i >> 1];
                return __uint_as_float((i & 1) ? (w & 0xFFFF0000u) : (w << 16)) * fa;
            };
            uint32_t breg[16];
            float c1 = 0.f, c2 = 0.f;
#pragma unroll
            for (int P = 0; P < 16; ++P) {
                const int lo = int3_pair_lo(P), hi = P == 15 ? 31 : lo + 5;
                const float fac = fb * (1.f / static_cast<float>(1 << int3_pair_shift(P)));
                const __half2 h2 = __floats2half2_rn(xs(lo) * fac, xs(hi) * fac);
                breg[P] = *reinterpret_cast<const uint32_t*>(&h2);
                const float2 bf = __half22float2(h2);
                const float ps = bf.x + bf.y;
                c1 += ps;
                c2 = fmaf(static_cast<float>(1 << int3_pair_shift(P)), ps, c2);
            }
            c1 += __shfl_xor_sync(0xffffffffu, c1, 1);
            c2 += __shfl_xor_sync(0xffffffffu, c2, 1);
            c1 += __shfl_xor_sync(0xffffffffu, c1, 2);
            c2 += __shfl_xor_sync(0xffffffffu, c2, 2);
            if (f < nflat) {
                const int m = f / cpc, r = f - m * cpc;
                const int blk = r >> 2, ch = r & 3;
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    bfrag[((blk * 4 + u) * cols + m) * 4 + ch] =
                        make_uint4(breg[4 * u], breg[4 * u + 1], breg[4 * u + 2], breg[4 * u + 3]);
                if (ch == 0) csum[blk * cols + m] = make_float4(1024.f * c1, c2, exp2i(-sh), 0.f);
            }
#pragma unroll
            for (int b = 0; b < 4; ++b) v[b] = vn[b];
        }
    }
    __syncthreads();

    const int g = lane >> 2, c = lane & 3;
    const int CS = ENTS;  // B column stride of the staged fragments
    const int lrow = (lane & 7) + (((lane >> 3) & 1) << 3);
    const int lch = lane >> 4;
    const int sw_s = lane & 7;
    const uint32_t ring_addr = smem_addr(ring) + static_cast<uint32_t>(lrow * kHmmaRowPitch);
    const uint32_t lve = (lch ^ (sw_s & 1)) << 4;
    const uint32_t lv0 = lve + ((0 ^ (sw_s & 2)) << 4) + ((0 ^ (sw_s & 4)) << 4);
    const uint32_t lv1 = lve + ((2 ^ (sw_s & 2)) << 4) + ((0 ^ (sw_s & 4)) << 4);
    const uint32_t lv2 = lve + ((0 ^ (sw_s & 2)) << 4) + ((4 ^ (sw_s & 4)) << 4);
    const uint32_t lv3 = lve + ((2 ^ (sw_s & 2)) << 4) + ((4 ^ (sw_s & 4)) << 4);

    float4 tacc = make_float4(0.f, 0.f, 0.f, 0.f);
    bool timed_out = false;
    int c_slot = 0, c_step = part, ti = 0, c_o = 0, c_i = 0, c_ent = 0, c_r = 0;
    if (nu > 0) {
        start_cursor(c_o, c_i);
        tile_of(c_o, c_i, c_ent, c_r);
    }
    // per tile: B column entity of lane g, C column entities 2c, 2c + 1
    // (launch 2: staged columns; scol0, scol1 the slots of C columns 2c, 2c + 1)
    int col_g = 0, col0 = 0, col1 = 0, scol0 = 0, scol1 = 0;
    bool use0 = false, use1 = false, two = false;
    int subz_a = 0, subz_b = 0, subs_a = 0, subs_b = 0;
    auto set_tile = [&]() {
        if (p1) {
            col_g = g < a.M ? g : 0;
            use0 = 2 * c < a.M;
            use1 = 2 * c + 1 < a.M;
            col0 = use0 ? 2 * c : 0;
            col1 = use1 ? 2 * c + 1 : 0;
            two = a.M > 1;
        } else {
            const int n = ent_n[c_ent];
            const int* cl = ent_col + c_ent * 8;
            col_g = cl[g < n ? g : 0];
            use0 = 2 * c < n;
            use1 = 2 * c + 1 < n;
            scol0 = cl[use0 ? 2 * c : 0];
            scol1 = cl[use1 ? 2 * c + 1 : 0];
            col0 = scol0;
            col1 = scol1;
            if (ALONE && a.xdiv != 1) {  // staged columns are tokens
                col_g /= a.xdiv;
                col0 /= a.xdiv;
                col1 /= a.xdiv;
            }
            two = n > 1;
        }
        const unsigned char *w0, *w8;
        long long z0, z8;
        tile_rows(c_o, c_i, w0, w8, z0, z8);
        subz_a = static_cast<int>(((z0 + g) * G) & 3);
        subz_b = static_cast<int>(((z8 + g) * G) & 3);
        subs_a = static_cast<int>(((z0 + g) * G * 2) & 3);
        subs_b = static_cast<int>(((z8 + g) * G * 2) & 3);
    };
    if (nu > 0) set_tile();
#pragma unroll 1
    for (int k = 0; k < nu; ++k) {
        cp_async_wait_pending(D - 1);
        __syncwarp();
        const int slot = c_slot;
        const int lstep = c_step;
        if (++c_slot == D) c_slot = 0;
        const int nbs = min(4, kblocks - 4 * lstep);
        const uint32_t wst = ring_addr + static_cast<uint32_t>(slot * kStage);
        const unsigned char* sz = ring + slot * kStage;
        const uint2 zwa = *reinterpret_cast<const uint2*>(sz + kZero + g * 8);
        const uint2 zwb = *reinterpret_cast<const uint2*>(sz + kZero + (g + 8) * 8);
        const uint4 swa = *reinterpret_cast<const uint4*>(sz + kScale + g * 16);
        const uint4 swb = *reinterpret_cast<const uint4*>(sz + kScale + (g + 8) * 16);
        const uint32_t za = __funnelshift_r(zwa.x, zwa.y, 8 * subz_a);
        const uint32_t zb = __funnelshift_r(zwb.x, zwb.y, 8 * subz_b);
        const uint32_t sa01 = __funnelshift_r(swa.x, swa.y, 8 * subs_a);
        const uint32_t sa23 = __funnelshift_r(swa.y, swa.z, 8 * subs_a);
        const uint32_t sb01 = __funnelshift_r(swb.x, swb.y, 8 * subs_b);
        const uint32_t sb23 = __funnelshift_r(swb.y, swb.z, 8 * subs_b);
        const uint4* bqu = bfrag + static_cast<size_t>(4 * lstep) * 4 * CS * 4 + col_g * 4 + c;
        const float4* csu = csum + static_cast<size_t>(4 * lstep) * CS;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int bb = 0; bb < 4; ++bb) {
            if (bb >= nbs) break;  // the same for the whole warp
            uint4 bq[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) bq[j] = bqu[(bb * 4 + j) * CS * 4];
            float d0[4], d1[4];
            if constexpr (BITS == 4) {
                const uint32_t hb = wst + static_cast<uint32_t>((bb >> 1) * 128);
                uint32_t q0[4], q1[4];
                ldmatrix_x4(q0, hb + ((bb & 1) ? lv2 : lv0));
                ldmatrix_x4(q1, hb + ((bb & 1) ? lv3 : lv1));
                const uint32_t wa[4] = {q0[0], q0[2], q1[0], q1[2]};
                const uint32_t wb[4] = {q0[1], q0[3], q1[1], q1[3]};
                {
                    const uint32_t ta = wa[0] >> 8, tb = wb[0] >> 8;
                    mma_f16_16816_zero(d0, f16_codes_lo(wa[0]), f16_codes_lo(wb[0]), f16_codes_hi(wa[0]),
                                       f16_codes_hi(wb[0]), bq[0].x, bq[0].y);
                    mma_f16_16816_zero(d1, f16_codes_lo(ta), f16_codes_lo(tb), f16_codes_hi(ta),
                                       f16_codes_hi(tb), bq[0].z, bq[0].w);
                }
#pragma unroll
                for (int j = 1; j < 4; ++j) {
                    const uint32_t ta = wa[j] >> 8, tb = wb[j] >> 8;
                    mma_f16_16816(d0, f16_codes_lo(wa[j]), f16_codes_lo(wb[j]), f16_codes_hi(wa[j]),
                                  f16_codes_hi(wb[j]), bq[j].x, bq[j].y);
                    mma_f16_16816(d1, f16_codes_lo(ta), f16_codes_lo(tb), f16_codes_hi(ta),
                                  f16_codes_hi(tb), bq[j].z, bq[j].w);
                }
            } else {
                // chunk c of block bb of rows g and g + 8: three words each
                const uint32_t* ra = reinterpret_cast<const uint32_t*>(sz + g * kPitch + bb * 48 + c * 12);
                const uint32_t* rb = ra + 2 * kPitch;  // 8 rows on
                uint32_t pa[16], pb[16];
                int3_pairs(ra[0], ra[1], ra[2], pa);
                int3_pairs(rb[0], rb[1], rb[2], pb);
                // MMA m: pairs 2m (k slots 2c, 2c + 1) and 2m + 1 (2c + 8, 2c + 9)
                mma_f16_16816_zero(d0, pa[0], pb[0], pa[1], pb[1], bq[0].x, bq[0].y);
                mma_f16_16816_zero(d1, pa[2], pb[2], pa[3], pb[3], bq[0].z, bq[0].w);
#pragma unroll
                for (int j = 1; j < 4; ++j) {
                    mma_f16_16816(d0, pa[4 * j], pb[4 * j], pa[4 * j + 1], pb[4 * j + 1], bq[j].x, bq[j].y);
                    mma_f16_16816(d1, pa[4 * j + 2], pb[4 * j + 2], pa[4 * j + 3], pb[4 * j + 3], bq[j].z,
                                  bq[j].w);
                }
            }
            const float zfa = zero_point_f32(za, bb), zfb = zero_point_f32(zb, bb);
            const uint32_t pa = bb < 2 ? sa01 : sa23, pb = bb < 2 ? sb01 : sb23;
            const float sfa = __uint_as_float((bb & 1) ? (pa & 0xFFFF0000u) : (pa << 16));
            const float sfb = __uint_as_float((bb & 1) ? (pb & 0xFFFF0000u) : (pb << 16));
            const float4 cs0 = csu[bb * CS + col0];
            acc[0] = fmaf(sfa * cs0.z, (d0[0] + d1[0]) - fmaf(zfa, cs0.y, cs0.x), acc[0]);
            acc[2] = fmaf(sfb * cs0.z, (d0[2] + d1[2]) - fmaf(zfb, cs0.y, cs0.x), acc[2]);
            if (two) {
                const float4 cs1 = csu[bb * CS + col1];
                acc[1] = fmaf(sfa * cs1.z, (d0[1] + d1[1]) - fmaf(zfa, cs1.y, cs1.x), acc[1]);
                acc[3] = fmaf(sfb * cs1.z, (d0[3] + d1[3]) - fmaf(zfb, cs1.y, cs1.x), acc[3]);
            }
        }
        __syncwarp();
        issue_next();
        tacc.x += acc[0];
        tacc.y += acc[1];
        tacc.z += acc[2];
        tacc.w += acc[3];
        c_step += WPT;
        if (c_step < nsteps) continue;
        c_step = part;
        // the tile is complete: partials to part 0, which stores
        if (WPT > 1) {
            if (part != 0) {
                timed_out |= !hand_partial<W>(red, gbar, grp, WPT, part, ti, lane, tacc);
            } else {
                const int b = ti & 1;
                const float4* rb = red + (b * W + grp * WPT) * 32;
                uint64_t* full = gbar + (grp * 2 + b) * 2;
                timed_out |= !mbar_wait_bounded(full, (ti >> 1) & 1);
                for (int q = 1; q < WPT; ++q) {
                    const float4 pv = rb[q * 32 + lane];
                    tacc.x += pv.x;
                    tacc.y += pv.y;
                    tacc.z += pv.z;
                    tacc.w += pv.w;
                }
                mbar_arrive(full + 1);
            }
        }
        if (part == 0) {
            const int e = ent_e[c_ent];
            if (p1) {
                // rows g, g + 8: gate and up row 8 r + g of expert e
                const size_t hr = static_cast<size_t>(c_r) * 8 + g;
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int t = 2 * c + q;
                    if (t >= a.M) continue;
                    const uint16_t hv = swiglu_of_sums(q ? tacc.y : tacc.x, q ? tacc.w : tacc.z);
                    for (int j = 0; j < a.topk; ++j)
                        if (s_ids[t * a.topk + j] == e)
                            a.h[static_cast<size_t>(t * a.topk + j) * a.N + hr] = hv;
                }
            } else if (slot_out) {
                // the entry's slots of output tile c_r, straight to y
                uint16_t* yr = a.y + static_cast<size_t>(c_r) * 16 + g;
                if (use0) {
                    yr[static_cast<size_t>(scol0) * a.N] = f32_to_bf16_rn(tacc.x);
                    yr[static_cast<size_t>(scol0) * a.N + 8] = f32_to_bf16_rn(tacc.z);
                }
                if (use1) {
                    yr[static_cast<size_t>(scol1) * a.N] = f32_to_bf16_rn(tacc.y);
                    yr[static_cast<size_t>(scol1) * a.N + 8] = f32_to_bf16_rn(tacc.w);
                }
            } else {
                // the entry's slot columns of output tile c_r, to shared memory
                float* yb = ybuf + static_cast<size_t>(c_r - rt0) * S * 16;
                if (use0) {
                    yb[scol0 * 16 + g] = tacc.x;
                    yb[scol0 * 16 + g + 8] = tacc.z;
                }
                if (use1) {
                    yb[scol1 * 16 + g] = tacc.y;
                    yb[scol1 * 16 + g + 8] = tacc.w;
                }
            }
        }
        tacc = make_float4(0.f, 0.f, 0.f, 0.f);
        ++ti;
        if (k + 1 < nu) {
            next_tile(c_o, c_i);
            tile_of(c_o, c_i, c_ent, c_r);
            set_tile();
        }
    }
    if (WPT > 1 && my_steps == 0)
        for (; ti < my_tiles; ++ti)
            timed_out |= !hand_partial<W>(red, gbar, grp, WPT, part, ti, lane,
                                          make_float4(0.f, 0.f, 0.f, 0.f));
    cp_async_wait_pending(0);
    if (timed_out && lane == 0) raise_device_error(a.err, W4A16_DEVERR_TIMEOUT);
    if (slot_out) {
        // the valid slots were stored as their tiles completed; the rows of
        // an invalid slot are zero (a row tile shared by two CTAs gets its
        // zeros twice)
        for (int idx = threadIdx.x; idx < nrt * S * 16; idx += T) {
            const int rl = idx / (S * 16);
            const int rem = idx - rl * S * 16;
            const int sl = rem >> 4, row = rem & 15;
            if (s_ids[sl] < 0) a.y[static_cast<size_t>(sl) * a.N + (rt0 + rl) * 16 + row] = 0;
        }
    } else if (!p1) {
        // routed sums of the CTA's output tiles: every slot's product is in
        // shared memory; slots in order, invalid ids skipped
        __syncthreads();
        for (int idx = threadIdx.x; idx < nrt * a.M * 16; idx += T) {
            const int rl = idx / (a.M * 16);
            const int rem = idx - rl * a.M * 16;
            const int t = rem >> 4, row = rem & 15;
            const float* yb = ybuf + static_cast<size_t>(rl) * S * 16;
            float v = 0.f;
            for (int j = 0; j < a.topk; ++j) {
                const int sl = t * a.topk + j;
                if (s_ids[sl] >= 0) v += a.route_w[sl] * yb[sl * 16 + row];
            }
            a.y[static_cast<size_t>(t) * a.N + (rt0 + rl) * 16 + row] = f32_to_bf16_rn(v);
        }
    }
}

struct MoeHPlan {
    int warps, ctas, wpt, depth, smem, max_rt, split;
};
// Warps per CTA: 16 (two per SMSP for the units' latency), or 8 where a
// 16-warp CTA's rings and staged activations do not fit in shared memory.
// Measured, MoE chain of 64 experts (2304 x 1024), top-8, 16- against 8-warp
// down launches: 35.9 / 43.0 us against 38.5 / 43.5 at M = 3 / 4 (INT3:
// 37.6 / 39.5 against 38.8 / 42.6); the down-shaped expert GEMV at M = 3:
// 13.0 against 14.4 us.  (With an earlier, slower unit the 8-warp CTAs had
// been ahead beyond 16 slots.)
// CTAs, warps per tile and ring depth for one launch, at most one CTA per SM
// (two fit where shared memory allows, for the next launch's).  Launch 1:
// tiles_max (entry, pair) tiles, the split of K steps over warps that
// minimises the busiest warp's units.  Launch 2: row_tiles output tiles over
// the CTAs, tiles_max entries at most; `slots` products per row tile kept
// in shared memory for the routed sums, or none with slot_out -- whose
// (row tile, entry) tiles are spread over all CTAs when there are fewer row
// tiles than SMs.
MoeHPlan plan_moe_hmma_w(const DeviceInfo& dev, int phase, int ents, int slots, int kblocks,
                         long long tiles_max, int row_tiles, int bits, int slot_out, int warps) {
    MoeHPlan p{};
    p.warps = warps;
    const int nsteps = (kblocks + 3) / 4;
    int ybuf_rt = 0;
    if (phase == 1) {
        if (tiles_max < 1) return p;
        p.ctas = static_cast<int>(tiles_max < dev.sms ? tiles_max : dev.sms);
        const long long max_tiles = (tiles_max + p.ctas - 1) / p.ctas;
        long long best = -1;
        for (int wpt = 1; wpt <= p.warps; wpt *= 2) {
            const int ng = p.warps / wpt;
            const long long u = ((max_tiles + ng - 1) / ng) * ((nsteps + wpt - 1) / wpt);
            const long long cost = 8 * u + ((max_tiles + ng - 1) / ng) * (wpt - 1);
            if (best < 0 || cost < best) {
                best = cost;
                p.wpt = wpt;
            }
        }
        p.max_rt = 0;
    } else {
        if (row_tiles < 1 || tiles_max < 1) return p;
        // tiles_max: at most this many entries.  Each entry's K steps go to
        // one warp, or to a power of two of warps while the CTA's tiles
        // leave warps idle (one token: 8 entries on 16 warps, two each)
        long long tiles;
        p.split = slot_out && row_tiles < dev.sms ? 1 : 0;
        if (p.split) {
            const long long tt = static_cast<long long>(row_tiles) * tiles_max;
            p.ctas = static_cast<int>(tt < dev.sms ? tt : dev.sms);
            tiles = (tt + p.ctas - 1) / p.ctas;
            p.max_rt = 0;
        } else {
            p.ctas = row_tiles < dev.sms ? row_tiles : dev.sms;
            p.max_rt = (row_tiles + p.ctas - 1) / p.ctas;
            tiles = static_cast<long long>(p.max_rt) * tiles_max;
        }
        // (spread tiles take at most two warps each: with four, the INT3
        // expert GEMV of one token, 64 experts of 1024 x 2304, measured 3 %
        // slower; INT4 the same either way)
        const int wpt_cap = p.split ? 2 : nsteps;
        p.wpt = 1;
        while (p.wpt * 2 <= nsteps && p.wpt * 2 <= wpt_cap && tiles * p.wpt * 2 <= p.warps) p.wpt *= 2;
        if (slot_out) p.max_rt = 0;  // nothing kept in shared memory
        ybuf_rt = p.max_rt;
    }
    const int half = dev.smem_per_sm / 2 - 1024;
    const int budget = p.warps == kMWPaired &&
                               moeh_layout(p.warps, ents, kblocks, 2, ybuf_rt, bits, slots, p.wpt).total <=
                                   half
                           ? half
                           : dev.max_smem_optin;
    // launch 1 keeps two stages per warp: deeper rings queue more weight
    // copies ahead of its activation loads (measured, 64 experts, top-8: the
    // chain at 2 tokens 22.49 -> 22.00 us, INT3 at 4 tokens 39.40 -> 39.00)
    const int max_depth = phase == 1 ? 2 : kMMaxDepth;
    p.depth = 2;
    while (p.depth < max_depth &&
           moeh_layout(p.warps, ents, kblocks, p.depth + 1, ybuf_rt, bits, slots, p.wpt).total <= budget)
        ++p.depth;
    p.smem = moeh_layout(p.warps, ents, kblocks, p.depth, ybuf_rt, bits, slots, p.wpt).total;
    if (p.smem > dev.max_smem_optin) p.ctas = 0;
    return p;
}
// 16-warp CTAs, or 8-warp CTAs where those do not fit
MoeHPlan plan_moe_hmma(const DeviceInfo& dev, int phase, int ents, int slots, int kblocks,
                       long long tiles_max, int row_tiles, int bits, int slot_out) {
    const MoeHPlan p =
        plan_moe_hmma_w(dev, phase, ents, slots, kblocks, tiles_max, row_tiles, bits, slot_out, kMWWide);
    if (p.ctas > 0) return p;
    return plan_moe_hmma_w(dev, phase, ents, slots, kblocks, tiles_max, row_tiles, bits, slot_out,
                           kMWPaired);
}

}  // namespace

bool moe_hmma_supports(int M, int topk, int64_t H, int64_t F, int64_t g) {
    return g == 128 && M >= 1 && M <= 8 && topk >= 1 && M * topk <= kMoeHmmaMaxSlots &&
           H % 128 == 0 && F % 128 == 0 && H >= 128 && F >= 128;
}

// Entries of launch 2 (groups of up to 8 slots of one expert): at most one
// per slot, and at most one per expert plus one per 8 slots.
static long long moe_entries_bound(int S, int E) {
    const long long b = static_cast<long long>(E) + S / 8;
    return b < S ? b : S;
}

bool moe_hmma_fits(const DeviceInfo& dev, int M, int topk, int E, int64_t H, int64_t F, int bits) {
    const int S = M * topk;
    const long long d = E < S ? E : S;
    return plan_moe_hmma(dev, 1, M, 0, static_cast<int>(H / 128), d * (F / 8), 0, bits, 0).ctas > 0 &&
           plan_moe_hmma(dev, 2, S, S, static_cast<int>(F / 128), moe_entries_bound(S, E),
                         static_cast<int>(H / 16), bits, 0).ctas > 0;
}

namespace {
// one launch of k_moe_hmma with plan p (BITS 3 or 4; 8- or 16-warp CTAs;
// ALONE: an expert GEMV of its own)
template <bool ALONE>
cudaError_t launch_moe_hmma_one(const MoeHK& k, const MoeHPlan& p, int bits, cudaStream_t s) {
    const bool wide = p.warps == kMWWide, b3 = bits == 3;
    const void* kern = b3 ? (wide ? reinterpret_cast<const void*>(k_moe_hmma<kMWWide, 3, ALONE>)
                                  : reinterpret_cast<const void*>(k_moe_hmma<kMWPaired, 3, ALONE>))
                          : (wide ? reinterpret_cast<const void*>(k_moe_hmma<kMWWide, 4, ALONE>)
                                  : reinterpret_cast<const void*>(k_moe_hmma<kMWPaired, 4, ALONE>));
    cudaError_t e = ensure_dynamic_smem(kern, p.smem);
    if (e != cudaSuccess) return e;
    // the two launches ask for different shared memory: with the largest
    // carve-out for both, a launch-2 CTA can be resident beside a
    // launch-1 CTA (an SM whose carve-out must change waits to drain)
    static bool carveout_set[4] = {false, false, false, false};
    const int ck = (b3 ? 2 : 0) + (wide ? 1 : 0);
    if (!carveout_set[ck]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        carveout_set[ck] = true;
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(p.ctas);
    cfg.blockDim = dim3(32 * p.warps);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return b3 ? (wide ? cudaLaunchKernelEx(&cfg, k_moe_hmma<kMWWide, 3, ALONE>, k)
                      : cudaLaunchKernelEx(&cfg, k_moe_hmma<kMWPaired, 3, ALONE>, k))
              : (wide ? cudaLaunchKernelEx(&cfg, k_moe_hmma<kMWWide, 4, ALONE>, k)
                      : cudaLaunchKernelEx(&cfg, k_moe_hmma<kMWPaired, 4, ALONE>, k));
}
}  // namespace

cudaError_t launch_moe_hmma(const MoeHmmaArgs& a, const DeviceInfo& dev, cudaStream_t s) {
    const int S = a.M * a.topk;
    for (int phase = 1; phase <= 2; ++phase) {
        MoeHK k{};
        k.phase = phase;
        k.ids = a.ids;
        k.route_w = a.route_w;
        k.M = a.M;
        k.topk = a.topk;
        k.E = a.E;
        k.err = a.err;
        k.h = a.h;
        k.y = a.y;
        k.xdiv = 1;
        long long tiles_max = 0;
        int row_tiles = 0;
        if (phase == 1) {
            k.x = a.x;
            k.wq_a = reinterpret_cast<const unsigned char*>(a.gate_wq);
            k.scale_a = a.gate_scale;
            k.zero_a = a.gate_zero;
            k.wq_b = reinterpret_cast<const unsigned char*>(a.up_wq);
            k.scale_b = a.up_scale;
            k.zero_b = a.up_zero;
            k.N = static_cast<int>(a.F);
            k.K = static_cast<int>(a.H);
            k.ents = a.M;
            tiles_max = static_cast<long long>(a.E < S ? a.E : S) * (a.F / 8);
        } else {
            k.x = a.h;
            k.wq_a = reinterpret_cast<const unsigned char*>(a.down_wq);
            k.scale_a = a.down_scale;
            k.zero_a = a.down_zero;
            k.N = static_cast<int>(a.H);
            k.K = static_cast<int>(a.F);
            k.ents = S;
            row_tiles = static_cast<int>(a.H / 16);
            tiles_max = moe_entries_bound(S, a.E);
        }
        const MoeHPlan p =
            plan_moe_hmma(dev, phase, k.ents, S, k.K / 128, tiles_max, row_tiles, a.bits, 0);
        if (p.ctas < 1) return cudaErrorInvalidConfiguration;
        k.max_rt = p.max_rt;
        k.wpt = p.wpt;
        k.depth = p.depth;
        const cudaError_t e = launch_moe_hmma_one<false>(k, p, a.bits, s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

bool moe_hmma_gemv_supports(int M, int topk, int64_t N, int64_t K, int64_t g) {
    return g == 128 && M >= 1 && topk >= 1 && M * topk <= kMoeHmmaMaxSlots && N >= 16 &&
           N % 16 == 0 && K >= 128 && K % 128 == 0 && N <= (int64_t(1) << 24) && K <= 65536;
}

// staged activation columns: one per slot, or one per token when the slots
// of a token share its row
static int moe_gemv_cols(int M, int topk, int x_per_slot) { return x_per_slot ? M * topk : M; }

bool moe_hmma_gemv_fits(const DeviceInfo& dev, int M, int topk, int E, int64_t N, int64_t K, int bits,
                        int x_per_slot, int routed) {
    const int S = M * topk;
    return plan_moe_hmma(dev, 2, moe_gemv_cols(M, topk, x_per_slot), S, static_cast<int>(K / 128),
                         moe_entries_bound(S, E), static_cast<int>(N / 16), bits, routed ? 0 : 1)
               .ctas > 0;
}

cudaError_t launch_moe_hmma_gemv(const MoeHmmaGemvArgs& a, const DeviceInfo& dev, cudaStream_t s) {
    const int S = a.M * a.topk;
    MoeHK k{};
    k.phase = 2;
    k.x = a.x;
    k.xdiv = a.x_per_slot ? 1 : a.topk;
    k.slot_out = a.route_w ? 0 : 1;
    k.ids = a.ids;
    k.route_w = a.route_w;
    k.wq_a = reinterpret_cast<const unsigned char*>(a.wq);
    k.scale_a = a.scale;
    k.zero_a = a.zero;
    k.y = a.y;
    k.M = a.M;
    k.topk = a.topk;
    k.E = a.E;
    k.N = static_cast<int>(a.N);
    k.K = static_cast<int>(a.K);
    k.ents = moe_gemv_cols(a.M, a.topk, a.x_per_slot);
    k.err = a.err;
    const MoeHPlan p = plan_moe_hmma(dev, 2, k.ents, S, k.K / 128, moe_entries_bound(S, a.E),
                                     static_cast<int>(a.N / 16), a.bits, k.slot_out);
    if (p.ctas < 1) return cudaErrorInvalidConfiguration;
    k.max_rt = p.max_rt;
    k.split = p.split;
    k.wpt = p.wpt;
    k.depth = p.depth;
    return launch_moe_hmma_one<true>(k, p, a.bits, s);
}

}  // namespace w4a16
