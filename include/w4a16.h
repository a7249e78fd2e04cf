/*
 * w4a16.h -- C ABI of the GB300 (sm_103a) W4A16 INT4-weight GEMV library.
 *
 * The operation is the decode-time product described in the local-kimi
 * README (RightNow-AI/local-kimi), technical-detail section: a matrix of
 * group-quantised 4-bit weights times a handful (M <= 16) of 16-bit
 * activation rows, done as a true matrix-vector product -- the reduction
 * axis K contiguous in memory, one accumulator row per output, and no
 * per-call partial buffers (same section).  The grouped-expert variant of the
 * same section is w4a16_moe_gemv.
 *
 * Data layout (all row-major, all device memory unless stated otherwise):
 *   x      bf16   [M][K]        activations (IEEE bfloat16 bit patterns)
 *   wq     uint32 [N][K/8]      packed codes: code(n,k) = (wq[n][k/8] >> 4*(k%8)) & 15,
 *                               i.e. eight codes per word, lowest nibble = lowest k
 *   scale  bf16   [N][K/g]      one scale per (row, group of g consecutive k)
 *   zero   uint8  [N][K/g]      one integer zero point per (row, group)
 *   W[n][k] = (code(n,k) - zero[n][k/g]) * scale[n][k/g]
 *   y      [M][N]  bf16 or fp32: y[m][n] = sum_k x[m][k] * W[n][k]
 *
 * Conventions shared by every call:
 *   - bf16 values are passed as uint16_t bit patterns.
 *   - Every pointer is a device pointer owned by the caller; the library never
 *     allocates device memory.  A `stream` is a cudaStream_t passed as void*
 *     (NULL = the legacy default stream).  Calls are asynchronous: they
 *     enqueue kernels on `stream` and return without synchronising.
 *   - Arguments are validated before anything is launched.  An invalid call
 *     returns a status other than W4A16_OK and leaves every output untouched.
 *     Nothing is thrown across this interface.  W4A16_ERR_CUDA means a launch
 *     was refused by the CUDA runtime; faults of kernels already enqueued
 *     surface, as usual in CUDA, at the caller's next synchronisation.
 *   - Data-dependent problems that only the GPU can see (an expert id out of
 *     range, a staging wait that timed out) never trap: the kernel skips the
 *     affected work, writes zeros there, and sets a bit in a per-device error
 *     word that w4a16_device_error reads.
 *   - All tensor pointers must be 16-byte aligned (W4A16_ERR_ALIGN otherwise).
 *   - Shape limits: 1 <= M <= 16; K % 32 == 0; g % 32 == 0; K % g == 0;
 *     N >= 1; K <= 65536; N*K/8 < 2^31 words per matrix.
 */
#ifndef W4A16_H
#define W4A16_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Symbol visibility: the library is built with hidden visibility and exports
 * exactly the functions declared here. */
#if defined(__GNUC__)
#define W4A16_API __attribute__((visibility("default")))
#else
#define W4A16_API
#endif

typedef enum w4a16_status {
    W4A16_OK = 0,
    W4A16_ERR_NULL = 1,        /* a required pointer is NULL */
    W4A16_ERR_SHAPE = 2,       /* a size is out of range or inconsistent */
    W4A16_ERR_ALIGN = 3,       /* a pointer is not 16-byte aligned */
    W4A16_ERR_UNSUPPORTED = 4, /* valid request outside what is implemented (e.g. M > 16) */
    W4A16_ERR_WORKSPACE = 5,   /* workspace missing or smaller than *_workspace_bytes */
    W4A16_ERR_CUDA = 6         /* the CUDA runtime refused a launch or query */
} w4a16_status;

typedef enum w4a16_out_dtype {
    W4A16_OUT_BF16 = 0, /* outputs rounded to bf16, nearest-even */
    W4A16_OUT_F32 = 1   /* outputs stored as fp32 (e.g. vocabulary logits) */
} w4a16_out_dtype;

/* Flags of w4a16_gemv_ex. */
#define W4A16_FLAG_WEIGHTS_STATIC 0x1u /* wq, scale and zero are not written by work
                                          still running on the stream (see w4a16_gemv_ex) */
#define W4A16_FLAG_SWIGLU_OUTPUT 0x2u  /* rows are gate/up pairs of 8-row blocks; y is
                                          bf16(silu(gate) * up) (see w4a16_gemv_ex) */
#define W4A16_FLAG_NO_CLUSTER 0x4u     /* keep the K split inside a CTA: no thread-block
                                          cluster launch (see w4a16_gemv_ex) */

/* Bits of the per-device error word (see w4a16_device_error). */
#define W4A16_DEVERR_EXPERT_ID 0x1u /* an expert id was outside [0, E) */
#define W4A16_DEVERR_TIMEOUT 0x2u   /* a bounded wait for staged data expired */
#define W4A16_DEVERR_RANGE 0x4u     /* an activation outside the CUDA-core kernel's
                                       input range: |x| >= 2^43 or not finite
                                       (see w4a16_gemv) */

/* Version of this interface; bumped on any incompatible change. */
W4A16_API int w4a16_abi_version(void);

/* Static, NUL-terminated description of a status code. */
W4A16_API const char* w4a16_status_string(w4a16_status status);

/*
 * int4_pack -- pack 4-bit codes into the wq layout above.
 *   codes  uint8 [N][K], each 0..15 (only the low nibble is used)
 *   wq     uint32 [N][K/8] output
 * Requires K % 8 == 0.  Bit-exact integer work.
 * (Packing order: the problem statement accompanying the README's
 *  technical-detail section -- eight codes per word, low nibble first along K.)
 */
W4A16_API w4a16_status int4_pack(const uint8_t* codes, uint32_t* wq, int64_t N, int64_t K, void* stream);

/*
 * int4_dequant -- expand packed weights to W[n][k] = (code - zero) * scale,
 * the group-quantised weights of the W4A16 kernels (README technical-detail
 * section; the problem statement accompanying it writes the product as
 * x . dequant(Wq, scale, zero) with one scale and zero point per g
 * consecutive k of a row).
 *   w  [N][K] output, bf16 (the exact value rounded to nearest-even) or fp32
 *      (exact: |code - zero| <= 15 times an 8-bit significand fits in 24 bits).
 * Requires K % 32 == 0, g % 32 == 0, K % g == 0.
 */
W4A16_API w4a16_status int4_dequant(const uint32_t* wq, const uint16_t* scale, const uint8_t* zero,
                          void* w, w4a16_out_dtype out_dtype, int64_t N, int64_t K, int64_t g,
                          void* stream);

/*
 * ~3-bit expert weights.  The README's hardware-requirements paragraph says
 * that fitting a 24 GB card needs the expert weights near three bits and
 * gives no format; this library's INT3 format (exactly three bits per code):
 *   codes 0..7, W[n][k] = (code - zero[n][k/g]) * scale[n][k/g] with the bf16
 *   scale and uint8 zero point of the INT4 path;
 *   a row of K codes (K % 128 == 0) is 3K/32 uint32 words; the 32 codes
 *   k = 32j .. 32j + 31 of a row (a chunk) are words 3j, 3j + 1, 3j + 2;
 *   code i < 30 of a chunk is the 3-bit field (lowest bit first) of word
 *   3j + i/10 at bit 16 * ((i % 10) / 5) + 3 * (i % 5): five codes in bits
 *   0..14 of each 16-bit half;
 *   bit b (b = 0, 1, 2) of code 30 is bit 15, and of code 31 bit 31, of word
 *   3j + b.
 * Uniform codes make uniform words: the 96 bits of a chunk hold its 32 codes.
 */

/*
 * int3_pack -- pack 3-bit codes into the INT3 layout above.
 *   codes  uint8 [N][K], each 0..7 (only the low three bits are used)
 *   wq3    uint32 [N][3K/32] output
 * Requires K % 128 == 0.  Bit-exact integer work.
 */
W4A16_API w4a16_status int3_pack(const uint8_t* codes, uint32_t* wq3, int64_t N, int64_t K, void* stream);

/*
 * int3_dequant -- expand INT3 weights to W[n][k] = (code - zero) * scale,
 * as int4_dequant does for INT4 (bf16: the exact value rounded to
 * nearest-even; fp32: exact).
 * Requires K % 128 == 0, g % 32 == 0, K % g == 0.
 */
W4A16_API w4a16_status int3_dequant(const uint32_t* wq3, const uint16_t* scale, const uint8_t* zero,
                                    void* w, w4a16_out_dtype out_dtype, int64_t N, int64_t K, int64_t g,
                                    void* stream);

/*
 * w4a16_gemv_workspace_bytes -- device workspace w4a16_gemv needs for this
 * shape.  The dense GEMV needs none (0): split-K partials are combined
 * on chip through thread-block-cluster shared memory.  Kept so callers can
 * size a workspace generically.
 */
W4A16_API size_t w4a16_gemv_workspace_bytes(int M, int64_t N, int64_t K, int64_t g);

/*
 * w4a16_gemv -- y[M][N] = x[M][K] . W^T with W dequantised on the fly
 * (README technical-detail section: the GEMV rewrite of the dense W4A16
 * kernel).  Products are formed exactly and accumulated in fp32; y is stored
 * as bf16 (round to nearest-even) or fp32 per out_dtype.
 *   workspace/workspace_bytes: may be NULL/0 (none is needed; see above).
 * Kernel choice (fixed by M, N, K, g; see w4a16_gemv_plan):
 *   - g == 128, K % 512 == 0 and either M <= 2, or M <= 4 with
 *     N * K >= 2^24, or M <= 16 with
 *     N * K >= 2^25 where it has a launch plan (9..16 tokens take K slices of
 *     at most 2048 k): the fp16 warp-MMA kernel (id 4), which takes any
 *     finite bf16 x (each 128-k block of x is scaled by a power of two into
 *     fp16, exactly where the block's values lie within 2^24 of its
 *     largest);
 *   - otherwise, g % 128 == 0: the bf16 warp-MMA kernel (id 2), any M;
 *   - otherwise (groups finer than 128 k), M <= 2: the CUDA-core kernel
 *     (id 1); M > 2 is W4A16_ERR_UNSUPPORTED.
 * Input range of the CUDA-core kernel (a precondition the call checks): it
 * needs |x| < 2^43 -- a larger or non-finite activation sets
 * W4A16_DEVERR_RANGE in the device error word (w4a16_device_error), and the
 * outputs are then not to be used (an activation at a k that is a multiple
 * of 8 overflows to infinity).  It forms products |code * x| >= 2^-62 exactly;
 * smaller ones round to fp32's subnormal grid, so activations below about
 * 2^-60 carry an absolute output error of up to (K + K/32) * 2^-86 *
 * max|scale| * max|code - zero|.  The two warp-MMA kernels have neither
 * limit beyond fp32's own range.
 * The kernel is launched with programmatic dependent launch: it may begin
 * while the previous kernel on `stream` drains, but reads and writes no
 * global memory until that kernel has completed, so stream order is kept.
 * Pointers are device-accessible addresses.  With M == 1, x and y may be
 * page-locked host memory mapped into the device's address space (every
 * kernel reads x and writes y with plain loads and stores): the kernel then
 * reads and writes them in place, with no copies around the call.
 */
W4A16_API w4a16_status w4a16_gemv(const uint16_t* x, const uint32_t* wq, const uint16_t* scale,
                        const uint8_t* zero, void* y, w4a16_out_dtype out_dtype, int M,
                        int64_t N, int64_t K, int64_t g, void* workspace, size_t workspace_bytes,
                        void* stream);

/*
 * w4a16_gemv_ex -- w4a16_gemv with flags.
 *   W4A16_FLAG_WEIGHTS_STATIC lets the kernel start loading wq/scale/zero
 *   before the previous kernel on `stream` has completed (x is still read,
 *   and y written, only after it completes).  Set it only when no kernel that
 *   may still be running on the stream writes those three buffers -- the
 *   case of resident model weights in a decode loop.  It is a permission:
 *   what it buys depends on the launch (measured on GB300, back-to-back
 *   4096 x 4096 GEMVs: 4.21 us per call with it, 4.39 us without).
 *   W4A16_FLAG_SWIGLU_OUTPUT fuses the SwiGLU of a decode MLP into the
 *   gate/up projection (README technical-detail section: the kernel
 *   registry's SwiGLU op; the expert FFN does the same inside
 *   w4a16_moe_ffn).  The N rows of wq/scale/zero hold the gate and up
 *   matrices (N/2 rows each) interleaved in blocks of 8: rows 16t..16t+7
 *   are gate rows 8t..8t+7 and rows 16t+8..16t+15 are up rows 8t..8t+7.
 *   y is then bf16 [M][N/2], y[m][i] = bf16(silu(gate) * up) with gate and
 *   up the bf16-rounded products of row i of each matrix, computed in fp32
 *   exactly as w4a16_swiglu computes it -- so the result equals that of the
 *   plain GEMV followed by w4a16_swiglu, bit for bit, in one launch.
 *   Requires N % 16 == 0, out_dtype W4A16_OUT_BF16 and a shape the fp16 or
 *   bf16 warp-MMA kernel serves (w4a16_gemv_plan kernel id 4 or 2: g a
 *   multiple of 128); otherwise W4A16_ERR_UNSUPPORTED.
 *   W4A16_FLAG_NO_CLUSTER plans the launch without a thread-block cluster
 *   (the K split stays among the warps of a CTA) where the shape allows one;
 *   otherwise the call plans as without the flag.  w4a16_gemv_plan reports
 *   the plan without flags.  Which plan is faster depends on the kernel
 *   before it: a cluster split wins in a run of identical launches, but
 *   after the 16-warp launch of a gate/up GEMV with the SwiGLU epilogue the
 *   down GEMV of a decode MLP starts sooner without one -- measured on
 *   GB300, that two-launch MLP takes 24.5 us per token with the flag on the
 *   down GEMV and 29.5 us without, although alone the down GEMV is 11 %
 *   slower with it (and after the small w4a16_swiglu kernel it is slower
 *   too).
 * Otherwise identical to w4a16_gemv (workspace is not needed).
 */
W4A16_API w4a16_status w4a16_gemv_ex(const uint16_t* x, const uint32_t* wq, const uint16_t* scale,
                                     const uint8_t* zero, void* y, w4a16_out_dtype out_dtype,
                                     int M, int64_t N, int64_t K, int64_t g, unsigned flags,
                                     void* stream);

/*
 * w4a16_gemv_plan -- describe the launch w4a16_gemv would make for a shape,
 * without launching: kernel id (1 = CUDA-core kernel, 2 = bf16 warp-MMA
 * kernel, 4 = fp16 warp-MMA kernel), CTAs, threads per CTA, K-split factor
 * (how many warps share one row tile, counting the CTAs of a thread-block
 * cluster) and dynamic shared memory bytes.  Any output pointer may be NULL.  Needs the current device's
 * properties (W4A16_ERR_CUDA without a device).
 */
W4A16_API w4a16_status w4a16_gemv_plan(int M, int64_t N, int64_t K, int64_t g, int* kernel_id, int* ctas,
                             int* threads, int* k_split, int* smem_bytes);

/*
 * w4a16_gemv_variant -- w4a16_gemv with the kernel forced (for measurement):
 * kernel_id 1 (CUDA-core, M <= 2), 2 (bf16 warp-MMA, any M, g % 128 == 0),
 * 3 (tensor-core tcgen05, any M, g % 128 == 0) or 4 (fp16 warp-MMA,
 * M <= 16, g == 128, K % 512 == 0); k_split 0 = automatic, else the K-split
 * factor, a power of two: for kernels 1 and 2, 1..32 (warps of a CTA first,
 * then up to 8 CTAs of a cluster); for kernels 3 and 4, 1..8 CTAs of a
 * cluster (kernel 4 then chooses its warps per tile itself).  A split the shape cannot use (a CTA's activation slice too large
 * for shared memory, or a CTA left without K range) is
 * W4A16_ERR_UNSUPPORTED.  Same contract as w4a16_gemv.
 */
W4A16_API w4a16_status w4a16_gemv_variant(const uint16_t* x, const uint32_t* wq, const uint16_t* scale,
                                const uint8_t* zero, void* y, w4a16_out_dtype out_dtype, int M,
                                int64_t N, int64_t K, int64_t g, int kernel_id, int k_split,
                                void* stream);

/*
 * w4a16_moe_workspace_bytes -- workspace w4a16_moe_gemv needs: fp32 partials
 * [M][topk][N] when route weights are given (route != 0), else 0.
 */
W4A16_API size_t w4a16_moe_workspace_bytes(int M, int topk, int64_t N, int route);

/*
 * w4a16_moe_gemv -- expert-indexed W4A16 GEMV (README technical-detail
 * section, the grouped expert kernel).  For token t and routed slot j with
 * e = expert_ids[t][j]:
 *     d[t][j][n] = sum_k xin[k] * W_e[n][k],
 *     xin = x[t] (x_per_slot == 0, x is [M][K]) or x[t][j] (x is [M][topk][K]).
 * Experts are stacked: wq [E][N][K/8], scale and zero [E][N][K/g].
 * Each distinct expert's weights are streamed once per call however many
 * slots select it.
 *   route_w == NULL: y is bf16 [M][topk][N], y[t][j] = d[t][j].
 *   route_w != NULL: fp32 [M][topk]; y is bf16 [M][N],
 *                    y[t][n] = sum_j route_w[t][j] * d[t][j][n] (fp32, j ascending);
 *                    needs a workspace of w4a16_moe_workspace_bytes(M, topk, N, 1).
 * Kernel: the fp16 warp-MMA expert kernel (w4a16_moe_gemv_variant's
 * kernel 4) where it applies -- M*topk <= 32, g == 128, K % 128 == 0,
 * N % 16 == 0, the staged activations in shared memory -- else the bf16
 * warp-MMA expert kernel (kernel 2).  Measured on one GB300, 64 experts,
 * top-8, M = 1 / 2 / 4: experts [1024, 2304] per slot 7.6 / 9.5 / 13.3 us
 * against 9.8 / 12.9 / 20.3 for kernel 2; experts [2304, 1024] routed 6.5 /
 * 9.0 / 17.4 against 9.8 / 13.4 / 21.3.
 * Limits: M*topk <= 256, E >= 1.  Expert ids outside [0, E) are skipped
 * (their contribution is zero) and flagged with W4A16_DEVERR_EXPERT_ID.
 */
W4A16_API w4a16_status w4a16_moe_gemv(const uint16_t* x, int x_per_slot, const int32_t* expert_ids,
                            const float* route_w, const uint32_t* wq, const uint16_t* scale,
                            const uint8_t* zero, uint16_t* y, int M, int topk, int E, int64_t N,
                            int64_t K, int64_t g, void* workspace, size_t workspace_bytes,
                            void* stream);

/*
 * w4a16_moe_gemv_variant -- w4a16_moe_gemv with the kernel named:
 *   0  the library's choice (what w4a16_moe_gemv runs);
 *   2  the bf16 warp-MMA expert kernel with TMA rings (any shape within
 *      w4a16_moe_gemv's limits);
 *   4  the fp16 warp-MMA expert kernel of w3a16_moe_gemv over INT4 codes
 *      (the down launch of w4a16_moe_ffn's fp16 path on its own), with its
 *      limits: M * topk <= 32, g == 128, K a multiple of 128, N a multiple
 *      of 16, the staged activations in shared memory; routed sums are
 *      formed in shared memory, so the workspace is not used.
 * Other ids, or a shape outside the named kernel's limits, give
 * W4A16_ERR_UNSUPPORTED.  Arguments and results are those of w4a16_moe_gemv.
 */
W4A16_API w4a16_status w4a16_moe_gemv_variant(const uint16_t* x, int x_per_slot,
                                              const int32_t* expert_ids, const float* route_w,
                                              const uint32_t* wq, const uint16_t* scale,
                                              const uint8_t* zero, uint16_t* y, int M, int topk,
                                              int E, int64_t N, int64_t K, int64_t g,
                                              int kernel_id, void* workspace,
                                              size_t workspace_bytes, void* stream);

/* Size of the library's fixed scratch buffer (per device), in bytes. */
#define W4A16_FIXED_SCRATCH_BYTES (1u << 20)

/*
 * w4a16_moe_gemv_fixed_scratch -- w4a16_moe_gemv for callers that cannot
 * allocate device memory or lend a workspace: engines whose device memory is
 * split into fixed pools, plug-ins whose host runtime owns the allocator.
 * (The README has no counterpart; this is an integration convenience of
 * this library.)  Same arguments, kernels and results as w4a16_moe_gemv,
 * minus the workspace: where the routed sum needs fp32 partials (the bf16
 * expert kernel; the fp16 one keeps them in shared memory) they go to a
 * buffer of W4A16_FIXED_SCRATCH_BYTES compiled into the library, one per
 * device, held until the process exits.  Nothing is allocated by the call.
 *   - Only calls with route_w use the buffer; calls without it need none.
 *   - Requests needing more than W4A16_FIXED_SCRATCH_BYTES
 *     (M * topk * N * 4 bytes with route_w) return W4A16_ERR_WORKSPACE,
 *     whichever kernel would run.
 *   - The first routed call on a device looks the buffer up
 *     (cudaGetSymbolAddress) and caches its address for the life of the
 *     process: do not use the call after cudaDeviceReset.
 *   - All calls on a device share the buffer: calls whose kernels can overlap
 *     on the GPU race on it; calls ordered on one stream are safe.  Nothing
 *     left in it by an earlier call is read.
 */
W4A16_API w4a16_status w4a16_moe_gemv_fixed_scratch(const uint16_t* x, int x_per_slot,
                                                    const int32_t* expert_ids, const float* route_w,
                                                    const uint32_t* wq, const uint16_t* scale,
                                                    const uint8_t* zero, uint16_t* y, int M,
                                                    int topk, int E, int64_t N, int64_t K,
                                                    int64_t g, void* stream);

/*
 * w4a16_moe_ffn_workspace_bytes -- workspace w4a16_moe_ffn needs: bf16 gate
 * and up outputs [M][topk][F], fp32 partials [M][topk][H] and one 32-bit
 * counter per 64 rows of H, each part rounded up to 256 bytes.  Its contents
 * need no initialisation.
 */
W4A16_API size_t w4a16_moe_ffn_workspace_bytes(int M, int topk, int64_t H, int64_t F);

/*
 * w4a16_moe_ffn -- the routed SwiGLU expert FFN of M tokens (README
 * technical-detail section: the grouped expert kernel; its kernel registry
 * names the SwiGLU op), in two launches:
 *   1. gate and up products of every routed slot, both banks in one launch:
 *        G[t][j] = bf16(W^gate_e x[t]),  U[t][j] = bf16(W^up_e x[t]),
 *      and h[t][j] = bf16(silu(G[t][j]) * U[t][j]) (in fp32 exactly as
 *      w4a16_swiglu computes it);
 *   2. down products and the routed sums
 *        y[t] = bf16(sum_j route_w[t][j] * (W^down_e h[t][j])) (fp32, j ascending).
 * With 1..8 tokens, M*topk <= 32 and g == 128 (H, F multiples of 128) this is
 * the fp16 warp-MMA path: launch 1 forms h in its epilogue, launch 2 owns
 * 16-row output tiles and forms their routed sums in shared memory.
 * Otherwise the bf16 warp-MMA expert kernel: h is formed while launch 2
 * stages its activations, and the last CTA to finish each row chunk forms
 * its routed sums.  Each distinct expert's three matrices are streamed once
 * per call.
 *   x: bf16 [M][H]; expert_ids: int32 [M][topk]; route_w: fp32 [M][topk];
 *   gate, up: wq [E][F][H/8], scale and zero [E][F][H/g];
 *   down: wq [E][H][F/8], scale and zero [E][H][F/g]; y: bf16 [M][H];
 *   workspace: >= w4a16_moe_ffn_workspace_bytes(M, topk, H, F) bytes,
 *   caller-owned, 16-byte aligned (W4A16_ERR_WORKSPACE if smaller).
 * Limits: M*topk <= 256, g % 128 == 0, H and F multiples of g.  Expert ids
 * outside [0, E) are skipped and flagged with W4A16_DEVERR_EXPERT_ID.
 */
W4A16_API w4a16_status w4a16_moe_ffn(const uint16_t* x, const int32_t* expert_ids,
                                     const float* route_w, const uint32_t* gate_wq,
                                     const uint16_t* gate_scale, const uint8_t* gate_zero,
                                     const uint32_t* up_wq, const uint16_t* up_scale,
                                     const uint8_t* up_zero, const uint32_t* down_wq,
                                     const uint16_t* down_scale, const uint8_t* down_zero,
                                     uint16_t* y, int M, int topk, int E, int64_t H, int64_t F,
                                     int64_t g, void* workspace, size_t workspace_bytes,
                                     void* stream);

/*
 * w3a16_moe_ffn_workspace_bytes -- workspace w3a16_moe_ffn needs: the bf16
 * intermediate h [M][topk][F], rounded up to 256 bytes.  Its contents need
 * no initialisation.
 */
W4A16_API size_t w3a16_moe_ffn_workspace_bytes(int M, int topk, int64_t H, int64_t F);

/*
 * w3a16_moe_ffn -- the routed SwiGLU expert FFN of w4a16_moe_ffn over INT3
 * expert banks (the ~3-bit expert weights above):
 *   y[t] = bf16(sum_j route_w[t][j] * (W^down_e h[t][j])),
 *   h[t][j] = bf16(silu(bf16(W^gate_e x[t])) * bf16(W^up_e x[t])), e = ids[t][j],
 * in two launches on the fp16 warp-MMA path (gate/up with the SwiGLU in the
 * epilogue, then the down products and routed sums).
 *   x: bf16 [M][H]; expert_ids: int32 [M][topk]; route_w: fp32 [M][topk];
 *   gate, up: wq3 [E][F][3H/32], scale and zero [E][F][H/g];
 *   down: wq3 [E][H][3F/32], scale and zero [E][H][F/g]; y: bf16 [M][H];
 *   workspace: >= w3a16_moe_ffn_workspace_bytes(M, topk, H, F) bytes,
 *   caller-owned, 16-byte aligned (W4A16_ERR_WORKSPACE if smaller).
 * Limits: 1 <= M <= 8, M * topk <= 32, g == 128, H and F multiples of 128
 * (W4A16_ERR_UNSUPPORTED otherwise).  Expert ids outside [0, E) are skipped
 * and flagged with W4A16_DEVERR_EXPERT_ID.
 */
W4A16_API w4a16_status w3a16_moe_ffn(const uint16_t* x, const int32_t* expert_ids,
                                     const float* route_w, const uint32_t* gate_wq3,
                                     const uint16_t* gate_scale, const uint8_t* gate_zero,
                                     const uint32_t* up_wq3, const uint16_t* up_scale,
                                     const uint8_t* up_zero, const uint32_t* down_wq3,
                                     const uint16_t* down_scale, const uint8_t* down_zero,
                                     uint16_t* y, int M, int topk, int E, int64_t H, int64_t F,
                                     int64_t g, void* workspace, size_t workspace_bytes,
                                     void* stream);

/*
 * w3a16_moe_gemv -- the expert-indexed GEMV of w4a16_moe_gemv over an INT3
 * expert bank (the ~3-bit expert weights above).  For token t and routed
 * slot j with e = expert_ids[t][j]:
 *     d[t][j][n] = sum_k xin[k] * W_e[n][k],
 *     xin = x[t] (x_per_slot == 0, x is [M][K]) or x[t][j] (x is [M][topk][K]).
 *   wq3 [E][N][3K/32], scale and zero [E][N][K/g].
 *   route_w == NULL: y is bf16 [M][topk][N], y[t][j] = bf16(d[t][j]), zero
 *                    rows for an invalid id;
 *   route_w != NULL: fp32 [M][topk]; y is bf16 [M][N],
 *                    y[t][n] = bf16(sum_j route_w[t][j] * d[t][j][n]) (fp32,
 *                    j ascending, invalid ids skipped).
 * One launch of the fp16 warp-MMA expert kernel (the down launch of
 * w3a16_moe_ffn on its own).  A tile is 16 output rows of one routed expert
 * against all of that expert's slots (up to 8 per tile), so each distinct
 * expert's rows are streamed once whatever the number of slots that select
 * it.  With route weights a CTA owns whole 16-row output tiles and forms
 * their routed sums in shared memory; per-slot outputs are stored as each
 * tile completes, the tiles spread over all CTAs when N / 16 is below the
 * SM count.  No workspace.
 * Limits: M * topk <= 32, g == 128, K a multiple of 128 (<= 65536), N a
 * multiple of 16 (W4A16_ERR_UNSUPPORTED otherwise, or if the staged
 * activations do not fit in shared memory: 2 * K bytes per token row, or
 * per slot with x_per_slot, next to the weight rings).
 * Expert ids outside [0, E) are skipped and flagged with
 * W4A16_DEVERR_EXPERT_ID.
 */
W4A16_API w4a16_status w3a16_moe_gemv(const uint16_t* x, int x_per_slot,
                                      const int32_t* expert_ids, const float* route_w,
                                      const uint32_t* wq3, const uint16_t* scale,
                                      const uint8_t* zero, uint16_t* y, int M, int topk, int E,
                                      int64_t N, int64_t K, int64_t g, void* stream);

/*
 * w4a16_swiglu -- h[r][n] = bf16(silu(gate[r][n]) * up[r][n]), computed in
 * fp32, silu(v) = v / (1 + e^-v).  The activation between the gate/up and
 * down expert products (the README's kernel registry names a SwiGLU op).
 *   gate, up: bf16 rows with leading dimension ld_in (elements); h: bf16 rows
 *   with leading dimension ld_out.  Lets gate/up be the two halves of one
 *   stacked [rows][2N] output (up = gate + N, ld_in = 2N).
 * Requires ld_in >= N, ld_out >= N; pointers 4-byte aligned; N even.
 */
W4A16_API w4a16_status w4a16_swiglu(const uint16_t* gate, const uint16_t* up, int64_t ld_in, uint16_t* h,
                          int64_t ld_out, int64_t rows, int64_t N, void* stream);

/*
 * w4a16_host_memory_mapped -- 1 if `p` is page-locked host memory that
 * kernels on the current device address at the same pointer (so it may be
 * passed as x or y of a one-token w4a16_gemv), else 0.  Host-side query, no
 * stream work.
 */
W4A16_API int w4a16_host_memory_mapped(const void* p);

/*
 * w4a16_wait_selftest -- one warp waits on a shared-memory mbarrier with the
 * bounded wait every kernel of this library uses (tries of up to 100 us
 * each, at most max_iters, 1..8192).  With arrive != 0 one arrival completes
 * the phase and the wait returns at once; with arrive == 0 nothing arrives,
 * the wait gives up after max_iters tries and W4A16_DEVERR_TIMEOUT is set in
 * the device error word -- the path an expired wait in a GEMV or expert
 * kernel takes (the kernel returns, the context stays usable).  For tests of
 * that failure path; asynchronous on `stream`.
 */
W4A16_API w4a16_status w4a16_wait_selftest(unsigned max_iters, int arrive, void* stream);

/*
 * w4a16_device_error -- synchronise `stream`, then copy the current device's
 * error word (W4A16_DEVERR_* bits set by kernels since the last clear) to
 * *bits_out (host pointer); reset it to 0 if clear != 0.
 */
W4A16_API w4a16_status w4a16_device_error(uint32_t* bits_out, int clear, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* W4A16_H */
