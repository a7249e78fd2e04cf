/*
 * Reference oracle for the W4A16 INT4-weight GEMV -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * may load this file's library.  The product path (the CUDA library and its
 * Python binding) never calls it and shares no code, header or table with it.
 *
 * What it computes is the plain definition of the method, in fp64, with no
 * blocking, fusion or reordering:
 *
 *   code(n,k)  = (Wq[n][k/8] >> 4*(k mod 8)) & 0xF        eight 4-bit codes per
 *                                                          32-bit word, lowest
 *                                                          nibble = lowest k
 *   W[n][k]    = (code(n,k) - zero[n][k/g]) * scale[n][k/g]
 *   y[m][n]    = sum_k x[m][k] * W[n][k]                   (fp64, natural k order)
 *
 * This is the decode-time W4A16 product of the local-kimi README
 * (RightNow-AI/local-kimi), technical-detail section: a group-quantised INT4
 * weight matrix times a few 16-bit activation rows, done as a true
 * matrix-vector product with the reduction axis K contiguous.  The packing
 * order, group size, (q - zero) * scale dequantisation and bf16 types are the
 * problem statement that accompanies that page; the README itself is silent on
 * them.
 *
 * The mixture-of-experts chain (grouped expert kernel of the same section):
 * per token t and routed slot j with expert e = ids[t][j],
 *   gate = bf16(gemv(x_t, Wg[e])),  up = bf16(gemv(x_t, Wu[e])),
 *   h    = bf16(silu(gate) * up),   d  = gemv(h, Wd[e])       (fp64)
 *   out[t] = sum_j r[t][j] * d                                  (fp64)
 * The rounding points to bf16 mirror the storage types a GPU chain uses
 * between its kernels.
 *
 * bf16 values cross this interface as their 16-bit IEEE patterns (uint16_t).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- bf16 <-> double ---------------------------------------------------- */

/* Exact widening: a bf16 pattern is the top half of an IEEE binary32. */
double oracle_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round an fp64 value to bf16 (8 significant bits, 8-bit exponent) with a
 * single round-to-nearest-even step taken directly from the double, so there
 * is no double rounding through binary32.  Subnormals (quantum 2^-133) and
 * overflow to infinity follow IEEE 754. */
uint16_t oracle_bf16_round(double v)
{
    if (isnan(v)) return (uint16_t)0x7FC0;
    uint16_t sign = signbit(v) ? (uint16_t)0x8000 : (uint16_t)0;
    double a = fabs(v);
    if (a == 0.0) return sign;
    if (isinf(a)) return (uint16_t)(sign | 0x7F80);
    int e;
    (void)frexp(a, &e);            /* a = m * 2^e with m in [0.5, 1) */
    int qexp = e - 8;              /* weight of the last kept bit */
    if (qexp < -133) qexp = -133;  /* subnormal range: fixed quantum */
    double r = nearbyint(ldexp(a, -qexp));  /* default mode: ties to even */
    double rv = ldexp(r, qexp);
    if (rv >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80);
    float f = (float)rv;           /* exact: rv has <= 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | (uint16_t)(u >> 16));
}

void oracle_bf16_round_array(const double* v, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_round(v[i]);
}

/* ---- packing ------------------------------------------------------------ */

/* codes[N][K] (each 0..15) -> wq[N][K/8], code k of a row in bits 4*(k%8). */
void oracle_pack(const uint8_t* codes, uint32_t* wq, int64_t N, int64_t K)
{
    for (int64_t n = 0; n < N; ++n)
        for (int64_t j = 0; j < K / 8; ++j) {
            uint32_t word = 0;
            for (int i = 0; i < 8; ++i)
                word |= (uint32_t)(codes[n * K + 8 * j + i] & 0xF) << (4 * i);
            wq[n * (K / 8) + j] = word;
        }
}

static inline int oracle_code(const uint32_t* wq, int64_t K, int64_t n, int64_t k)
{
    uint32_t word = wq[n * (K / 8) + k / 8];
    return (int)((word >> (4 * (k % 8))) & 0xFu);
}

void oracle_unpack(const uint32_t* wq, uint8_t* codes, int64_t N, int64_t K)
{
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            codes[n * K + k] = (uint8_t)oracle_code(wq, K, n, k);
}

/* ---- dequantisation ----------------------------------------------------- */

static inline double oracle_weight(const uint32_t* wq, const uint16_t* scale,
                                   const uint8_t* zero, int64_t K, int64_t g,
                                   int64_t n, int64_t k)
{
    int64_t G = K / g;
    double s = oracle_bf16_to_double(scale[n * G + k / g]);
    double z = (double)zero[n * G + k / g];
    return ((double)oracle_code(wq, K, n, k) - z) * s;
}

/* w[N][K] = (code - zero) * scale, exact in fp64. */
void oracle_dequant(const uint32_t* wq, const uint16_t* scale, const uint8_t* zero,
                    double* w, int64_t N, int64_t K, int64_t g)
{
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            w[n * K + k] = oracle_weight(wq, scale, zero, K, g, n, k);
}

/* ---- GEMV --------------------------------------------------------------- */

/* y[M][n_rows]: for each listed output row n = rows[i],
 * y[m][i] = sum_k x[m][k] * W[n][k] in fp64, k ascending. */
void oracle_gemv_rows(const uint16_t* x, const uint32_t* wq, const uint16_t* scale,
                      const uint8_t* zero, const int64_t* rows, int64_t n_rows,
                      double* y, int64_t M, int64_t K, int64_t g)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t i = 0; i < n_rows; ++i) {
            int64_t n = rows[i];
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += oracle_bf16_to_double(x[m * K + k]) *
                       oracle_weight(wq, scale, zero, K, g, n, k);
            y[m * n_rows + i] = acc;
        }
}

/* y[M][N] over every output row. */
void oracle_gemv(const uint16_t* x, const uint32_t* wq, const uint16_t* scale,
                 const uint8_t* zero, double* y, int64_t M, int64_t N, int64_t K,
                 int64_t g)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += oracle_bf16_to_double(x[m * K + k]) *
                       oracle_weight(wq, scale, zero, K, g, n, k);
            y[m * N + n] = acc;
        }
}

/* The same y[M][N] with the output rows shared among `threads` host threads
 * (OpenMP when the library is built with it, else one thread).  Every
 * element is the loop of oracle_gemv -- one fp64 sum in ascending k -- so the
 * values are identical to it; only the rows' order of evaluation differs. */
void oracle_gemv_parallel(const uint16_t* x, const uint32_t* wq, const uint16_t* scale,
                          const uint8_t* zero, double* y, int64_t M, int64_t N, int64_t K,
                          int64_t g, int64_t threads)
{
    (void)threads;
#ifdef _OPENMP
#pragma omp parallel for num_threads((int)threads) schedule(static)
#endif
    for (int64_t n = 0; n < N; ++n)
        for (int64_t m = 0; m < M; ++m) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += oracle_bf16_to_double(x[m * K + k]) *
                       oracle_weight(wq, scale, zero, K, g, n, k);
            y[m * N + n] = acc;
        }
}

/* Host threads oracle_gemv_parallel can use (1 without OpenMP). */
int64_t oracle_max_threads(void)
{
#ifdef _OPENMP
    return (int64_t)omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---- SwiGLU ------------------------------------------------------------- */

/* h = bf16(silu(gate) * up), silu(v) = v / (1 + exp(-v)), all in fp64. */
void oracle_swiglu(const uint16_t* gate, const uint16_t* up, uint16_t* h, int64_t count)
{
    for (int64_t i = 0; i < count; ++i) {
        double a = oracle_bf16_to_double(gate[i]);
        double b = oracle_bf16_to_double(up[i]);
        double silu = a / (1.0 + exp(-a));
        h[i] = oracle_bf16_round(silu * b);
    }
}

/* ---- expert-indexed GEMV ------------------------------------------------ */

/* For token t (0..M-1) and routed slot j (0..topk-1), with e = ids[t][j]:
 *   d[t][j][n] = sum_k xin[k] * W_e[n][k]
 * where xin is x[t] (x_per_slot == 0, x is [M][K]) or x[t][j]
 * (x_per_slot != 0, x is [M][topk][K]).  Expert e's matrices start at
 * wq + e*N*K/8, scale + e*N*(K/g), zero + e*N*(K/g).
 * If route_w is NULL, d is written to y[M][topk][N]; otherwise
 *   y[t][n] = sum_j route_w[t][j] * d[t][j][n]   (fp64, j ascending).
 * Returns -1 (and writes nothing for that slot) if an id is out of [0, E). */
int oracle_moe_gemv(const uint16_t* x, int x_per_slot, const int32_t* ids,
                    const float* route_w, const uint32_t* wq, const uint16_t* scale,
                    const uint8_t* zero, double* y, int64_t M, int64_t topk, int64_t E,
                    int64_t N, int64_t K, int64_t g)
{
    int bad = 0;
    int64_t G = K / g;
    if (route_w)
        for (int64_t i = 0; i < M * N; ++i) y[i] = 0.0;
    for (int64_t t = 0; t < M; ++t)
        for (int64_t j = 0; j < topk; ++j) {
            int64_t e = ids[t * topk + j];
            if (e < 0 || e >= E) { bad = 1; continue; }
            const uint16_t* xin = x_per_slot ? x + (t * topk + j) * K : x + t * K;
            const uint32_t* wq_e = wq + e * N * (K / 8);
            const uint16_t* s_e = scale + e * N * G;
            const uint8_t* z_e = zero + e * N * G;
            for (int64_t n = 0; n < N; ++n) {
                double acc = 0.0;
                for (int64_t k = 0; k < K; ++k)
                    acc += oracle_bf16_to_double(xin[k]) *
                           oracle_weight(wq_e, s_e, z_e, K, g, n, k);
                if (route_w)
                    y[t * N + n] += (double)route_w[t * topk + j] * acc;
                else
                    y[(t * topk + j) * N + n] = acc;
            }
        }
    return bad ? -1 : 0;
}

/* The whole routed FFN chain for M tokens (see the header comment):
 * gate/up experts are [E][F][H] (F = intermediate width, H = hidden),
 * down experts are [E][H][F]; out is [M][H] in fp64.
 * Scratch: gate_bf/up_bf/h_bf are caller arrays of M*topk*F uint16, d is
 * M*topk*H doubles (kept so a test can inspect the stages). */
int oracle_moe_ffn(const uint16_t* x, const int32_t* ids, const float* route_w,
                   const uint32_t* wq_gate, const uint16_t* s_gate, const uint8_t* z_gate,
                   const uint32_t* wq_up, const uint16_t* s_up, const uint8_t* z_up,
                   const uint32_t* wq_down, const uint16_t* s_down, const uint8_t* z_down,
                   uint16_t* gate_bf, uint16_t* up_bf, uint16_t* h_bf, double* d, double* out,
                   int64_t M, int64_t topk, int64_t E, int64_t H, int64_t F, int64_t g)
{
    int64_t S = M * topk;
    int bad = 0;
    for (int64_t t = 0; t < M; ++t)
        for (int64_t j = 0; j < topk; ++j) {
            int64_t e = ids[t * topk + j];
            if (e < 0 || e >= E) { bad = 1; continue; }
            int64_t sl = t * topk + j;
            const uint16_t* xt = x + t * H;
            int64_t Gh = H / g;
            for (int64_t f = 0; f < F; ++f) {
                double ag = 0.0, au = 0.0;
                for (int64_t k = 0; k < H; ++k) {
                    double xv = oracle_bf16_to_double(xt[k]);
                    ag += xv * oracle_weight(wq_gate + e * F * (H / 8), s_gate + e * F * Gh,
                                             z_gate + e * F * Gh, H, g, f, k);
                    au += xv * oracle_weight(wq_up + e * F * (H / 8), s_up + e * F * Gh,
                                             z_up + e * F * Gh, H, g, f, k);
                }
                gate_bf[sl * F + f] = oracle_bf16_round(ag);
                up_bf[sl * F + f] = oracle_bf16_round(au);
            }
        }
    oracle_swiglu(gate_bf, up_bf, h_bf, S * F);
    for (int64_t i = 0; i < M * H; ++i) out[i] = 0.0;
    for (int64_t t = 0; t < M; ++t)
        for (int64_t j = 0; j < topk; ++j) {
            int64_t e = ids[t * topk + j];
            if (e < 0 || e >= E) continue;
            int64_t sl = t * topk + j;
            int64_t Gf = F / g;
            for (int64_t n = 0; n < H; ++n) {
                double acc = 0.0;
                for (int64_t k = 0; k < F; ++k)
                    acc += oracle_bf16_to_double(h_bf[sl * F + k]) *
                           oracle_weight(wq_down + e * H * (F / 8), s_down + e * H * Gf,
                                         z_down + e * H * Gf, F, g, n, k);
                d[sl * H + n] = acc;
                out[t * H + n] += (double)route_w[t * topk + j] * acc;
            }
        }
    return bad ? -1 : 0;
}
