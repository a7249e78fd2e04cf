/*
 * Reference oracle for the ~3-bit expert weights -- TEST INFRASTRUCTURE ONLY.
 *
 * Built into the same library as w4a16_oracle.c and under the same rule: only
 * the test suite, the smoke check and the benchmark's CPU-baseline leg load
 * it; the product path never calls it and shares no code or table with it.
 *
 * The local-kimi README (hardware-requirements paragraph) says that fitting a
 * 24 GB card needs the expert weights near three bits, and gives no format.
 * The format below is this library's reading, chosen so that it is exactly
 * three bits per code and so that a GPU decodes it with a few bit operations:
 *
 *   codes      q in 0..7 (unsigned), W[n][k] = (q - zero[n][k/g]) * scale[n][k/g]
 *              with the same bf16 scale and uint8 zero point as the INT4 path
 *   row n      K/128 blocks of 48 bytes (twelve little-endian 32-bit words),
 *              block b holding codes k = 128 b .. 128 b + 127; K % 128 == 0
 *   block      four chunks of 32 codes; chunk c (k = 128 b + 32 c + i,
 *              i = 0..31) in words 3c, 3c+1, 3c+2 of the block
 *   chunk      for i < 30: word 3c + i/10 holds the code's three bits (lowest
 *              bit first) at bit 16 * ((i % 10) / 5) + 3 * ((i % 10) % 5) --
 *              five codes in bits 0..14 of each 16-bit half, bits 15 and 31
 *              left over;
 *              for i = 30 and 31: bit j (j = 0, 1, 2) of the code is bit 15
 *              (i = 30) or bit 31 (i = 31) of word 3c + j.
 *
 * So the 96 bits of a chunk hold its 32 codes exactly once, and uniform codes
 * make uniform words.  Everything else -- GEMV, the routed SwiGLU FFN chain,
 * the bf16 rounding points -- is the INT4 path's definition (w4a16_oracle.c)
 * with this code lookup in place of the nibble lookup.
 */
#include <math.h>
#include <stdint.h>

double oracle_bf16_to_double(uint16_t b);
uint16_t oracle_bf16_round(double v);
void oracle_swiglu(const uint16_t* gate, const uint16_t* up, uint16_t* h, int64_t count);

/* ---- packing ------------------------------------------------------------ */

/* 32-bit words per row of K codes */
static inline int64_t oracle3_row_words(int64_t K) { return K / 128 * 12; }

/* word index (within the row) and bit of bit j (0..2) of code k */
static inline void oracle3_bit_place(int64_t k, int j, int64_t* word, int* bit)
{
    int64_t b = k / 128;
    int64_t c = (k % 128) / 32;
    int64_t i = k % 32;
    int64_t first = 12 * b + 3 * c;
    if (i < 30) {
        int64_t r = i % 10;
        *word = first + i / 10;
        *bit = (int)(16 * (r / 5) + 3 * (r % 5)) + j;
    } else {
        *word = first + j;
        *bit = (i == 30) ? 15 : 31;
    }
}

static inline int oracle3_code(const uint32_t* wq3, int64_t K, int64_t n, int64_t k)
{
    const uint32_t* row = wq3 + n * oracle3_row_words(K);
    int q = 0;
    for (int j = 0; j < 3; ++j) {
        int64_t word;
        int bit;
        oracle3_bit_place(k, j, &word, &bit);
        q |= (int)((row[word] >> bit) & 1u) << j;
    }
    return q;
}

/* codes[N][K] (each 0..7; higher bits ignored) -> wq3[N][3K/32] */
void oracle3_pack(const uint8_t* codes, uint32_t* wq3, int64_t N, int64_t K)
{
    int64_t wpr = oracle3_row_words(K);
    for (int64_t i = 0; i < N * wpr; ++i) wq3[i] = 0;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            for (int j = 0; j < 3; ++j) {
                int64_t word;
                int bit;
                oracle3_bit_place(k, j, &word, &bit);
                wq3[n * wpr + word] |= (uint32_t)((codes[n * K + k] >> j) & 1) << bit;
            }
}

void oracle3_unpack(const uint32_t* wq3, uint8_t* codes, int64_t N, int64_t K)
{
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            codes[n * K + k] = (uint8_t)oracle3_code(wq3, K, n, k);
}

/* ---- dequantisation and GEMV -------------------------------------------- */

static inline double oracle3_weight(const uint32_t* wq3, const uint16_t* scale,
                                    const uint8_t* zero, int64_t K, int64_t g,
                                    int64_t n, int64_t k)
{
    int64_t G = K / g;
    double s = oracle_bf16_to_double(scale[n * G + k / g]);
    double z = (double)zero[n * G + k / g];
    return ((double)oracle3_code(wq3, K, n, k) - z) * s;
}

/* w[N][K] = (code - zero) * scale, exact in fp64. */
void oracle3_dequant(const uint32_t* wq3, const uint16_t* scale, const uint8_t* zero,
                     double* w, int64_t N, int64_t K, int64_t g)
{
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            w[n * K + k] = oracle3_weight(wq3, scale, zero, K, g, n, k);
}

/* y[m][n] = sum_k x[m][k] * W[n][k], fp64, k ascending. */
void oracle3_gemv(const uint16_t* x, const uint32_t* wq3, const uint16_t* scale,
                  const uint8_t* zero, double* y, int64_t M, int64_t N, int64_t K, int64_t g)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += oracle_bf16_to_double(x[m * K + k]) *
                       oracle3_weight(wq3, scale, zero, K, g, n, k);
            y[m * N + n] = acc;
        }
}

/* ---- expert-indexed GEMV over INT3 experts ------------------------------ */

/* The expert-indexed GEMV of oracle_moe_gemv with INT3 experts: for token t
 * and slot j with e = ids[t][j], d[t][j][n] = sum_k xin[k] * W_e[n][k], xin
 * = x[t] (x_per_slot == 0, x [M][K]) or x[t][j] (x [M][topk][K]); expert
 * e's rows start at wq3 + e*N*3K/32, scale and zero + e*N*(K/g).  Without
 * route_w, d goes to y[M][topk][N] (zero rows for an invalid id); with it,
 * y[t][n] = sum_j route_w[t][j] * d[t][j][n] (fp64, j ascending, invalid ids
 * skipped).  Returns -1 if an id is outside [0, E). */
int oracle3_moe_gemv(const uint16_t* x, int x_per_slot, const int32_t* ids,
                     const float* route_w, const uint32_t* wq3, const uint16_t* scale,
                     const uint8_t* zero, double* y, int64_t M, int64_t topk, int64_t E,
                     int64_t N, int64_t K, int64_t g)
{
    int bad = 0;
    int64_t G = K / g, wpr = oracle3_row_words(K);
    if (route_w)
        for (int64_t i = 0; i < M * N; ++i) y[i] = 0.0;
    for (int64_t t = 0; t < M; ++t)
        for (int64_t j = 0; j < topk; ++j) {
            int64_t e = ids[t * topk + j];
            if (e < 0 || e >= E) {
                bad = 1;
                if (!route_w)
                    for (int64_t n = 0; n < N; ++n) y[(t * topk + j) * N + n] = 0.0;
                continue;
            }
            const uint16_t* xin = x_per_slot ? x + (t * topk + j) * K : x + t * K;
            for (int64_t n = 0; n < N; ++n) {
                double acc = 0.0;
                for (int64_t k = 0; k < K; ++k)
                    acc += oracle_bf16_to_double(xin[k]) *
                           oracle3_weight(wq3 + e * N * wpr, scale + e * N * G, zero + e * N * G,
                                          K, g, n, k);
                if (route_w)
                    y[t * N + n] += (double)route_w[t * topk + j] * acc;
                else
                    y[(t * topk + j) * N + n] = acc;
            }
        }
    return bad ? -1 : 0;
}

/* ---- routed SwiGLU FFN over INT3 experts -------------------------------- */

/* The chain of oracle_moe_ffn with INT3 experts: gate/up banks [E][F] rows
 * of H codes, down bank [E][H] rows of F codes (3*K/32 words per row); the
 * same scratch arrays and the same return value (-1 if an id is outside
 * [0, E), that slot skipped). */
int oracle3_moe_ffn(const uint16_t* x, const int32_t* ids, const float* route_w,
                    const uint32_t* wq_gate, const uint16_t* s_gate, const uint8_t* z_gate,
                    const uint32_t* wq_up, const uint16_t* s_up, const uint8_t* z_up,
                    const uint32_t* wq_down, const uint16_t* s_down, const uint8_t* z_down,
                    uint16_t* gate_bf, uint16_t* up_bf, uint16_t* h_bf, double* d, double* out,
                    int64_t M, int64_t topk, int64_t E, int64_t H, int64_t F, int64_t g)
{
    int64_t S = M * topk;
    int64_t Gh = H / g, Gf = F / g;
    int64_t wh = oracle3_row_words(H), wf = oracle3_row_words(F);
    int bad = 0;
    for (int64_t t = 0; t < M; ++t)
        for (int64_t j = 0; j < topk; ++j) {
            int64_t e = ids[t * topk + j];
            if (e < 0 || e >= E) { bad = 1; continue; }
            int64_t sl = t * topk + j;
            const uint16_t* xt = x + t * H;
            for (int64_t f = 0; f < F; ++f) {
                double ag = 0.0, au = 0.0;
                for (int64_t k = 0; k < H; ++k) {
                    double xv = oracle_bf16_to_double(xt[k]);
                    ag += xv * oracle3_weight(wq_gate + e * F * wh, s_gate + e * F * Gh,
                                              z_gate + e * F * Gh, H, g, f, k);
                    au += xv * oracle3_weight(wq_up + e * F * wh, s_up + e * F * Gh,
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
            for (int64_t n = 0; n < H; ++n) {
                double acc = 0.0;
                for (int64_t k = 0; k < F; ++k)
                    acc += oracle_bf16_to_double(h_bf[sl * F + k]) *
                           oracle3_weight(wq_down + e * H * wf, s_down + e * H * Gf,
                                          z_down + e * H * Gf, F, g, n, k);
                d[sl * H + n] = acc;
                out[t * H + n] += (double)route_w[t * topk + j] * acc;
            }
        }
    return bad ? -1 : 0;
}
