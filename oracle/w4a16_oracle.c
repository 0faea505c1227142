/*
 * CPU oracle for the int4 group-quantised, weight-only, affine linear layer
 * (W4A16).  TEST INFRASTRUCTURE: only the test suite, the smoke check and the
 * benchmark's CPU-baseline / reference arm may load this library.  It shares
 * no source with the CUDA library and includes none of its headers.
 *
 * Everything is plain scalar C in binary64, with no blocking, fusion or
 * reordering beyond what the definitions below state.  Compile with
 * -ffp-contract=off so that every + and * is a separately rounded IEEE
 * operation on every host.
 *
 * Sources (page title, section):
 *  - "The inference engine - Mojo 1.0 on Metal", "Crossing Mojo 1.0": the
 *    decode path is a weight-streaming GEMV with on-device token selection;
 *    prefill dequantises each weight once into a transposed half-precision
 *    scratch and runs a half-precision GEMM.  "What's inside the engine
 *    today": greedy / top-k selection checked bit-exact against a host
 *    reference; int4 projections and LM head.
 *  - "engine-mlx", "Tech details": models in the MLX 4-bit quantised format.
 *  - "Engineering investigation ... 10x faster?", "Selective quantization":
 *    nn.quantize with affine quantisation, group size 64.
 *  - "The inference engine - Mojo 1.0 on Metal", "What's inside the engine
 *    today" and the appendix on porting MLX's kernels: that engine's own
 *    weights are symmetric int4 in groups of 128 (a scale, no bias).
 *
 * Readings (the pages print neither the formula nor the packing):
 *  - affine dequantisation per group of G consecutive k (G = 64 in the
 *    workloads; any G dividing K here):
 *        w[n][k] = scale[n][k/G] * q[n][k] + bias[n][k/G],  q in 0..15;
 *  - symmetric codes (no bias array, passed as NULL): the code is a signed
 *    4-bit value stored with offset 8,
 *        w[n][k] = scale[n][k/G] * (q[n][k] - 8);
 *  - qweight is uint32 [N][K/8]; word j of row n holds q[n][8j+i] in bits
 *    4i..4i+3 (lowest nibble = lowest k), the MLX packing order;
 *  - scales and biases are binary16 [N][K/G], row-major;
 *  - the dequantised half scratch is the correctly rounded (round to nearest,
 *    ties to even) binary16 of the exact real scale*q + bias (or
 *    scale*(q - 8)), stored transposed as w16[K][N]; a zero result keeps the
 *    sign binary64 arithmetic gives it;
 *  - token selection orders logits by value, descending, ties to the lowest
 *    index.
 *
 * Exactness: a binary16 value is an 11-bit integer times 2^e with
 * -24 <= e <= 5, so scale*q (q < 16) is exact in binary64 and the sum
 * scale*q + bias spans at most 20 + 24 + 1 bits < 53: dequant_exact is the
 * exact real value.  GEMV and GEMM sums are binary64 in k-ascending order.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- binary16 <-> binary64 (IEEE 754-2008, 16-bit interchange format) ---- */

/* Exact value of a binary16 bit pattern: 1 sign bit, 5 exponent bits
 * (bias 15), 10 fraction bits; exponent 0 encodes subnormals f * 2^-24. */
double orc_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int f = h & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);
    return sign ? -v : v;
}

/* Round a non-negative binary64 value that is below 2^12 to an integer,
 * ties to even.  m - floor(m) is exact for such m. */
static double round_half_even(double m)
{
    double fl = floor(m);
    double d = m - fl;
    if (d > 0.5)
        return fl + 1.0;
    if (d < 0.5)
        return fl;
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/* Correctly rounded binary64 -> binary16 conversion, round to nearest with
 * ties to even; overflow to infinity; sign of zero kept; NaN -> quiet NaN. */
uint16_t orc_double_to_half(double v)
{
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (isnan(v))
        return (uint16_t)(sign | 0x7E00);
    if (isinf(a))
        return (uint16_t)(sign | 0x7C00);
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: the quantum is 2^-24 */
        double r = round_half_even(ldexp(a, 24)); /* 0 .. 1024 */
        return (uint16_t)(sign | (uint16_t)r);   /* 1024 -> min normal */
    }
    int e;
    frexp(a, &e);                 /* a in [2^(e-1), 2^e) */
    int E = e - 1;                /* unbiased binary16 exponent */
    double r = round_half_even(ldexp(a, 10 - E)); /* 1024 .. 2048 */
    if (r == 2048.0) {
        r = 1024.0;
        E += 1;
    }
    if (E > 15)
        return (uint16_t)(sign | 0x7C00);
    return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | (uint16_t)(r - 1024.0));
}

/* ---- unpack and dequantise ---- */

/* q[n][k] = bits 4*(k%8) .. 4*(k%8)+3 of word qweight[n][k/8]. */
void orc_unpack(const uint32_t *qweight, int N, int K, uint8_t *q)
{
    for (int n = 0; n < N; ++n)
        for (int k = 0; k < K; ++k) {
            uint32_t word = qweight[(size_t)n * (K / 8) + k / 8];
            q[(size_t)n * K + k] = (uint8_t)((word >> (4 * (k % 8))) & 0xFu);
        }
}

/* Exact dequantised weight of one element; biases == NULL: symmetric codes.
 * s * (q - 8) has at most 11 + 4 significant bits: exact in binary64. */
static double dequant_one(const uint32_t *qweight, const uint16_t *scales,
                          const uint16_t *biases, int K, int G, int n, int k)
{
    uint32_t word = qweight[(size_t)n * (K / 8) + k / 8];
    int q = (int)((word >> (4 * (k % 8))) & 0xFu);
    double s = orc_half_to_double(scales[(size_t)n * (K / G) + k / G]);
    if (biases == NULL)
        return s * (double)(q - 8);
    double b = orc_half_to_double(biases[(size_t)n * (K / G) + k / G]);
    return s * (double)q + b;
}

/* w[r][k] = scale*q + bias (exact) for the listed rows; w is [nrows][K]. */
void orc_dequant_exact_rows(const uint32_t *qweight, const uint16_t *scales,
                            const uint16_t *biases, int K, int G,
                            const int32_t *rows, int nrows, double *w)
{
    for (int r = 0; r < nrows; ++r)
        for (int k = 0; k < K; ++k)
            w[(size_t)r * K + k] = dequant_one(qweight, scales, biases, K, G, rows[r], k);
}

/* Transposed half scratch w16[k][n] = RNE_binary16(scale*q + bias). */
void orc_dequant_f16_t(const uint32_t *qweight, const uint16_t *scales,
                       const uint16_t *biases, int N, int K, int G, uint16_t *w16)
{
    for (int n = 0; n < N; ++n)
        for (int k = 0; k < K; ++k)
            w16[(size_t)k * N + n] =
                orc_double_to_half(dequant_one(qweight, scales, biases, K, G, n, k));
}

/* The same values for the listed rows only, as out[r][k] (row r of W, i.e.
 * column rows[r] of the transposed scratch). */
void orc_dequant_f16_rows(const uint32_t *qweight, const uint16_t *scales,
                          const uint16_t *biases, int K, int G,
                          const int32_t *rows, int nrows, uint16_t *out)
{
    for (int r = 0; r < nrows; ++r)
        for (int k = 0; k < K; ++k)
            out[(size_t)r * K + k] =
                orc_double_to_half(dequant_one(qweight, scales, biases, K, G, rows[r], k));
}

/* ---- GEMV: y[m][n] = sum_k w[n][k] * x[m][k] ---- */

/* For the listed output rows n = rows[r]:
 *   y[m][r]      = sum_k w[n][k] * x[m][k]      (binary64, k ascending)
 *   absdot[m][r] = sum_k |w[n][k] * x[m][k]|
 * x is binary16 [M][K]; y and absdot are [M][nrows]. */
void orc_gemv_rows(const uint16_t *x, const uint32_t *qweight, const uint16_t *scales,
                   const uint16_t *biases, int M, int K, int G,
                   const int32_t *rows, int nrows, double *y, double *absdot)
{
    for (int m = 0; m < M; ++m)
        for (int r = 0; r < nrows; ++r) {
            double acc = 0.0, aacc = 0.0;
            for (int k = 0; k < K; ++k) {
                double w = dequant_one(qweight, scales, biases, K, G, rows[r], k);
                double p = w * orc_half_to_double(x[(size_t)m * K + k]);
                acc += p;
                aacc += fabs(p);
            }
            y[(size_t)m * nrows + r] = acc;
            if (absdot)
                absdot[(size_t)m * nrows + r] = aacc;
        }
}

/* ---- token selection: top-k by (value desc, index asc) ---- */

static const double *g_sort_vals;

static int cmp_rank(const void *pa, const void *pb)
{
    int32_t a = *(const int32_t *)pa, b = *(const int32_t *)pb;
    double va = g_sort_vals[a], vb = g_sort_vals[b];
    if (va > vb)
        return -1;
    if (va < vb)
        return 1;
    return (a < b) ? -1 : (a > b);
}

/* Sort all N indices by (logits desc, index asc) and keep the first k.
 * Not thread-safe (qsort comparator state). */
void orc_topk(const double *logits, int N, int k, int32_t *idx, double *val)
{
    int32_t *order = (int32_t *)malloc(sizeof(int32_t) * (size_t)N);
    for (int i = 0; i < N; ++i)
        order[i] = i;
    g_sort_vals = logits;
    qsort(order, (size_t)N, sizeof(int32_t), cmp_rank);
    for (int i = 0; i < k; ++i) {
        idx[i] = order[i];
        val[i] = logits[order[i]];
    }
    free(order);
}

/* ---- dense half GEMM: y[m][n] = sum_k x16[m][k] * w16[k][n] ---- */

/* Selected entries (ms[i], ns[i]); x16 is [M][K], w16 is [K][N]; binary64,
 * k ascending; absdot[i] = sum_k |x16 * w16|. */
void orc_gemm_entries(const uint16_t *x16, const uint16_t *w16, int N, int K,
                      const int32_t *ms, const int32_t *ns, int count,
                      double *y, double *absdot)
{
    for (int i = 0; i < count; ++i) {
        double acc = 0.0, aacc = 0.0;
        for (int k = 0; k < K; ++k) {
            double p = orc_half_to_double(x16[(size_t)ms[i] * K + k]) *
                       orc_half_to_double(w16[(size_t)k * N + ns[i]]);
            acc += p;
            aacc += fabs(p);
        }
        y[i] = acc;
        if (absdot)
            absdot[i] = aacc;
    }
}

/* Full product for small cases: y is [M][N]. */
void orc_gemm(const uint16_t *x16, const uint16_t *w16, int M, int N, int K,
              double *y, double *absdot)
{
    for (int m = 0; m < M; ++m)
        for (int n = 0; n < N; ++n) {
            double acc = 0.0, aacc = 0.0;
            for (int k = 0; k < K; ++k) {
                double p = orc_half_to_double(x16[(size_t)m * K + k]) *
                           orc_half_to_double(w16[(size_t)k * N + n]);
                acc += p;
                aacc += fabs(p);
            }
            y[(size_t)m * N + n] = acc;
            if (absdot)
                absdot[(size_t)m * N + n] = aacc;
        }
}
