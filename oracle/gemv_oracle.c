/*
 * Plain CPU oracle for the decode GEMV  y[b][n] = sum_k W[n][k] * x[b][k].
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or call
 * this file: only the tests, the package's smoke check and the benchmark's CPU
 * baseline leg use it. It shares no code, header or constant with the CUDA
 * library.
 *
 * What it follows:
 *   - "Decode GEMV at half of HBM bandwidth" (inferenceinterviews.com), the
 *     split-K listing in "A strong answer": each output row is the dot product of
 *     one weight row (row-major, row stride in elements) with the activation
 *     vector, the BF16 inputs widened before the multiply-add, and columns at or
 *     beyond K masked out. Split-K and vector loads only reorder the additions,
 *     so the oracle is that definition with no reordering at all: k ascending.
 *   - The same page, "What interviewers probe next": the order of additions is
 *     what the reproducibility question turns on, so the oracle fixes one order.
 *   - Precision: the page accumulates in FP32; the oracle accumulates in FP64
 *     so that its own rounding is far below any FP32 result it checks.
 *
 * Layouts (all row-major):
 *   W  : N rows of ldw BF16 values; only columns k < K are read.
 *   x  : B rows of K BF16 values (row stride K).
 *   y  : B rows of N doubles (row stride N).
 *   s  : same shape as y; s[b][n] = sum_k |W[n][k] * x[b][k]|, the scale the
 *        acceptance tolerance is measured against.
 *
 * BF16 -> double: a BF16 value is the high half of an IEEE binary32 pattern,
 * so shifting its 16 bits up by 16 gives that binary32 exactly; widening to
 * double is exact as well.
 */
#include <stdint.h>
#include <math.h>
#include <string.h>

static double bf16_to_double(uint16_t h)
{
    uint32_t bits = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/*
 * Rows [n0, n1) of every batch row. Returns 0, or -1 on a bad argument.
 * y and s hold B*N doubles each; only the columns n in [n0, n1) are written.
 */
int oracle_gemv_f64(const uint16_t *W, const uint16_t *x,
                    int64_t N, int64_t K, int64_t B, int64_t ldw,
                    int64_t n0, int64_t n1, double *y, double *s)
{
    if (!W || !x || !y || !s) return -1;
    if (N < 1 || K < 1 || B < 1 || ldw < K) return -1;
    if (n0 < 0 || n1 > N || n0 > n1) return -1;

    for (int64_t b = 0; b < B; ++b) {
        const uint16_t *xb = x + b * K;
        for (int64_t n = n0; n < n1; ++n) {
            const uint16_t *wn = W + n * ldw;
            double acc = 0.0;
            double mag = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double term = bf16_to_double(wn[k]) * bf16_to_double(xb[k]);
                acc += term;
                mag += term < 0.0 ? -term : term;
            }
            y[b * N + n] = acc;
            s[b * N + n] = mag;
        }
    }
    return 0;
}

/*
 * One output element (b, n), for checking sampled outputs of very large
 * problems without computing every row. Returns 0, or -1 on a bad argument.
 */
int oracle_gemv_f64_one(const uint16_t *W, const uint16_t *x,
                        int64_t N, int64_t K, int64_t B, int64_t ldw,
                        int64_t b, int64_t n, double *y_out, double *s_out)
{
    if (!W || !x || !y_out || !s_out) return -1;
    if (N < 1 || K < 1 || B < 1 || ldw < K) return -1;
    if (b < 0 || b >= B || n < 0 || n >= N) return -1;

    const uint16_t *xb = x + b * K;
    const uint16_t *wn = W + n * ldw;
    double acc = 0.0;
    double mag = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        double term = bf16_to_double(wn[k]) * bf16_to_double(xb[k]);
        acc += term;
        mag += term < 0.0 ? -term : term;
    }
    *y_out = acc;
    *s_out = mag;
    return 0;
}

/*
 * The GEMV with an RMSNorm prologue on x ("GPU performance chains", "Fused
 * RMSNorm traffic": at decode the norm's launches, not its bytes, are the cost,
 * so it is fused into the projection that reads x). RMSNorm scales each
 * activation row by r_b = (mean_k x[b][k]^2 + eps)^(-1/2); its elementwise
 * weight is taken as already folded into W's columns, so
 *
 *     y[b][n] = r_b * sum_k W[n][k] * x[b][k]
 *     s[b][n] = r_b * sum_k |W[n][k] * x[b][k]|   (the tolerance scale)
 *     r[b]    = r_b
 *
 * for rows [n0, n1). FP64 throughout; the mean divides by K. Returns 0, or -1
 * on a bad argument (eps < 0 included).
 */
int oracle_gemv_rmsnorm_f64(const uint16_t *W, const uint16_t *x,
                            int64_t N, int64_t K, int64_t B, int64_t ldw, double eps,
                            int64_t n0, int64_t n1, double *y, double *s, double *r)
{
    if (!r || !(eps >= 0.0)) return -1;
    int rc = oracle_gemv_f64(W, x, N, K, B, ldw, n0, n1, y, s);
    if (rc != 0) return rc;
    for (int64_t b = 0; b < B; ++b) {
        const uint16_t *xb = x + b * K;
        double sq = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double v = bf16_to_double(xb[k]);
            sq += v * v;
        }
        double rb = 1.0 / sqrt(sq / (double)K + eps);
        r[b] = rb;
        for (int64_t n = n0; n < n1; ++n) {
            y[b * N + n] *= rb;
            s[b * N + n] *= rb;
        }
    }
    return 0;
}

/*
 * The GEMV with group-quantised INT4 weights ("Decode GEMV at half of HBM
 * bandwidth", "What interviewers probe next": with INT4 weights the bytes fall
 * four times). Element (n, k) of W is (u - 8) * scale, u its 4-bit code and
 * scale = S[n][k / group] (BF16). Codes are packed eight to a little-endian
 * 32-bit word per row, word w of row n at byte n*ldq + 4w holding
 * k = 8w .. 8w+7: k = 8w + 2j in bits 4j..4j+3, k = 8w + 2j + 1 in bits
 * 16+4j..16+4j+3. Rows [n0, n1); FP64; the same y and tolerance scale s as
 * oracle_gemv_f64. Returns 0, or -1 on a bad argument.
 */
static double w4_element(const uint8_t *Wq, const uint16_t *S, int64_t ldq, int64_t lds,
                         int64_t group, int64_t n, int64_t k)
{
    const uint8_t *p = Wq + n * ldq + 4 * (k / 8);
    uint32_t word = (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
    int64_t i = k % 8;
    int shift = (i % 2 == 0) ? (int)(4 * (i / 2)) : (int)(16 + 4 * (i / 2));
    int code = (int)((word >> shift) & 0xFu);
    return (double)(code - 8) * bf16_to_double(S[n * lds + k / group]);
}

int oracle_gemv_w4_f64(const uint8_t *Wq, const uint16_t *S, const uint16_t *x,
                       int64_t N, int64_t K, int64_t B, int64_t ldq, int64_t lds, int64_t group,
                       int64_t n0, int64_t n1, double *y, double *s)
{
    if (!Wq || !S || !x || !y || !s) return -1;
    if (N < 1 || K < 1 || B < 1 || group < 1 || K % 8 != 0) return -1;
    if (ldq < K / 2 || lds < (K + group - 1) / group) return -1;
    if (n0 < 0 || n1 > N || n0 > n1) return -1;

    for (int64_t b = 0; b < B; ++b) {
        const uint16_t *xrow = x + b * K;
        for (int64_t n = n0; n < n1; ++n) {
            double dot = 0.0;
            double absdot = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double t = w4_element(Wq, S, ldq, lds, group, n, k) * bf16_to_double(xrow[k]);
                dot += t;
                absdot += fabs(t);
            }
            y[b * N + n] = dot;
            s[b * N + n] = absdot;
        }
    }
    return 0;
}

/*
 * The GEMV with FP8 weights ("Decode GEMV at half of HBM bandwidth", "What
 * interviewers probe next": INT4, then FP8 weights, with the unpacking done in
 * registers). Each weight is an 8-bit E4M3 code c: sign in bit 7, exponent
 * field e in bits 3..6 with bias 7, mantissa m in bits 0..2. e = 0 encodes the
 * subnormals (m / 8) * 2^-6; e = 15 with m = 7 is NaN; the format has no
 * infinities, so e = 15 with m < 7 are finite (the largest is 448). Element
 * (n, k) of W is e4m3(Wq[n * ldq + k]) * S[n], with S one FP32 scale per output
 * row. Every product w * S * x is exact in FP64 (4 + 24 + 8 significant bits).
 * Rows [n0, n1); FP64; the same y and tolerance scale s as oracle_gemv_f64.
 * Returns 0, or -1 on a bad argument.
 */
static double e4m3_to_double(uint8_t c)
{
    int e8 = (c >> 3) & 0xF;
    int m8 = c & 0x7;
    double mag8;
    if (e8 == 0xF && m8 == 0x7) return NAN;
    if (e8 == 0) mag8 = ldexp((double)m8 / 8.0, -6);
    else mag8 = ldexp(1.0 + (double)m8 / 8.0, e8 - 7);
    return (c & 0x80) ? -mag8 : mag8;
}

int oracle_gemv_fp8_f64(const uint8_t *Wq, const float *S, const uint16_t *x,
                        int64_t N, int64_t K, int64_t B, int64_t ldq,
                        int64_t n0, int64_t n1, double *y, double *s)
{
    if (!Wq || !S || !x || !y || !s) return -1;
    if (N < 1 || K < 1 || B < 1 || ldq < K) return -1;
    if (n0 < 0 || n1 > N || n0 > n1) return -1;

    for (int64_t b = 0; b < B; ++b) {
        const uint16_t *xr8 = x + b * K;
        for (int64_t n = n0; n < n1; ++n) {
            const uint8_t *row8 = Wq + n * ldq;
            double sum8 = 0.0;
            double abs8 = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double t8 = e4m3_to_double(row8[k]) * (double)S[n] * bf16_to_double(xr8[k]);
                sum8 += t8;
                abs8 += fabs(t8);
            }
            y[b * N + n] = sum8;
            s[b * N + n] = abs8;
        }
    }
    return 0;
}
