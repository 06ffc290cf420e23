/*
 * qmm_oracle.c -- plain CPU oracle for GGUF Q4_0 / Q8_0 block-quantized
 * matrix products.  TEST INFRASTRUCTURE ONLY (see qmm_oracle.h): it is the
 * definition the GPU path is checked against and is never part of it.
 *
 * Everything follows the definition literally: decode one weight from its
 * block, multiply by the activation, add into a binary64 sum.  There is no
 * blocking, vectorisation or reordering; the only parallelism is an OpenMP
 * loop over independent outputs, which does not change any sum.
 *
 * Build: cc -O2 -ffp-contract=off -fopenmp -shared -fPIC (no fast-math).
 */
#include "qmm_oracle.h"

#include <math.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define QK 32               /* weights per block (both formats)          */
#define Q4_0_BYTES 18       /* 2-byte binary16 d + 16 bytes of nibbles    */
#define Q8_0_BYTES 34       /* 2-byte binary16 d + 32 int8 values         */

static int g_threads = 0;

void qmm_oracle_set_threads(int nthreads) { g_threads = nthreads; }

int qmm_oracle_get_threads(void) {
#ifdef _OPENMP
    return g_threads > 0 ? g_threads : omp_get_max_threads();
#else
    return 1;
#endif
}

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction
 * bits.  Exponent 0 = zero/subnormal (fraction * 2^-24), exponent 31 =
 * infinity (fraction 0) or NaN. */
double qmm_oracle_fp16_to_f64(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);
    } else if (e == 31) {
        v = (f == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(1024 + f), e - 25);
    }
    return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE binary32. */
double qmm_oracle_bf16_to_f64(uint16_t h) {
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* The scale d of a block: little-endian binary16 at bytes 0-1. */
static double block_scale(const uint8_t *blk) {
    uint16_t h = (uint16_t)(blk[0] | ((uint16_t)blk[1] << 8));
    return qmm_oracle_fp16_to_f64(h);
}

/* Weight j (0..31) of a Q4_0 block: qs = blk + 2; weight j < 16 is the low
 * nibble of qs[j], weight j >= 16 the high nibble of qs[j-16];
 * w = (nibble - 8) * d.  The product is formed as (double)(nibble-8) * d so
 * that the sign of a zero follows IEEE multiplication. */
static double q4_0_weight(const uint8_t *blk, int j) {
    const uint8_t *qs = blk + 2;
    int nib = (j < 16) ? (qs[j] & 0x0f) : (qs[j - 16] >> 4);
    return (double)(nib - 8) * block_scale(blk);
}

/* Weight j of a Q8_0 block: w = q[j] * d, q a two's-complement int8. */
static double q8_0_weight(const uint8_t *blk, int j) {
    int8_t q = (int8_t)blk[2 + j];
    return (double)q * block_scale(blk);
}

typedef double (*weight_fn)(const uint8_t *blk, int j);

/* w[n][k] of the whole matrix. */
static double weight_at(const uint8_t *w, int64_t k, int64_t n, int64_t kk,
                        weight_fn fn, int block_bytes) {
    int64_t nb = k / QK;
    const uint8_t *blk = w + (n * nb + kk / QK) * block_bytes;
    return fn(blk, (int)(kk % QK));
}

static void dequant(const uint8_t *w, int64_t n, int64_t k, float *out,
                    weight_fn fn, int block_bytes) {
    int64_t total = n * k;
#pragma omp parallel for schedule(static) num_threads(qmm_oracle_get_threads())
    for (int64_t i = 0; i < total; i++) {
        /* exact: |nibble-8| <= 8 (or |q| <= 128) times an 11-bit significand */
        out[i] = (float)weight_at(w, k, i / k, i % k, fn, block_bytes);
    }
}

void qmm_oracle_dequant_q4_0(const uint8_t *w, int64_t n, int64_t k, float *out) {
    dequant(w, n, k, out, q4_0_weight, Q4_0_BYTES);
}

void qmm_oracle_dequant_q8_0(const uint8_t *w, int64_t n, int64_t k, float *out) {
    dequant(w, n, k, out, q8_0_weight, Q8_0_BYTES);
}

/* One output: sum over k of x[k] * w[n][k] in binary64, and sum of |x*w|. */
typedef double (*act_fn)(const void *x, int64_t idx);

static double act_f32(const void *x, int64_t idx) {
    return (double)((const float *)x)[idx];
}

static double act_bf16(const void *x, int64_t idx) {
    return qmm_oracle_bf16_to_f64(((const uint16_t *)x)[idx]);
}

static void dot(const uint8_t *w, const void *x, int64_t k, int64_t mi, int64_t ni,
                weight_fn wf, int block_bytes, act_fn af, double *y, double *bound) {
    double acc = 0.0, abs_acc = 0.0;
    for (int64_t kk = 0; kk < k; kk++) {
        double p = af(x, mi * k + kk) * weight_at(w, k, ni, kk, wf, block_bytes);
        acc += p;
        abs_acc += fabs(p);
    }
    *y = acc;
    if (bound) *bound = abs_acc;
}

static void product(const uint8_t *w, const void *x, int64_t m, int64_t n, int64_t k,
                    double *y, double *bound, weight_fn wf, int block_bytes, act_fn af) {
    int64_t total = m * n;
#pragma omp parallel for schedule(dynamic, 16) num_threads(qmm_oracle_get_threads())
    for (int64_t i = 0; i < total; i++) {
        int64_t mi = i / n, ni = i % n;
        dot(w, x, k, mi, ni, wf, block_bytes, af, &y[i], bound ? &bound[i] : NULL);
    }
}

static void product_at(const uint8_t *w, const void *x, int64_t k, const int64_t *mi,
                       const int64_t *ni, int64_t count, double *y, double *bound,
                       weight_fn wf, int block_bytes, act_fn af) {
#pragma omp parallel for schedule(dynamic, 4) num_threads(qmm_oracle_get_threads())
    for (int64_t i = 0; i < count; i++) {
        dot(w, x, k, mi[i], ni[i], wf, block_bytes, af, &y[i], bound ? &bound[i] : NULL);
    }
}

void qmm_oracle_gemv_q4_0(const uint8_t *w, const float *x, int64_t m, int64_t n,
                          int64_t k, double *y, double *bound) {
    product(w, x, m, n, k, y, bound, q4_0_weight, Q4_0_BYTES, act_f32);
}

void qmm_oracle_gemv_q8_0(const uint8_t *w, const float *x, int64_t m, int64_t n,
                          int64_t k, double *y, double *bound) {
    product(w, x, m, n, k, y, bound, q8_0_weight, Q8_0_BYTES, act_f32);
}

void qmm_oracle_gemm_q4_0(const uint8_t *w, const uint16_t *x_bf16, int64_t m,
                          int64_t n, int64_t k, double *y, double *bound) {
    product(w, x_bf16, m, n, k, y, bound, q4_0_weight, Q4_0_BYTES, act_bf16);
}

void qmm_oracle_gemv_q4_0_at(const uint8_t *w, const float *x, int64_t k,
                             const int64_t *mi, const int64_t *ni, int64_t count,
                             double *y, double *bound) {
    product_at(w, x, k, mi, ni, count, y, bound, q4_0_weight, Q4_0_BYTES, act_f32);
}

void qmm_oracle_gemv_q8_0_at(const uint8_t *w, const float *x, int64_t k,
                             const int64_t *mi, const int64_t *ni, int64_t count,
                             double *y, double *bound) {
    product_at(w, x, k, mi, ni, count, y, bound, q8_0_weight, Q8_0_BYTES, act_f32);
}

void qmm_oracle_gemm_q4_0_at(const uint8_t *w, const uint16_t *x_bf16, int64_t k,
                             const int64_t *mi, const int64_t *ni, int64_t count,
                             double *y, double *bound) {
    product_at(w, x_bf16, k, mi, ni, count, y, bound, q4_0_weight, Q4_0_BYTES, act_bf16);
}

/* GELU, tanh form, in binary64 (libm tanh). */
static double gelu_tanh(double z) {
    const double c = sqrt(2.0 / 3.14159265358979323846);
    return 0.5 * z * (1.0 + tanh(c * (z + 0.044715 * z * z * z)));
}

void qmm_oracle_geglu_q4_0(const uint8_t *wg, const uint8_t *wu, const float *x, int64_t m,
                           int64_t n, int64_t k, double *h, double *g, double *u,
                           double *bound_g, double *bound_u) {
    int64_t total = m * n;
#pragma omp parallel for schedule(dynamic, 16) num_threads(qmm_oracle_get_threads())
    for (int64_t i = 0; i < total; i++) {
        int64_t mi = i / n, ni = i % n;
        double gv, uv, bg, bu;
        dot(wg, x, k, mi, ni, q4_0_weight, Q4_0_BYTES, act_f32, &gv, &bg);
        dot(wu, x, k, mi, ni, q4_0_weight, Q4_0_BYTES, act_f32, &uv, &bu);
        h[i] = gelu_tanh(gv) * uv;
        if (g) g[i] = gv;
        if (u) u[i] = uv;
        if (bound_g) bound_g[i] = bg;
        if (bound_u) bound_u[i] = bu;
    }
}

void qmm_oracle_geglu_q4_0_at(const uint8_t *wg, const uint8_t *wu, const float *x, int64_t k,
                              const int64_t *mi, const int64_t *ni, int64_t count, double *h,
                              double *g, double *u, double *bound_g, double *bound_u) {
#pragma omp parallel for schedule(dynamic, 4) num_threads(qmm_oracle_get_threads())
    for (int64_t i = 0; i < count; i++) {
        double gv, uv, bg, bu;
        dot(wg, x, k, mi[i], ni[i], q4_0_weight, Q4_0_BYTES, act_f32, &gv, &bg);
        dot(wu, x, k, mi[i], ni[i], q4_0_weight, Q4_0_BYTES, act_f32, &uv, &bu);
        h[i] = gelu_tanh(gv) * uv;
        if (g) g[i] = gv;
        if (u) u[i] = uv;
        if (bound_g) bound_g[i] = bg;
        if (bound_u) bound_u[i] = bu;
    }
}
