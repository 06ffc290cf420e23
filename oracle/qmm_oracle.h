/*
 * qmm_oracle.h -- plain CPU oracle for GGUF Q4_0 / Q8_0 block-quantized
 * matrix products.
 *
 * TEST INFRASTRUCTURE ONLY.  This library is the slow, obviously correct
 * definition that the GPU kernels are checked against.  Only the test suite,
 * the smoke check and the CPU-baseline leg of the benchmark may load it.  It
 * shares no code, header, table or constant with the CUDA library, and the
 * CUDA library never calls it.
 *
 * Source of the method: "Add generated quant-kernel JIT and accelerate Gemma4,
 * BGE-M3, and GLiNER2" (antfly PR #372), section "Validation": each Gemma4
 * decode token runs 342 Q4_0 and one Q8_0 generated quant dispatch, i.e. the
 * products of GGUF block-quantized weights with activations.  The pages name
 * the formats but print no layout; the GGUF layouts used here are:
 *
 *   Q4_0 block (18 bytes, 32 weights): bytes 0-1 = IEEE binary16 scale d,
 *        little endian; bytes 2..17 = qs[0..15].  qs[j] holds weight j in its
 *        low nibble and weight j+16 in its high nibble; w = (nibble - 8) * d.
 *   Q8_0 block (34 bytes, 32 weights): bytes 0-1 = binary16 d (LE), then
 *        32 int8 q[j]; w = q[j] * d.
 *
 * A weight matrix W has N rows and K columns (K a multiple of 32).  Row n is
 * K/32 consecutive blocks and rows are consecutive, so block b of row n starts
 * at byte (n*(K/32) + b) * block_bytes.  Activations are row-major [M][K].
 *
 * Every result is computed in IEEE binary64.  Each dequantized weight is
 * exact in binary64 (and in binary32), every product w*x is exact in
 * binary64, and only the running sums round.  Alongside each output the
 * oracle returns bound = sum_k |w[n][k] * x[m][k]|, the scale of the error
 * tolerance.
 *
 * Parity status: every function here is pinned by the CPU tests (format
 * values, exhaustive binary16 decode against numpy, closed forms, linearity,
 * one-hot columns, brute force on tiny inputs, numpy matmul of the pinned
 * dequantization).
 */
#ifndef QMM_ORACLE_H
#define QMM_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* IEEE 754 binary16 bit pattern -> exact binary64 value (bit-field decode). */
double qmm_oracle_fp16_to_f64(uint16_t h);
/* bfloat16 bit pattern -> exact binary64 value. */
double qmm_oracle_bf16_to_f64(uint16_t h);

/* Dense dequantization: out[n][k] (binary32, exact) from N*K/32 blocks. */
void qmm_oracle_dequant_q4_0(const uint8_t *w, int64_t n, int64_t k, float *out);
void qmm_oracle_dequant_q8_0(const uint8_t *w, int64_t n, int64_t k, float *out);

/* y[m][n] = sum_k x[m][k] * w[n][k] for fp32 x [M][K].  y and bound are
 * binary64 [M][N]; bound may be NULL. */
void qmm_oracle_gemv_q4_0(const uint8_t *w, const float *x, int64_t m, int64_t n,
                          int64_t k, double *y, double *bound);
void qmm_oracle_gemv_q8_0(const uint8_t *w, const float *x, int64_t m, int64_t n,
                          int64_t k, double *y, double *bound);

/* Same product with bf16 activations X [M][K] given as raw bf16 bit patterns
 * (the exact bf16 values are used; W is not rounded). */
void qmm_oracle_gemm_q4_0(const uint8_t *w, const uint16_t *x_bf16, int64_t m,
                          int64_t n, int64_t k, double *y, double *bound);

/* Sampled outputs: for i < count, y[i] and bound[i] are output
 * (mi[i], ni[i]) of the corresponding full product above. */
void qmm_oracle_gemv_q4_0_at(const uint8_t *w, const float *x, int64_t k,
                             const int64_t *mi, const int64_t *ni, int64_t count,
                             double *y, double *bound);
void qmm_oracle_gemv_q8_0_at(const uint8_t *w, const float *x, int64_t k,
                             const int64_t *mi, const int64_t *ni, int64_t count,
                             double *y, double *bound);
void qmm_oracle_gemm_q4_0_at(const uint8_t *w, const uint16_t *x_bf16, int64_t k,
                             const int64_t *mi, const int64_t *ni, int64_t count,
                             double *y, double *bound);

/* Gated feed-forward input (GeGLU): the fused FFN paths of "Add generated
 * quant-kernel JIT and accelerate Gemma4, BGE-M3, and GLiNER2" (section
 * "Summary").  The pages do not name the activation; the reading taken is
 * the Gemma family's GELU in its tanh form, applied to the gate:
 *   g = x . Wg^T,  u = x . Wu^T  (Q4_0 weights, fp32 x, binary64 sums),
 *   h[m][n] = gelu(g[m][n]) * u[m][n],
 *   gelu(z) = z/2 * (1 + tanh(sqrt(2/pi) * (z + 0.044715 z^3))).
 * h, g, u, bound_g, bound_u are binary64 [M][N]; the bounds are those of the
 * two products (sum_k |w*x|).  Any output pointer but h may be NULL. */
void qmm_oracle_geglu_q4_0(const uint8_t *wg, const uint8_t *wu, const float *x, int64_t m,
                           int64_t n, int64_t k, double *h, double *g, double *u,
                           double *bound_g, double *bound_u);

/* Sampled outputs of qmm_oracle_geglu_q4_0: for i < count, element i of
 * each output array is that function's output (mi[i], ni[i]). */
void qmm_oracle_geglu_q4_0_at(const uint8_t *wg, const uint8_t *wu, const float *x, int64_t k,
                              const int64_t *mi, const int64_t *ni, int64_t count, double *h,
                              double *g, double *u, double *bound_g, double *bound_u);

/* Host threads used by the loops over outputs (OpenMP); <=0 means all. */
void qmm_oracle_set_threads(int nthreads);
int qmm_oracle_get_threads(void);

#ifdef __cplusplus
}
#endif

#endif
