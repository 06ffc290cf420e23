/*
 * qmm.h -- C ABI of the GB300 (sm_103a) GGUF block-quantized matmul library
 * (libqmm.so).
 *
 * What it computes.  "Add generated quant-kernel JIT and accelerate Gemma4,
 * BGE-M3, and GLiNER2" (antfly PR #372), section "Validation", counts 343
 * generated quant dispatches per Gemma4 decode token: 342 apply Q4_0 weights
 * and one (the LM head) applies Q8_0 weights.  Its "Summary" adds batching
 * and prefill (the TTFT rows of "Benchmarks").  This library provides those
 * products:
 *
 *   dequant : W (blocks) -> dense fp32 W[N][K], bit-exact
 *   gemv    : y[m][n] = sum_k x[m][k] * w[n][k], fp32 x, M = 1..16 rows
 *             (one weight matrix, or up to four sharing x in one launch)
 *   gemm    : Y[m][n] = sum_k X[m][k] * w[n][k], bf16 X, M >= 1 (prefill),
 *             fused, or in two phases through a bf16 workspace
 *   geglu   : h = gelu(x.Wg^T) * (x.Wu^T), the feed-forward input, for
 *             decode (gemv) and prefill (gemm)
 *
 * Block formats (GGUF; 32 weights per block, K a multiple of 32):
 *   Q4_0, 18 bytes: binary16 scale d (little endian) then qs[16]; qs[j] holds
 *         weight j in its low nibble and weight j+16 in its high nibble;
 *         w = (nibble - 8) * d.
 *   Q8_0, 34 bytes: binary16 d then int8 q[32]; w = q * d.
 *
 * Layout.  W has N rows and K columns; row n is K/32 consecutive blocks and
 * rows are consecutive (block b of row n at byte (n*K/32 + b) * block bytes).
 * Activations and outputs are dense row-major: x[M][K], y[M][N].
 *
 * Ownership and execution.  Every pointer is a caller-owned DEVICE pointer on
 * the current CUDA device.  Outputs are overwritten, never accumulated into.
 * Calls are asynchronous on `stream` (NULL = legacy default stream) and never
 * synchronise.  The library allocates no device memory; its device state is
 * one error word per GPU and the 64 MB scratch array of
 * qmm_gemm_q4_0_prefill (module-scope variables).  Calls on different
 * streams may run concurrently, except qmm_gemm_q4_0_prefill (shared
 * scratch) and _ws calls sharing a workspace.  Kernels are launched with
 * programmatic dependent launch: a call may start while the preceding
 * kernel of this library in the same stream is finishing, and waits for it
 * before reading activations or writing outputs.  A GEMV may read its weight
 * bytes before that wait (weights are read-only model data; no entry point
 * writes block-format bytes), so a weight buffer must not alias the output
 * of the immediately preceding call in the stream.  Kernels from elsewhere
 * never trigger the early start: after them a call starts as usual.
 *
 * Errors.  Arguments are checked before anything is launched; a failed check
 * returns its status and launches nothing.  A launch failure returns
 * QMM_ERR_CUDA; a call that launches several kernels may have launched some
 * of them by then, so after QMM_ERR_CUDA the contents of its outputs (and of
 * any workspace) are undefined.  Device-side waits are bounded: a kernel that gives up
 * records QMM_ERR_TIMEOUT in the device error word, which
 * qmm_get_device_error() reports.  No entry point aborts the process.
 */
#ifndef QMM_H
#define QMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum qmm_status {
    QMM_OK = 0,
    QMM_ERR_NULL = 1,        /* a required pointer is NULL                     */
    QMM_ERR_SHAPE = 2,       /* K % 32 != 0, a size < 1, or M outside its range */
    QMM_ERR_ALIGN = 3,       /* a pointer lacks the alignment the call needs    */
    QMM_ERR_UNSUPPORTED = 4, /* valid arguments this build does not handle     */
    QMM_ERR_CUDA = 5,        /* a CUDA runtime call or launch failed           */
    QMM_ERR_TIMEOUT = 6,     /* a device-side wait hit its limit               */
    QMM_ERR_SCRATCH = 7      /* the problem exceeds an entry point's fixed
                                scratch (qmm_gemm_q4_0_prefill only)          */
} qmm_status;

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *qmm_stream_t;

/* Largest M accepted by the GEMV entry points. */
#define QMM_GEMV_MAX_M 16

/* ---- Dequantization (bit-exact) ---------------------------------------
 * w   : N*K/32 blocks (18 or 34 bytes each), any byte alignment.
 * out : fp32 [N][K], 4-byte aligned.  out[n][k] = (float)(nibble-8) * d for
 *       Q4_0, (float)q * d for Q8_0, the exact IEEE binary32 product (the
 *       sign of zero and inf/NaN follow IEEE multiplication).
 * Requires n >= 1, k >= 32, k % 32 == 0. */
qmm_status qmm_dequant_q4_0(const void *w, float *out, int64_t n, int64_t k,
                            qmm_stream_t stream);
qmm_status qmm_dequant_q8_0(const void *w, float *out, int64_t n, int64_t k,
                            qmm_stream_t stream);

/* ---- Decode GEMV ------------------------------------------------------
 * y[i][j] = sum_k x[i][k] * w[j][k] for i < m, j < n, computed in fp32
 * (one fp32 product per weight and row, fp32 sums; no tensor cores).
 * w : N*K/32 blocks.   x : fp32 [m][k].   y : fp32 [m][n].
 * Requires 1 <= m <= QMM_GEMV_MAX_M, n >= 1, k >= 32, k % 32 == 0, x and y
 * 4-byte aligned, y not overlapping w or x.  The streaming kernel is used
 * when k % 256 == 0 and w and x are 16-byte aligned; other valid arguments
 * take a slower byte-wise kernel.  Accuracy: |y - y_exact| <=
 * 1e-4 * sum_k |w*x| + 1e-6 per output. */
qmm_status qmm_gemv_q4_0(const void *w, const float *x, float *y, int m, int64_t n,
                         int64_t k, qmm_stream_t stream);
qmm_status qmm_gemv_q8_0(const void *w, const float *x, float *y, int m, int64_t n,
                         int64_t k, qmm_stream_t stream);

/* ---- Grouped decode GEMV -----------------------------------------------
 * Several weight matrices applied to the same activations in one launch:
 * the q/k/v (or gate/up) projections of a layer read one hidden state, and
 * the packed QKV / fused FFN paths of "Add generated quant-kernel JIT and
 * accelerate Gemma4, BGE-M3, and GLiNER2" (second revision, "Summary") batch
 * such projections.  Output i is y_i[r][j] = sum_k x[r][k] * w_i[j][k] for
 * r < m, j < n_i; each output is computed exactly as by qmm_gemv_q4_0 /
 * qmm_gemv_q8_0 on its own (same arithmetic, same accuracy bound).
 * outs : host array of `count` (1..QMM_GEMV_MAX_OUTPUTS) descriptors read
 *        during the call; each w and y is a device pointer as above.
 * Requires what the single call requires for every output, and no output
 * may overlap x, any weight buffer or another output. */
#define QMM_GEMV_MAX_OUTPUTS 4
typedef struct qmm_gemv_out {
    const void *w; /* N_i*K/32 blocks */
    float *y;      /* fp32 [m][n] */
    int64_t n;     /* rows of w_i */
} qmm_gemv_out;

qmm_status qmm_gemv_q4_0_multi(const qmm_gemv_out *outs, int count, const float *x, int m,
                               int64_t k, qmm_stream_t stream);
qmm_status qmm_gemv_q8_0_multi(const qmm_gemv_out *outs, int count, const float *x, int m,
                               int64_t k, qmm_stream_t stream);

/* ---- Fused GeGLU decode (feed-forward input) ---------------------------
 * h[r][j] = gelu(g[r][j]) * u[r][j] with g[r][j] = sum_k x[r][k] * wg[j][k]
 * and u[r][j] = sum_k x[r][k] * wu[j][k], for r < m, j < n: the gate and up
 * projections of a feed-forward block and their gated product in one
 * launch, the fused FFN path of "Add generated quant-kernel JIT and
 * accelerate Gemma4, BGE-M3, and GLiNER2" (second revision, "Summary").
 * The pages do not name the activation; this call takes the GELU in its
 * tanh form, gelu(z) = z/2 * (1 + tanh(sqrt(2/pi) * (z + 0.044715 z^3))),
 * applied to the gate product (the GeGLU of Gemma-family feed-forward
 * blocks).  g and u are computed as by qmm_gemv_q4_0 and never stored.
 * wg, wu : N*K/32 Q4_0 blocks each.   x : fp32 [m][k].   h : fp32 [m][n].
 * Requires what qmm_gemv_q4_0 requires of each weight matrix, and h not
 * overlapping wg, wu or x.  Accuracy, with e_g = 1e-4 * sum_k |wg*x| + 1e-6
 * and e_u likewise: |h - h_exact| <= 1.13 * |u| * e_g + |gelu(g)| * e_u
 * + 1e-5 * (1 + g^2) * |h| + 1e-6 (1.13 bounds |gelu'|; the third term is
 * the fp32 evaluation of the GELU). */
qmm_status qmm_gemv_q4_0_geglu(const void *wg, const void *wu, const float *x, float *h, int m,
                               int64_t n, int64_t k, qmm_stream_t stream);

/* ---- Batched decode GEMV on the tensor cores ----------------------------
 * The product of qmm_gemv_q4_0 (same layouts, same accuracy bound
 * |y - y_exact| <= 1e-4 * sum_k |w*x| + 1e-6), computed on the tcgen05
 * tensor cores, for the small batches of tokens that decode batching and
 * MTP verification produce ("Add generated quant-kernel JIT and accelerate
 * Gemma4, BGE-M3, and GLiNER2", first revision, "Summary" and "Benchmarks":
 * Gemma4 QAT batching, E4B MTP k=1).  Arithmetic: per 32-weight block the
 * exact integers (nibble - 8) (bf16) multiply x split into two bf16 parts,
 * x_hi = bf16(x) and x_lo = bf16(x - x_hi) (|x - x_hi - x_lo| <= 2^-16 |x|),
 * summed in fp32 in tensor memory; each block's sum is then scaled by its d
 * and accumulated in fp32.  qmm_gemv_q4_0 remains the fp32 CUDA-core call.
 * Requires 1 <= m <= QMM_GEMV_MAX_M, n >= 1, k % 256 == 0, k >= 256, w and x
 * 16-byte aligned, y 4-byte aligned and not overlapping w or x.  Valid
 * shapes it does not take return QMM_ERR_UNSUPPORTED: k % 256 != 0, n > 2^30,
 * and shapes whose share of the activations per CTA does not fit shared
 * memory with the K range split at most 8 ways (a power of two dividing
 * k / 256).  Every k up to 5632 (m <= 8) or 2560 (m > 8) is taken; larger k
 * needs such a split, up to k = 36864 (m <= 8) or 14336 (m > 8). */
qmm_status qmm_gemv_q4_0_tc(const void *w, const float *x, float *y, int m, int64_t n,
                            int64_t k, qmm_stream_t stream);

/* ---- Prefill GEMM (tcgen05 tensor cores) ------------------------------
 * Y[i][j] = sum_k X[i][k] * w[j][k] for i < m, j < n.  X is bf16 [m][k]
 * given as raw bf16 bit patterns; each weight is rounded once to bf16
 * ((nibble-8)*d, round to nearest even) and products are summed in fp32
 * in tensor memory.  Y : fp32 [m][n].
 * Requires m >= 1, n >= 1, k % 256 == 0, k >= 256, w and x 16-byte aligned,
 * y 4-byte aligned, y not overlapping w or x, and m <= 2^30, n <= 2^30,
 * k <= 2^24.  Valid shapes outside these (k % 256 != 0, the size limits, an
 * overlapping y) return QMM_ERR_UNSUPPORTED.  Accuracy: |Y - Y_exact| <=
 * 2e-3 * sum_k |w*x| + 1e-6 per output. */
qmm_status qmm_gemm_q4_0(const void *w, const uint16_t *x_bf16, float *y, int64_t m,
                         int64_t n, int64_t k, qmm_stream_t stream);

/* The same product for Q8_0 weights (each w = q*d, exact in fp32, rounded
 * once to bf16), with the same requirements, layout and accuracy bound.
 * Q8_0 at prefill: the weight format of the LM head ("Validation" of the
 * quant-kernel JIT page) when every prompt position's logits are wanted. */
qmm_status qmm_gemm_q8_0(const void *w, const uint16_t *x_bf16, float *y, int64_t m,
                         int64_t n, int64_t k, qmm_stream_t stream);

/* ---- Prefill GEMM with a workspace (long prompts) -----------------------
 * The same products as qmm_gemm_q4_0 / qmm_gemm_q8_0 / qmm_gemm_q4_0_geglu,
 * with the same arithmetic (each weight rounded once to bf16, fp32 sums in
 * tensor memory) and accuracy bound.  With a workspace, a call takes one
 * of two forms, chosen from (m, n, k) and the GPU's SM count:
 *   two phases: the weights are first dequantised once into the workspace
 *     as bf16 (so that they are not decoded again for every 256-token
 *     block) and a second kernel runs the tensor-core GEMM from it;
 *   one phase: the fused call; when its 256 x 256 tiles are too few to
 *     occupy the GPU's SM pairs, it splits K into 2, 4 or 8 parts whose
 *     fp32 partial products go to the workspace, and a second kernel adds
 *     them in part order.  Split results differ from qmm_gemm_q4_0's by
 *     rounding only (same bound) and are the same for every workspace of a
 *     call's shape.
 * Two phases are taken from the third 256-token block on (m > 512), except
 * that three or four blocks (m <= 1024) stay in one phase when the fused
 * call splits K there.  For the GeGLU form (no K split): two phases when
 * m > 512, or m > 256 with k >= 4096.
 * workspace : caller-owned device memory, 16-byte aligned, at least
 *             qmm_gemm_workspace_bytes(n, k) bytes (qmm_gemm_geglu_
 *             workspace_bytes for the GeGLU form), not overlapping any
 *             argument; NULL selects the fused call.  Its contents are
 *             scratch: overwritten by the call, meaningless after it.  Calls
 *             that may run concurrently need separate workspaces.
 * Returns QMM_ERR_SHAPE if workspace_bytes is too small, QMM_ERR_ALIGN if
 * the workspace is misaligned; other checks as for the calls without it. */
size_t qmm_gemm_workspace_bytes(int64_t n, int64_t k);
size_t qmm_gemm_geglu_workspace_bytes(int64_t n, int64_t k);
qmm_status qmm_gemm_q4_0_ws(const void *w, const uint16_t *x_bf16, float *y, int64_t m,
                            int64_t n, int64_t k, void *workspace, size_t workspace_bytes,
                            qmm_stream_t stream);
qmm_status qmm_gemm_q8_0_ws(const void *w, const uint16_t *x_bf16, float *y, int64_t m,
                            int64_t n, int64_t k, void *workspace, size_t workspace_bytes,
                            qmm_stream_t stream);

/* The Q4_0 product of qmm_gemm_q4_0_ws for callers that cannot allocate
 * device memory.  The pages have no counterpart of this entry point: it
 * exists for hosts whose device memory is all owned by their own allocator
 * (a serving engine's arena or a framework's caching allocator with a fixed
 * budget), which forbid a library from calling cudaMalloc, and for plugin
 * interfaces that hand an operator only its inputs and outputs, with no
 * workspace slot and no allocator to ask.
 *
 * Instead of a caller workspace it uses a 64 MiB scratch array that is part
 * of the library (a module-scope __device__ array: every GPU that loads the
 * library holds it until the process exits).  Where qmm_gemm_q4_0_ws runs
 * in two phases, the weights are dequantised into it in column chunks of
 * whole 256-row tiles, each chunk followed by its GEMM; elsewhere it runs
 * the fused kernel with the K split of qmm_gemm_q4_0_ws through the
 * scratch.  The call makes no cudaMalloc, cudaFree or other
 * allocating call.  Same arithmetic, result and accuracy as
 * qmm_gemm_q4_0_ws (bit-identical to it; to qmm_gemm_q4_0 too except where
 * short prompts split K), and the same requirements, plus:
 *   k <= 131072: one 256-row chunk (256 * k bf16 values) must fit the
 *     scratch; a larger k returns QMM_ERR_SCRATCH and launches nothing.
 * Set-up: the first call on a device (with that device current) resolves
 * the scratch's device address once; make that first call before any
 * stream capture begins on the device.
 * Sharing: every call of this entry point on a device uses the same
 * scratch, which keeps the last call's contents (nothing in it needs to
 * start at zero: each chunk's rows are written before they are read).
 * Calls that overlap on the GPU -- on different streams, or from different
 * threads without ordering -- race on the scratch and give wrong results;
 * the caller orders them (one stream, or events).  Calls on one stream are
 * ordered by the stream. */
qmm_status qmm_gemm_q4_0_prefill(const void *w, const uint16_t *x_bf16, float *y, int64_t m,
                                 int64_t n, int64_t k, qmm_stream_t stream);

/* ---- Prefill GeGLU (tcgen05 tensor cores) -----------------------------
 * h[i][j] = bf16(gelu(g[i][j]) * u[i][j]) with g[i][j] = sum_k X[i][k] *
 * wg[j][k] and u[i][j] = sum_k X[i][k] * wu[j][k], for i < m, j < n: the
 * prefill side of the fused FFN path (same page and section as
 * qmm_gemv_q4_0_geglu, same GELU), written as bf16 because it is the
 * activation operand of the down-projection GEMM.  g and u are formed as by
 * qmm_gemm_q4_0 (weights rounded once to bf16, fp32 sums in tensor memory)
 * and never stored; h is rounded once to bf16 (nearest even).
 * wg, wu : N*K/32 Q4_0 blocks each, 16-byte aligned.  x : bf16 [m][k],
 * 16-byte aligned.  h : bf16 [m][n], 2-byte aligned, not overlapping wg, wu
 * or x.  Requires m >= 1, n >= 1, k % 256 == 0 (else QMM_ERR_UNSUPPORTED).
 * Accuracy, with e_g = 2e-3 * sum_k |wg*x| + 1e-6 and e_u likewise:
 * |h - h_exact| <= 1.13 * |u| * e_g + |gelu(g)| * e_u
 * + (2^-8 + 1e-5 * (1 + g^2)) * |h| + 1e-6. */
qmm_status qmm_gemm_q4_0_geglu(const void *wg, const void *wu, const uint16_t *x_bf16,
                               uint16_t *h_bf16, int64_t m, int64_t n, int64_t k,
                               qmm_stream_t stream);
qmm_status qmm_gemm_q4_0_geglu_ws(const void *wg, const void *wu, const uint16_t *x_bf16,
                                  uint16_t *h_bf16, int64_t m, int64_t n, int64_t k,
                                  void *workspace, size_t workspace_bytes, qmm_stream_t stream);

/* ---- Stream-ordered copies by the SMs ----------------------------------
 * Copies `bytes` bytes from src to dst in stream order, as one kernel launch
 * that loads and stores through the device's address space.  The pages have
 * no counterpart of this entry point: it exists for the end-to-end decode
 * step, whose activations go in and whose outputs come out every step (a
 * few tens of kilobytes).  There a copy-engine transfer (cudaMemcpyAsync)
 * costs several microseconds whatever its size, while this launch overlaps
 * its start with its neighbours like the GEMV launches do.
 * src, dst : device memory of the current device, or page-locked host memory
 *            mapped into the device's address space at its host address
 *            (cudaHostAlloc / cudaMallocHost memory under unified
 *            addressing, which is how PyTorch's pin_memory allocates); each
 *            holds `bytes` bytes; any alignment (16-byte aligned pointers
 *            move 16 bytes per access).  Checked with cudaPointerGetAttributes
 *            before anything is launched: other memory (pageable host memory,
 *            another device's memory) returns QMM_ERR_UNSUPPORTED.
 * Overlapping ranges return QMM_ERR_UNSUPPORTED; bytes == 0 launches
 * nothing and returns QMM_OK.  The copy is complete, and host memory
 * written by it visible to the host, once the stream has been synchronised.
 * It waits for the previous launch on the stream before reading src or
 * writing dst, so it may read that launch's output or overwrite its input. */
qmm_status qmm_copy(void *dst, const void *src, size_t bytes, qmm_stream_t stream);

/* ---- Utilities --------------------------------------------------------- */

/* Static English text for a status code (never NULL). */
const char *qmm_status_string(qmm_status status);

/* Library version: major*10000 + minor*100 + patch. */
int qmm_version(void);

/* Synchronises `stream`, then returns and clears the current device's error
 * word: QMM_OK, QMM_ERR_TIMEOUT if a kernel gave up a bounded wait since the
 * last call, or QMM_ERR_CUDA if the synchronisation itself failed. */
qmm_status qmm_get_device_error(qmm_stream_t stream);

/* Time limit, in nanoseconds of the GPU global timer, of every device-side
 * wait (default 2e9 = 2 s; 0 restores the default).  Applies to launches
 * made after the call, from any thread. */
void qmm_set_wait_timeout_ns(uint64_t ns);

/* Launches one kernel that waits on a barrier nothing ever completes, for at
 * most `timeout_ns`, so that the timeout path can be exercised without a
 * fault: the kernel records QMM_ERR_TIMEOUT in the error word and returns.
 * Returns QMM_ERR_CUDA if the launch fails. */
qmm_status qmm_selftest_wait_timeout(uint64_t timeout_ns, qmm_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif
