// qmm_internal.h -- host-side declarations shared by the library's
// translation units (not part of the public ABI; see include/qmm.h).
#pragma once

#include <cstdint>
#include <utility>

#include <cuda_runtime.h>

#include <cuda.h>

#include "qmm_device.cuh"

namespace qmm {

enum class Fmt : int { Q4_0 = 0, Q8_0 = 1 };

constexpr int kQK = 32;            // weights per block
constexpr int kQ4_0Bytes = 18;     // binary16 d + 16 nibble bytes
constexpr int kQ8_0Bytes = 34;     // binary16 d + 32 int8

inline int block_bytes(Fmt f) { return f == Fmt::Q4_0 ? kQ4_0Bytes : kQ8_0Bytes; }

// Launch with programmatic dependent launch allowed (the kernel itself
// waits for its predecessor before touching global memory) and an optional
// cluster width along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, unsigned cluster_x, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attrs[2];
    unsigned na = 0;
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (cluster_x > 1) {
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = cluster_x;
        attrs[na].val.clusterDim.y = 1;
        attrs[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Number of SMs of the current device (cached per device).
int device_sm_count();

// Current device ordinal (0 if the query fails).
int current_device();

// Raise a kernel's dynamic shared-memory limit to at least `bytes` on the
// current device.  `limits` is the caller's per-kernel cache (one slot per
// device, a static array local to the launcher of that one kernel), so the
// attribute call is made only when that kernel's limit grows and launches
// inside stream capture make no attribute calls once warmed up.
constexpr int kMaxDevices = 64;

template <typename Kernel>
cudaError_t ensure_smem(Kernel kernel, size_t bytes, bool cluster, int (&limits)[kMaxDevices]) {
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (static_cast<int>(bytes) <= __atomic_load_n(&limits[dev], __ATOMIC_ACQUIRE))
        return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(bytes));
    if (e == cudaSuccess && cluster)
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e == cudaSuccess) __atomic_store_n(&limits[dev], static_cast<int>(bytes), __ATOMIC_RELEASE);
    return e;
}

// Encode a 2-D tiled TMA descriptor (no swizzle unless given): dims
// {inner, outer} elements, outer stride in bytes, box {box_inner, box_outer}.
// Returns false if the driver entry point is missing or rejects the shape.
bool encode_tmap_2d(CUtensorMap *map, CUtensorMapDataType dtype, const void *base,
                    uint64_t inner, uint64_t outer, uint64_t outer_stride_bytes,
                    uint32_t box_inner, uint32_t box_outer,
                    CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_NONE);

cudaError_t launch_dequant(Fmt fmt, const uint8_t *w, float *out, int64_t n, int64_t k,
                           cudaStream_t stream, const LaunchCtx &ctx);

// Stream-ordered copy of `bytes` bytes by the SMs; both pointers device
// accessible (device memory, or page-locked host memory mapped at its host
// address), the ranges disjoint.
cudaError_t launch_copy(void *dst, const void *src, size_t bytes, cudaStream_t stream);

// One weight matrix of a GEMV call: w (n rows of blocks) applied to the
// call's shared activations, written to y [m][n].
struct GemvProblem {
    const void *w;
    float *y;
    int64_t n;
};

// GEMV over `count` (1..4) problems that share x [m][k]; one launch when the
// streaming kernel applies.  Implemented per format and range of m.
cudaError_t launch_gemv_q4_0_m1_2(const GemvProblem *probs, int count, const float *x, int m,
                                  int64_t k, cudaStream_t stream, const LaunchCtx &ctx);
cudaError_t launch_gemv_q4_0_m3_4(const GemvProblem *probs, int count, const float *x, int m,
                                  int64_t k, cudaStream_t stream, const LaunchCtx &ctx);
cudaError_t launch_gemv_q4_0_m5_10(const GemvProblem *probs, int count, const float *x, int m,
                                  int64_t k, cudaStream_t stream, const LaunchCtx &ctx);
cudaError_t launch_gemv_q4_0_m11_16(const GemvProblem *probs, int count, const float *x, int m,
                                  int64_t k, cudaStream_t stream, const LaunchCtx &ctx);
cudaError_t launch_gemv_q8_0_m1_2(const GemvProblem *probs, int count, const float *x, int m,
                                  int64_t k, cudaStream_t stream, const LaunchCtx &ctx);
cudaError_t launch_gemv_q8_0_m3_4(const GemvProblem *probs, int count, const float *x, int m,
                                  int64_t k, cudaStream_t stream, const LaunchCtx &ctx);
cudaError_t launch_gemv_q8_0_m5_10(const GemvProblem *probs, int count, const float *x, int m,
                                  int64_t k, cudaStream_t stream, const LaunchCtx &ctx);
cudaError_t launch_gemv_q8_0_m11_16(const GemvProblem *probs, int count, const float *x, int m,
                                  int64_t k, cudaStream_t stream, const LaunchCtx &ctx);

inline cudaError_t launch_gemv(Fmt fmt, const GemvProblem *probs, int count, const float *x,
                               int m, int64_t k, cudaStream_t stream, const LaunchCtx &ctx) {
    if (fmt == Fmt::Q4_0) {
        if (m <= 2) return launch_gemv_q4_0_m1_2(probs, count, x, m, k, stream, ctx);
        if (m <= 4) return launch_gemv_q4_0_m3_4(probs, count, x, m, k, stream, ctx);
        if (m <= 10) return launch_gemv_q4_0_m5_10(probs, count, x, m, k, stream, ctx);
        return launch_gemv_q4_0_m11_16(probs, count, x, m, k, stream, ctx);
    }
    if (m <= 2) return launch_gemv_q8_0_m1_2(probs, count, x, m, k, stream, ctx);
    if (m <= 4) return launch_gemv_q8_0_m3_4(probs, count, x, m, k, stream, ctx);
    if (m <= 10) return launch_gemv_q8_0_m5_10(probs, count, x, m, k, stream, ctx);
    return launch_gemv_q8_0_m11_16(probs, count, x, m, k, stream, ctx);
}

// Fused GeGLU decode: h[m][i] = gelu(x[m] . wg[i]) * (x[m] . wu[i]) with
// gate_up[0] = {wg, h, n} and gate_up[1] = {wu, unused, n}.
cudaError_t launch_geglu_q4_0_m1_4(const GemvProblem *gate_up, const float *x, int m, int64_t k,
                                   cudaStream_t stream, const LaunchCtx &ctx);
cudaError_t launch_geglu_q4_0_m5_10(const GemvProblem *gate_up, const float *x, int m, int64_t k,
                                    cudaStream_t stream, const LaunchCtx &ctx);
cudaError_t launch_geglu_q4_0_m11_16(const GemvProblem *gate_up, const float *x, int m,
                                     int64_t k, cudaStream_t stream, const LaunchCtx &ctx);

inline cudaError_t launch_geglu_q4_0(const GemvProblem *gate_up, const float *x, int m,
                                     int64_t k, cudaStream_t stream, const LaunchCtx &ctx) {
    if (m <= 4) return launch_geglu_q4_0_m1_4(gate_up, x, m, k, stream, ctx);
    if (m <= 10) return launch_geglu_q4_0_m5_10(gate_up, x, m, k, stream, ctx);
    return launch_geglu_q4_0_m11_16(gate_up, x, m, k, stream, ctx);
}

// Fused prefill GEMM.  part / part_bytes (optional, 16-byte aligned, not
// overlapping any operand): room for K-split partial products, used when the
// product has too few tiles to fill the SMs (short prompts); the call then
// adds the parts into y with a second kernel, in a fixed order.
cudaError_t launch_gemm_q4_0(const uint8_t *w, const uint16_t *x, float *y, int64_t m,
                             int64_t n, int64_t k, cudaStream_t stream, const LaunchCtx &ctx,
                             float *part = nullptr, size_t part_bytes = 0);

cudaError_t launch_gemm_q8_0(const uint8_t *w, const uint16_t *x, float *y, int64_t m,
                             int64_t n, int64_t k, cudaStream_t stream, const LaunchCtx &ctx,
                             float *part = nullptr, size_t part_bytes = 0);

// Prefill GeGLU: h[i][j] = bf16(gelu(X[i] . wg[j]) * (X[i] . wu[j])).
cudaError_t launch_gemm_q4_0_geglu(const uint8_t *wg, const uint8_t *wu, const uint16_t *x,
                                   uint16_t *h, int64_t m, int64_t n, int64_t k,
                                   cudaStream_t stream, const LaunchCtx &ctx);

// The K split the fused plain GEMM takes for an (m, n, k) product given
// part_bytes of room for partial products (1: none).
int gemm_fused_ksplit(int64_t m, int64_t n, int64_t k, size_t part_bytes);

// Room for K-split partial products that the one-phase product takes, out of
// a caller workspace of gemm_workspace_bytes(n, k, false) or out of the
// prefill entry's 64 MiB scratch: the same for both, so that both choose the
// same split and give the same bits.
size_t fused_part_budget(int64_t n, int64_t k);

// When the two-phase plain GEMM pays, from measurements of both forms at
// N x K = 2048 x 8192, 8192 x 2048, 16384 x 2048, 4096 x 4096 and
// 8192 x 8192 for m = 256..2048.  The dequant pass costs about 0.65 us per
// million weights; the fused kernel decodes the weights again for every
// 256-token block, and a product whose pair tiles leave pairs idle runs the
// fused kernel with a K split instead.  So: never for one or two token
// blocks; not for three or four blocks when the fused kernel splits K (the
// two-phase GEMM has as few tiles, each running all of K); otherwise always.
bool use_two_phase_gemm(int64_t m, int64_t n, int64_t k);

// The GeGLU form has no K split: two phases from the third token block, or
// from the second at K >= 4096 (where the unsplit fused kernel's few tiles
// run all of a long K).
inline bool use_two_phase_geglu(int64_t m, int64_t k) { return m > 512 || (m > 256 && k >= 4096); }

// Two-phase prefill GEMM (weights dequantised once into a bf16 workspace,
// then a shared-memory-operand tensor-core GEMM).  gemm_workspace_bytes is
// the workspace it needs.
size_t gemm_workspace_bytes(int64_t n, int64_t k, bool geglu);
cudaError_t launch_gemm_two_phase(Fmt fmt, const uint8_t *w, const uint16_t *x, float *y,
                                  int64_t m, int64_t n, int64_t k, uint16_t *ws,
                                  cudaStream_t stream, const LaunchCtx &ctx);
cudaError_t launch_gemm_geglu_two_phase(const uint8_t *wg, const uint8_t *wu, const uint16_t *x,
                                        uint16_t *h, int64_t m, int64_t n, int64_t k, uint16_t *ws,
                                        cudaStream_t stream, const LaunchCtx &ctx);

// Largest K of qmm_gemm_q4_0_prefill: one 256-row chunk of bf16 weights
// (256 * K * 2 bytes) must fit its 64 MiB static scratch.
constexpr int64_t kPrefillMaxK = 131072;

// Largest sizes the tensor-core GEMM launchers take (tile indices and tensor
// map extents stay in 32-bit range); the API returns QMM_ERR_UNSUPPORTED
// beyond them before launching anything.
constexpr int64_t kGemmMaxM = int64_t(1) << 30;
constexpr int64_t kGemmMaxN = int64_t(1) << 30;
constexpr int64_t kGemmMaxK = int64_t(1) << 24;

// Two-phase Q4_0 prefill GEMM on the library's own static scratch (column
// chunks that fit it; the fused kernel below the two-phase length rule).
// Every host step that can fail for the call's chunk shapes runs before the
// first launch.
cudaError_t launch_gemm_q4_0_prefill(const uint8_t *w, const uint16_t *x, float *y, int64_t m,
                                     int64_t n, int64_t k, cudaStream_t stream,
                                     const LaunchCtx &ctx);

// Batched decode GEMV on the tensor cores (Q4_0, 1 <= m <= 16, k % 256 == 0,
// w and x 16-byte aligned).  gemv_tc_shape_ok: the launcher has a launch
// shape for (m, n, k) (the CTA's activation slice fits shared memory).
bool gemv_tc_shape_ok(int m, int64_t n, int64_t k);
cudaError_t launch_gemv_tc_q4_0(const uint8_t *w, const float *x, float *y, int m, int64_t n,
                                int64_t k, cudaStream_t stream, const LaunchCtx &ctx);

cudaError_t launch_selftest_wait(cudaStream_t stream, const LaunchCtx &ctx);

}  // namespace qmm
