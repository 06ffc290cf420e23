// qmm_api.cu -- the C ABI (include/qmm.h): argument checks, per-device state
// (error word, SM count), launches.  No entry point allocates device memory.
#include "../../include/qmm.h"
#include "qmm_internal.h"

#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

namespace qmm {

// Device error word: written by kernels that give up a bounded wait, read
// and cleared by qmm_get_device_error().  One per GPU (module-scope device
// variable; no allocation).
__device__ uint32_t g_device_error = 0;

namespace {

constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;

std::atomic<uint64_t> g_timeout_ns{kDefaultTimeoutNs};

struct DeviceState {
    std::once_flag once;
    cudaError_t init_err = cudaSuccess;
    uint32_t *err_word = nullptr;
    int sms = 0;
};
DeviceState g_dev[kMaxDevices];

// Per-device set-up, once, with that device current.
DeviceState *device_state(cudaError_t *err) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *err = e != cudaSuccess ? e : cudaErrorInvalidDevice;
        return nullptr;
    }
    DeviceState &st = g_dev[dev];
    std::call_once(st.once, [&st, dev]() {
        void *p = nullptr;
        st.init_err = cudaGetSymbolAddress(&p, g_device_error);
        if (st.init_err == cudaSuccess) {
            st.err_word = static_cast<uint32_t *>(p);
            st.init_err = cudaDeviceGetAttribute(&st.sms, cudaDevAttrMultiProcessorCount, dev);
        }
    });
    *err = st.init_err;
    return st.init_err == cudaSuccess ? &st : nullptr;
}

bool make_ctx(LaunchCtx *ctx) {
    cudaError_t e;
    DeviceState *st = device_state(&e);
    if (!st) return false;
    ctx->err = st->err_word;
    ctx->timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);
    return true;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

qmm_status from_cuda(cudaError_t e) { return e == cudaSuccess ? QMM_OK : QMM_ERR_CUDA; }

qmm_status check_wk(const void *w, int64_t n, int64_t k) {
    if (!w) return QMM_ERR_NULL;
    if (n < 1 || k < kQK || k % kQK != 0) return QMM_ERR_SHAPE;
    // byte offsets of the largest index must fit comfortably in 64 bits
    if (n > (int64_t(1) << 40) || k > (int64_t(1) << 31)) return QMM_ERR_SHAPE;
    return QMM_OK;
}

// [a, a+an) and [b, b+bn) overlap
bool overlaps(const void *a, size_t an, const void *b, size_t bn) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + bn && y < x + an;
}

qmm_status dequant(Fmt fmt, const void *w, float *out, int64_t n, int64_t k,
                   qmm_stream_t stream) {
    qmm_status s = check_wk(w, n, k);
    if (s != QMM_OK) return s;
    if (!out) return QMM_ERR_NULL;
    if (!aligned(out, 4)) return QMM_ERR_ALIGN;
    LaunchCtx ctx;
    if (!make_ctx(&ctx)) return QMM_ERR_CUDA;
    return from_cuda(launch_dequant(fmt, static_cast<const uint8_t *>(w), out, n, k,
                                    reinterpret_cast<cudaStream_t>(stream), ctx));
}

qmm_status gemv(Fmt fmt, const qmm_gemv_out *outs, int count, const float *x, int m, int64_t k,
                qmm_stream_t stream) {
    if (!outs || !x) return QMM_ERR_NULL;
    if (count < 1 || count > QMM_GEMV_MAX_OUTPUTS) return QMM_ERR_SHAPE;
    if (m < 1 || m > QMM_GEMV_MAX_M) return QMM_ERR_SHAPE;
    if (!aligned(x, 4)) return QMM_ERR_ALIGN;
    GemvProblem probs[QMM_GEMV_MAX_OUTPUTS];
    for (int i = 0; i < count; ++i) {
        const qmm_status s = check_wk(outs[i].w, outs[i].n, k);
        if (s != QMM_OK) return s;
        if (!outs[i].y) return QMM_ERR_NULL;
        if (!aligned(outs[i].y, 4)) return QMM_ERR_ALIGN;
        probs[i] = GemvProblem{outs[i].w, outs[i].y, outs[i].n};
    }
    // no output may overlap an input or another output
    const size_t xbytes = sizeof(float) * static_cast<size_t>(m) * k;
    for (int i = 0; i < count; ++i) {
        const size_t ybytes = sizeof(float) * static_cast<size_t>(m) * outs[i].n;
        if (overlaps(outs[i].y, ybytes, x, xbytes)) return QMM_ERR_UNSUPPORTED;
        for (int j = 0; j < count; ++j) {
            const size_t wbytes = static_cast<size_t>(outs[j].n) * (k / kQK) * block_bytes(fmt);
            if (overlaps(outs[i].y, ybytes, outs[j].w, wbytes)) return QMM_ERR_UNSUPPORTED;
            if (j != i && overlaps(outs[i].y, ybytes, outs[j].y,
                                   sizeof(float) * static_cast<size_t>(m) * outs[j].n))
                return QMM_ERR_UNSUPPORTED;
        }
    }
    LaunchCtx ctx;
    if (!make_ctx(&ctx)) return QMM_ERR_CUDA;
    return from_cuda(launch_gemv(fmt, probs, count, x, m, k,
                                 reinterpret_cast<cudaStream_t>(stream), ctx));
}

// Memory a kernel on the current device may read and write at address p:
// that device's memory, managed memory, or page-locked host memory mapped
// at its host address.  Pageable host memory is refused (a kernel access
// to it would fault).
bool device_accessible(const void *p) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        (void)cudaGetLastError();  // the failed query is not a launch error: clear it
        return false;
    }
    switch (a.type) {
    case cudaMemoryTypeDevice:
        return a.device == dev;
    case cudaMemoryTypeManaged:
        return true;
    case cudaMemoryTypeHost:
        return a.devicePointer == p;
    default:
        return false;
    }
}

qmm_status check_workspace(const void *ws, size_t ws_bytes, size_t need) {
    if (!aligned(ws, 16)) return QMM_ERR_ALIGN;
    if (ws_bytes < need) return QMM_ERR_SHAPE;
    return QMM_OK;
}

// Checks shared by the tensor-core GEMM entry points (plain product): y is
// fp32 [m][n], written with 4-byte stores; y may overlap neither input.
qmm_status check_gemm(Fmt fmt, const void *w, const uint16_t *x_bf16, const float *y, int64_t m,
                      int64_t n, int64_t k) {
    qmm_status s = check_wk(w, n, k);
    if (s != QMM_OK) return s;
    if (!x_bf16 || !y) return QMM_ERR_NULL;
    if (m < 1) return QMM_ERR_SHAPE;
    if (k % 256 != 0 || m > kGemmMaxM || n > kGemmMaxN || k > kGemmMaxK)
        return QMM_ERR_UNSUPPORTED;
    if (!aligned(w, 16) || !aligned(x_bf16, 16) || !aligned(y, 4)) return QMM_ERR_ALIGN;
    const size_t ybytes = sizeof(float) * static_cast<size_t>(m) * n;
    const size_t wbytes = static_cast<size_t>(n) * (k / kQK) * block_bytes(fmt);
    if (overlaps(y, ybytes, w, wbytes) || overlaps(y, ybytes, x_bf16, 2 * static_cast<size_t>(m) * k))
        return QMM_ERR_UNSUPPORTED;
    return QMM_OK;
}

qmm_status gemm(Fmt fmt, const void *w, const uint16_t *x_bf16, float *y, int64_t m, int64_t n,
                int64_t k, qmm_stream_t stream, void *ws = nullptr, size_t ws_bytes = 0) {
    qmm_status s = check_gemm(fmt, w, x_bf16, y, m, n, k);
    if (s != QMM_OK) return s;
    const bool two_phase = ws != nullptr && use_two_phase_gemm(m, n, k);
    const size_t wbytes = static_cast<size_t>(n) * (k / kQK) * block_bytes(fmt);
    const size_t ybytes = sizeof(float) * static_cast<size_t>(m) * n;
    if (ws != nullptr) {
        // two phases: the dequantised weights; one phase (short prompts):
        // room for K-split partial products
        const size_t need = gemm_workspace_bytes(n, k, false);
        s = check_workspace(ws, ws_bytes, need);
        if (s != QMM_OK) return s;
        if (overlaps(ws, need, w, wbytes) || overlaps(ws, need, x_bf16, 2 * static_cast<size_t>(m) * k) ||
            overlaps(ws, need, y, ybytes))
            return QMM_ERR_UNSUPPORTED;
    }
    LaunchCtx ctx;
    if (!make_ctx(&ctx)) return QMM_ERR_CUDA;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const uint8_t *wb = static_cast<const uint8_t *>(w);
    if (two_phase)
        return from_cuda(launch_gemm_two_phase(fmt, wb, x_bf16, y, m, n, k,
                                               static_cast<uint16_t *>(ws), st, ctx));
    // K-split budget: fixed by the shape (not by what this caller happens to
    // give), so that every workspace and the prefill entry's scratch choose
    // the same split and give the same bits
    float *part = static_cast<float *>(ws);
    const size_t budget = ws != nullptr ? fused_part_budget(n, k) : 0;
    return from_cuda(fmt == Fmt::Q4_0 ? launch_gemm_q4_0(wb, x_bf16, y, m, n, k, st, ctx, part, budget)
                                      : launch_gemm_q8_0(wb, x_bf16, y, m, n, k, st, ctx, part, budget));
}

}  // namespace

bool encode_tmap_2d(CUtensorMap *map, CUtensorMapDataType dtype, const void *base,
                    uint64_t inner, uint64_t outer, uint64_t outer_stride_bytes,
                    uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle) {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, []() {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {outer_stride_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, dtype, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int current_device() {
    int dev = 0;
    return cudaGetDevice(&dev) == cudaSuccess ? dev : 0;
}

int device_sm_count() {
    cudaError_t e;
    DeviceState *st = device_state(&e);
    return st ? st->sms : 1;
}

// ---- self-test: a wait that nothing completes ---------------------------------
__global__ void selftest_wait_kernel(LaunchCtx ctx) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) mbar_init(&bar, 1);
    fence_mbar_init();
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait(&bar, 0, ctx);  // never completes: bounded by ctx.timeout_ns
    __syncthreads();
}

cudaError_t launch_selftest_wait(cudaStream_t stream, const LaunchCtx &ctx) {
    return launch_kernel(selftest_wait_kernel, dim3(1), dim3(32), 0, stream, 1, ctx);
}

}  // namespace qmm

using namespace qmm;

extern "C" {

qmm_status qmm_dequant_q4_0(const void *w, float *out, int64_t n, int64_t k,
                            qmm_stream_t stream) {
    return dequant(Fmt::Q4_0, w, out, n, k, stream);
}

qmm_status qmm_dequant_q8_0(const void *w, float *out, int64_t n, int64_t k,
                            qmm_stream_t stream) {
    return dequant(Fmt::Q8_0, w, out, n, k, stream);
}

qmm_status qmm_copy(void *dst, const void *src, size_t bytes, qmm_stream_t stream) {
    if (bytes == 0) return QMM_OK;
    if (!dst || !src) return QMM_ERR_NULL;
    if (overlaps(dst, bytes, src, bytes)) return QMM_ERR_UNSUPPORTED;
    if (!device_accessible(src) || !device_accessible(dst)) return QMM_ERR_UNSUPPORTED;
    cudaError_t e;
    if (!device_state(&e)) return QMM_ERR_CUDA;  // the SM count for the grid
    return from_cuda(launch_copy(dst, src, bytes, reinterpret_cast<cudaStream_t>(stream)));
}

qmm_status qmm_gemv_q4_0(const void *w, const float *x, float *y, int m, int64_t n, int64_t k,
                         qmm_stream_t stream) {
    const qmm_gemv_out one = {w, y, n};
    return gemv(Fmt::Q4_0, &one, 1, x, m, k, stream);
}

qmm_status qmm_gemv_q8_0(const void *w, const float *x, float *y, int m, int64_t n, int64_t k,
                         qmm_stream_t stream) {
    const qmm_gemv_out one = {w, y, n};
    return gemv(Fmt::Q8_0, &one, 1, x, m, k, stream);
}

qmm_status qmm_gemv_q4_0_multi(const qmm_gemv_out *outs, int count, const float *x, int m,
                               int64_t k, qmm_stream_t stream) {
    return gemv(Fmt::Q4_0, outs, count, x, m, k, stream);
}

qmm_status qmm_gemv_q8_0_multi(const qmm_gemv_out *outs, int count, const float *x, int m,
                               int64_t k, qmm_stream_t stream) {
    return gemv(Fmt::Q8_0, outs, count, x, m, k, stream);
}

qmm_status qmm_gemv_q4_0_geglu(const void *wg, const void *wu, const float *x, float *h, int m,
                               int64_t n, int64_t k, qmm_stream_t stream) {
    qmm_status s = check_wk(wg, n, k);
    if (s == QMM_OK) s = check_wk(wu, n, k);
    if (s != QMM_OK) return s;
    if (!x || !h) return QMM_ERR_NULL;
    if (m < 1 || m > QMM_GEMV_MAX_M) return QMM_ERR_SHAPE;
    if (!aligned(x, 4) || !aligned(h, 4)) return QMM_ERR_ALIGN;
    const size_t hbytes = sizeof(float) * static_cast<size_t>(m) * n;
    const size_t wbytes = static_cast<size_t>(n) * (k / kQK) * kQ4_0Bytes;
    if (overlaps(h, hbytes, x, sizeof(float) * static_cast<size_t>(m) * k) ||
        overlaps(h, hbytes, wg, wbytes) || overlaps(h, hbytes, wu, wbytes))
        return QMM_ERR_UNSUPPORTED;
    LaunchCtx ctx;
    if (!make_ctx(&ctx)) return QMM_ERR_CUDA;
    const GemvProblem gate_up[2] = {{wg, h, n}, {wu, nullptr, n}};
    return from_cuda(launch_geglu_q4_0(gate_up, x, m, k, reinterpret_cast<cudaStream_t>(stream), ctx));
}

qmm_status qmm_gemv_q4_0_tc(const void *w, const float *x, float *y, int m, int64_t n, int64_t k,
                            qmm_stream_t stream) {
    qmm_status s = check_wk(w, n, k);
    if (s != QMM_OK) return s;
    if (!x || !y) return QMM_ERR_NULL;
    if (m < 1 || m > QMM_GEMV_MAX_M) return QMM_ERR_SHAPE;
    if (!gemv_tc_shape_ok(m, n, k)) return QMM_ERR_UNSUPPORTED;
    if (!aligned(w, 16) || !aligned(x, 16) || !aligned(y, 4)) return QMM_ERR_ALIGN;
    const size_t ybytes = sizeof(float) * static_cast<size_t>(m) * n;
    const size_t wbytes = static_cast<size_t>(n) * (k / kQK) * kQ4_0Bytes;
    if (overlaps(y, ybytes, w, wbytes) || overlaps(y, ybytes, x, sizeof(float) * static_cast<size_t>(m) * k))
        return QMM_ERR_UNSUPPORTED;
    LaunchCtx ctx;
    if (!make_ctx(&ctx)) return QMM_ERR_CUDA;
    return from_cuda(launch_gemv_tc_q4_0(static_cast<const uint8_t *>(w), x, y, m, n, k,
                                         reinterpret_cast<cudaStream_t>(stream), ctx));
}

qmm_status qmm_gemm_q4_0(const void *w, const uint16_t *x_bf16, float *y, int64_t m, int64_t n,
                         int64_t k, qmm_stream_t stream) {
    return gemm(Fmt::Q4_0, w, x_bf16, y, m, n, k, stream);
}

qmm_status qmm_gemm_q8_0(const void *w, const uint16_t *x_bf16, float *y, int64_t m, int64_t n,
                         int64_t k, qmm_stream_t stream) {
    return gemm(Fmt::Q8_0, w, x_bf16, y, m, n, k, stream);
}

qmm_status qmm_gemm_q4_0_prefill(const void *w, const uint16_t *x_bf16, float *y, int64_t m,
                                 int64_t n, int64_t k, qmm_stream_t stream) {
    qmm_status s = check_gemm(Fmt::Q4_0, w, x_bf16, y, m, n, k);
    if (s != QMM_OK) return s;
    if (k > kPrefillMaxK) return QMM_ERR_SCRATCH;
    LaunchCtx ctx;
    if (!make_ctx(&ctx)) return QMM_ERR_CUDA;
    return from_cuda(launch_gemm_q4_0_prefill(static_cast<const uint8_t *>(w), x_bf16, y, m, n, k,
                                              reinterpret_cast<cudaStream_t>(stream), ctx));
}

size_t qmm_gemm_workspace_bytes(int64_t n, int64_t k) {
    if (n < 1 || k < 1) return 0;
    return gemm_workspace_bytes(n, k, false);
}

size_t qmm_gemm_geglu_workspace_bytes(int64_t n, int64_t k) {
    if (n < 1 || k < 1) return 0;
    return gemm_workspace_bytes(n, k, true);
}

qmm_status qmm_gemm_q4_0_ws(const void *w, const uint16_t *x_bf16, float *y, int64_t m, int64_t n,
                            int64_t k, void *workspace, size_t workspace_bytes,
                            qmm_stream_t stream) {
    return gemm(Fmt::Q4_0, w, x_bf16, y, m, n, k, stream, workspace, workspace_bytes);
}

qmm_status qmm_gemm_q8_0_ws(const void *w, const uint16_t *x_bf16, float *y, int64_t m, int64_t n,
                            int64_t k, void *workspace, size_t workspace_bytes,
                            qmm_stream_t stream) {
    return gemm(Fmt::Q8_0, w, x_bf16, y, m, n, k, stream, workspace, workspace_bytes);
}

qmm_status qmm_gemm_q4_0_geglu(const void *wg, const void *wu, const uint16_t *x_bf16,
                               uint16_t *h_bf16, int64_t m, int64_t n, int64_t k,
                               qmm_stream_t stream) {
    return qmm_gemm_q4_0_geglu_ws(wg, wu, x_bf16, h_bf16, m, n, k, nullptr, 0, stream);
}

qmm_status qmm_gemm_q4_0_geglu_ws(const void *wg, const void *wu, const uint16_t *x_bf16,
                                  uint16_t *h_bf16, int64_t m, int64_t n, int64_t k,
                                  void *workspace, size_t workspace_bytes, qmm_stream_t stream) {
    qmm_status s = check_wk(wg, n, k);
    if (s == QMM_OK) s = check_wk(wu, n, k);
    if (s != QMM_OK) return s;
    if (!x_bf16 || !h_bf16) return QMM_ERR_NULL;
    if (m < 1) return QMM_ERR_SHAPE;
    if (k % 256 != 0 || m > kGemmMaxM || n > kGemmMaxN || k > kGemmMaxK) return QMM_ERR_UNSUPPORTED;
    if (!aligned(wg, 16) || !aligned(wu, 16) || !aligned(x_bf16, 16) || !aligned(h_bf16, 2))
        return QMM_ERR_ALIGN;
    const size_t hbytes = sizeof(uint16_t) * static_cast<size_t>(m) * n;
    const size_t wbytes = static_cast<size_t>(n) * (k / kQK) * kQ4_0Bytes;
    if (overlaps(h_bf16, hbytes, x_bf16, sizeof(uint16_t) * static_cast<size_t>(m) * k) ||
        overlaps(h_bf16, hbytes, wg, wbytes) || overlaps(h_bf16, hbytes, wu, wbytes))
        return QMM_ERR_UNSUPPORTED;
    const bool two_phase = workspace != nullptr && use_two_phase_geglu(m, k);
    if (two_phase) {
        const size_t need = gemm_workspace_bytes(n, k, true);
        s = check_workspace(workspace, workspace_bytes, need);
        if (s != QMM_OK) return s;
        if (overlaps(workspace, need, wg, wbytes) || overlaps(workspace, need, wu, wbytes) ||
            overlaps(workspace, need, x_bf16, sizeof(uint16_t) * static_cast<size_t>(m) * k) ||
            overlaps(workspace, need, h_bf16, hbytes))
            return QMM_ERR_UNSUPPORTED;
    }
    LaunchCtx ctx;
    if (!make_ctx(&ctx)) return QMM_ERR_CUDA;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (two_phase)
        return from_cuda(launch_gemm_geglu_two_phase(static_cast<const uint8_t *>(wg),
                                                     static_cast<const uint8_t *>(wu), x_bf16,
                                                     h_bf16, m, n, k,
                                                     static_cast<uint16_t *>(workspace), st, ctx));
    return from_cuda(launch_gemm_q4_0_geglu(static_cast<const uint8_t *>(wg),
                                            static_cast<const uint8_t *>(wu), x_bf16, h_bf16, m, n,
                                            k, st, ctx));
}

const char *qmm_status_string(qmm_status status) {
    switch (status) {
        case QMM_OK: return "ok";
        case QMM_ERR_NULL: return "null pointer argument";
        case QMM_ERR_SHAPE: return "invalid shape (k % 32 != 0, a size < 1, or m out of range)";
        case QMM_ERR_ALIGN: return "pointer alignment not supported by this call";
        case QMM_ERR_UNSUPPORTED: return "valid arguments not supported by this build";
        case QMM_ERR_CUDA: return "CUDA runtime error";
        case QMM_ERR_TIMEOUT: return "a device-side wait timed out";
        case QMM_ERR_SCRATCH:
            return "problem larger than the entry point's fixed scratch (qmm_gemm_q4_0_prefill: k > 131072)";
    }
    return "unknown status";
}

int qmm_version(void) { return 400; }  // 0.4.0: qmm_copy added

qmm_status qmm_get_device_error(qmm_stream_t stream) {
    cudaError_t e;
    if (!device_state(&e)) return QMM_ERR_CUDA;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return QMM_ERR_CUDA;
    uint32_t word = 0;
    const uint32_t zero = 0;
    if (cudaMemcpyFromSymbol(&word, g_device_error, sizeof word) != cudaSuccess) return QMM_ERR_CUDA;
    if (word != 0 && cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero) != cudaSuccess)
        return QMM_ERR_CUDA;
    return word == 0 ? QMM_OK : static_cast<qmm_status>(word);
}

void qmm_set_wait_timeout_ns(uint64_t ns) {
    g_timeout_ns.store(ns == 0 ? kDefaultTimeoutNs : ns, std::memory_order_relaxed);
}

qmm_status qmm_selftest_wait_timeout(uint64_t timeout_ns, qmm_stream_t stream) {
    LaunchCtx ctx;
    if (!make_ctx(&ctx)) return QMM_ERR_CUDA;
    ctx.timeout_ns = timeout_ns;
    return from_cuda(launch_selftest_wait(reinterpret_cast<cudaStream_t>(stream), ctx));
}

}  // extern "C"
