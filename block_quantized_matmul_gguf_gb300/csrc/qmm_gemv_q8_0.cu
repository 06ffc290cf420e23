// qmm_gemv_q8_0.cu -- Q8_0 instantiation of the decode GEMV kernels
// (kernels and design notes in qmm_gemv_impl.cuh; one translation unit per
// format so the two build in parallel).
#include "qmm_gemv_impl.cuh"

namespace qmm {

cudaError_t launch_gemv_q8_0(const uint8_t *w, const float *x, float *y, int m, int64_t n,
                             int64_t k, cudaStream_t stream, const LaunchCtx &ctx) {
    return launch_fmt<Fmt::Q8_0>(w, x, y, m, n, k, stream, ctx);
}

}  // namespace qmm
