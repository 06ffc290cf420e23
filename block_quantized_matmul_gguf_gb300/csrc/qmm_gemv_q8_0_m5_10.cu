// qmm_gemv_q8_0_m5_10.cu -- Q8_0 decode GEMV kernels for M = 5..10
// (kernels and design notes in qmm_gemv_impl.cuh; split by M so that the
// translation units build in parallel).
#include "qmm_gemv_impl.cuh"

namespace qmm {

cudaError_t launch_gemv_q8_0_m5_10(const GemvProblem *probs, int count, const float *x, int m,
                                  int64_t k, cudaStream_t stream, const LaunchCtx &ctx) {
    return launch_m_range<Fmt::Q8_0, 5, 10>(probs, count, x, m, k, stream, ctx);
}

}  // namespace qmm
