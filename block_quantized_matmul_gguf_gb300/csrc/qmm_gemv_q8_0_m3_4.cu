// qmm_gemv_q8_0_m3_4.cu -- Q8_0 decode GEMV kernels for M = 3..4
// (kernels and design notes in qmm_gemv_impl.cuh; split by M so that the
// translation units build in parallel).
#include "qmm_gemv_impl.cuh"

namespace qmm {

cudaError_t launch_gemv_q8_0_m3_4(const GemvProblem *probs, int count, const float *x, int m,
                                  int64_t k, cudaStream_t stream, const LaunchCtx &ctx) {
    return launch_m_range<Fmt::Q8_0, 3, 4>(probs, count, x, m, k, stream, ctx);
}

}  // namespace qmm
