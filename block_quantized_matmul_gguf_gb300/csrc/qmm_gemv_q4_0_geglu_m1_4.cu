// qmm_gemv_q4_0_geglu_m1_4.cu -- fused GeGLU decode kernels (Q4_0 gate and up
// weights) for M = 1..4 (kernels and design notes in qmm_gemv_impl.cuh).
#include "qmm_gemv_impl.cuh"

namespace qmm {

cudaError_t launch_geglu_q4_0_m1_4(const GemvProblem *gate_up, const float *x, int m,
                                   int64_t k, cudaStream_t stream, const LaunchCtx &ctx) {
    return launch_m_range<Fmt::Q4_0, 1, 4, true>(gate_up, 2, x, m, k, stream, ctx);
}

}  // namespace qmm
