// Host-only check of the decode GEMV's launch-shape chooser (stream_shape in
// qmm_gemv_impl.cuh), compiled with nvcc and run by test_launch_shapes.py on
// a machine without a GPU.  For every format, M = 1..16, every lanes-per-row
// / rows-per-lane form the dispatcher uses, and a grid of K and N, it checks
// the shape's structure and prints each shape that does not fit the shared-
// memory budget (those take the byte-wise kernel).
#include <cstdio>

#include "qmm_gemv_impl.cuh"

using namespace qmm;

namespace {

bool pow2(int v) { return v > 0 && (v & (v - 1)) == 0; }

int violations = 0;

void fail(const char *what, const char *fmt, int M, int L, int R, long long k, long long n) {
    std::printf("VIOLATION %s: %s M=%d L=%d R=%d k=%lld n=%lld\n", what, fmt, M, L, R, k, n);
    ++violations;
}

template <Fmt F, int M, int L, int R, bool RP = false>
void check(const char *fmt) {
    constexpr int kRowsPerWarp = 32 / L * R;
    for (long long k : {256LL, 512LL, 768LL, 1024LL, 1280LL, 2048LL, 4096LL, 8192LL, 16384LL,
                        32768LL, 65536LL, 1LL << 20}) {
        for (long long n : {1LL, 31LL, 100LL, 512LL, 2048LL, 3072LL, 8192LL, 16384LL, 262144LL,
                            1LL << 22}) {
            const long long tiles = (n + kRowsPerWarp - 1) / kRowsPerWarp;
            const StreamShape sh = stream_shape<F, M, L, R>(tiles, k, 152);
            const long long chunks = k / kChunkK;
            if (!pow2(sh.kw) || sh.kw > QMM_GEMV_MAX_KW) fail("kw", fmt, M, L, R, k, n);
            if (!pow2(sh.ksplit) || sh.ksplit > QMM_GEMV_MAX_KSPLIT) fail("ksplit", fmt, M, L, R, k, n);
            if (static_cast<long long>(sh.kw) * sh.ksplit * sh.cpw != chunks) fail("K cover", fmt, M, L, R, k, n);
            if (sh.stages < 1 || sh.stages > sh.cpw) fail("stages", fmt, M, L, R, k, n);
            if (sh.rw < 1 || sh.rw * sh.kw * 32 > QMM_GEMV_MAX_THREADS) fail("threads", fmt, M, L, R, k, n);
            if (RP && (sh.smem > kGemvSmemCap || sh.cpw * (kChunkK / L) > kRpMaxProducts))  // another form runs
                std::printf("ROWPAIR_REFUSED %s M=%d L=%d R=%d k=%lld n=%lld\n", fmt, M, L, R, k, n);
            else if (sh.smem > kGemvSmemCap)
                std::printf("REFUSED %s M=%d L=%d R=%d k=%lld n=%lld\n", fmt, M, L, R, k, n);
        }
    }
}

// the (lanes per row, rows per lane) forms launch_m can pick for this M
template <Fmt F, int M>
void check_m(const char *fmt) {
    if constexpr (M <= QMM_GEMV_R2_MAX_M) {
        check<F, M, 2, QMM_GEMV_R_SMALL>(fmt);
        check<F, M, 1, 2>(fmt);
        check<F, M, 2, 2>(fmt);  // GeGLU, small problems
    } else if constexpr (M <= QMM_GEMV_R_WIDE_MAX_M) {
        check<F, M, 1, 2>(fmt);
        check<F, M, 1, 1>(fmt);
    } else {
        check<F, M, 1, 1>(fmt);
        check<F, M, 1, 2>(fmt);  // GeGLU
    }
    if constexpr (F == Fmt::Q4_0 && M >= QMM_GEMV_RP_MIN_M)  // the row-pair form
        check<F, M, QMM_GEMV_RP_L, QMM_GEMV_RP_R, true>(fmt);
}

template <Fmt F, int... Ms>
void all(const char *fmt) {
    (check_m<F, Ms>(fmt), ...);
}

}  // namespace

int main() {
    all<Fmt::Q4_0, 1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12, 13, 14, 15, 16>("q4_0");
    all<Fmt::Q8_0, 1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12, 13, 14, 15, 16>("q8_0");
    std::printf("violations %d\n", violations);
    return violations != 0;
}
