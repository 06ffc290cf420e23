// qmm_dequant.cu -- bit-exact dequantization of GGUF Q4_0 / Q8_0 blocks to a
// dense fp32 matrix.
//
// Formats (the Q4_0 and Q8_0 dispatches of "Add generated quant-kernel JIT
// and accelerate Gemma4, BGE-M3, and GLiNER2", section "Validation"):
//   Q4_0: binary16 d, then qs[16]; weight j < 16 is the low nibble of qs[j],
//         weight j >= 16 the high nibble of qs[j-16]; w = (nibble - 8) * d.
//   Q8_0: binary16 d, then int8 q[32]; w = q * d.
//
// The path is write-bound (18 or 34 bytes in, 128 bytes out per block): eight
// lanes share a block and each writes four consecutive outputs, so a warp
// stores 512 contiguous bytes (four blocks) per instruction.  Each output is
// the IEEE binary32 product (float)(nibble-8) * d or (float)q * d, which is
// exact, so the result matches the definition bit for bit, including the
// sign of zero.
#include "qmm_internal.h"

namespace qmm {
namespace {

template <Fmt F>
__device__ __forceinline__ float4 dequant_quad(const uint8_t *__restrict__ blk, int quad,
                                               float d) {
    float v[4];
    if constexpr (F == Fmt::Q4_0) {
        const uint8_t *qs = blk + 2 + (quad & 3) * 4;
        const bool high = quad >= 4;  // quads 4..7 are weights 16..31
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const int byte = __ldg(qs + t);
            const int nib = high ? (byte >> 4) : (byte & 0x0F);
            v[t] = static_cast<float>(nib - 8) * d;
        }
    } else {
        const uint8_t *q = blk + 2 + quad * 4;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const int8_t qv = static_cast<int8_t>(__ldg(q + t));
            v[t] = static_cast<float>(qv) * d;
        }
    }
    return make_float4(v[0], v[1], v[2], v[3]);
}

template <Fmt F, bool kVecStore>
__global__ void __launch_bounds__(256) dequant_kernel(const uint8_t *__restrict__ w,
                                                      float *__restrict__ out,
                                                      int64_t nblocks, LaunchCtx ctx) {
    constexpr int kBB = F == Fmt::Q4_0 ? kQ4_0Bytes : kQ8_0Bytes;
    pdl_wait();
    pdl_launch_dependents();
    const int64_t total = nblocks * 8;  // eight quads of four outputs per block
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; g < total;
         g += stride) {
        const int64_t b = g >> 3;
        const int quad = static_cast<int>(g & 7);
        const uint8_t *blk = w + b * kBB;
        const uint32_t dbits = __ldg(blk) | (static_cast<uint32_t>(__ldg(blk + 1)) << 8);
        const float d = half_bits_to_float(dbits);
        const float4 v = dequant_quad<F>(blk, quad, d);
        float *dst = out + b * kQK + quad * 4;
        if constexpr (kVecStore) {
            *reinterpret_cast<float4 *>(dst) = v;
        } else {
            dst[0] = v.x;
            dst[1] = v.y;
            dst[2] = v.z;
            dst[3] = v.w;
        }
    }
}

template <Fmt F>
cudaError_t launch_fmt(const uint8_t *w, float *out, int64_t nblocks, cudaStream_t stream,
                       const LaunchCtx &ctx) {
    const int threads = 256;
    const int64_t want = (nblocks * 8 + threads - 1) / threads;
    const int64_t cap = static_cast<int64_t>(device_sm_count()) * 16;
    const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
    if ((reinterpret_cast<uintptr_t>(out) & 15) == 0)
        return launch_kernel(dequant_kernel<F, true>, dim3(grid), dim3(threads), 0, stream, 1,
                             w, out, nblocks, ctx);
    return launch_kernel(dequant_kernel<F, false>, dim3(grid), dim3(threads), 0, stream, 1, w,
                         out, nblocks, ctx);
}

}  // namespace

cudaError_t launch_dequant(Fmt fmt, const uint8_t *w, float *out, int64_t n, int64_t k,
                           cudaStream_t stream, const LaunchCtx &ctx) {
    const int64_t nblocks = n * (k / kQK);
    return fmt == Fmt::Q4_0 ? launch_fmt<Fmt::Q4_0>(w, out, nblocks, stream, ctx)
                            : launch_fmt<Fmt::Q8_0>(w, out, nblocks, stream, ctx);
}

}  // namespace qmm
