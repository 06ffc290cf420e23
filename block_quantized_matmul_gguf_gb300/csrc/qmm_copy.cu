// qmm_copy.cu -- stream-ordered copies made by the SMs (qmm_copy): the few
// kilobytes of activations and outputs that a decode step moves between
// page-locked host memory and the device.  Such memory is mapped into the
// device's address space at its host address, so a kernel reads and writes it
// with plain loads and stores.  A copy-engine transfer in the same place costs
// several microseconds whatever its size; a launch with programmatic
// dependent launch starts while its predecessor drains, and lets its
// successor start (and prefetch its weights) while it runs.
#include "qmm_internal.h"

#include <algorithm>

namespace qmm {
namespace {

// n16 pieces of 16 bytes, then `tail` bytes (src and dst 16-byte aligned).
__global__ void __launch_bounds__(256) copy16_kernel(const uint4 *__restrict__ src,
                                                     uint4 *__restrict__ dst, int64_t n16,
                                                     int tail) {
    // src may be the previous launch's output and dst its input: both wait
    pdl_wait();
    pdl_launch_dependents();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t first = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (int64_t i = first; i < n16; i += stride) dst[i] = src[i];
    if (first < tail) {
        const uint8_t *s = reinterpret_cast<const uint8_t *>(src + n16);
        uint8_t *d = reinterpret_cast<uint8_t *>(dst + n16);
        d[first] = s[first];
    }
}

// Any alignment: one byte per thread and step.
__global__ void __launch_bounds__(256) copy1_kernel(const uint8_t *__restrict__ src,
                                                    uint8_t *__restrict__ dst, int64_t n) {
    pdl_wait();
    pdl_launch_dependents();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
        dst[i] = src[i];
}

}  // namespace

cudaError_t launch_copy(void *dst, const void *src, size_t bytes, cudaStream_t stream) {
    if (bytes == 0) return cudaSuccess;
    const int64_t cap = static_cast<int64_t>(device_sm_count()) * 4;  // CTAs: a few per SM at most
    const bool vec = ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15) == 0;
    if (vec) {
        const int64_t n16 = static_cast<int64_t>(bytes / 16);
        const int tail = static_cast<int>(bytes % 16);
        const int64_t threads = std::max<int64_t>(n16, tail);
        const unsigned blocks = static_cast<unsigned>(std::min<int64_t>((threads + 255) / 256, cap));
        return launch_kernel(copy16_kernel, dim3(blocks), dim3(256), 0, stream, 1,
                             static_cast<const uint4 *>(src), static_cast<uint4 *>(dst), n16, tail);
    }
    const int64_t n = static_cast<int64_t>(bytes);
    const unsigned blocks = static_cast<unsigned>(std::min<int64_t>((n + 255) / 256, cap));
    return launch_kernel(copy1_kernel, dim3(blocks), dim3(256), 0, stream, 1,
                         static_cast<const uint8_t *>(src), static_cast<uint8_t *>(dst), n);
}

}  // namespace qmm
