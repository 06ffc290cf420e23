// qmm_device.cuh -- device-side helpers shared by the library's kernels:
// launch context, bounded mbarrier waits, bulk copies, PDL control.
//
// Inline PTX only for operations CUDA C++ does not expose (mbarrier with
// transaction counts, cp.async.bulk, griddepcontrol, tcgen05).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace qmm {

// Error codes written to the device error word (match qmm_status values).
enum : uint32_t { kDevErrTimeout = 6 };

// Per-launch context every kernel receives.
struct LaunchCtx {
    uint32_t *err;        // device error word (device-global, one per GPU)
    uint64_t timeout_ns;  // limit of each bounded wait (GPU global timer)
};

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void record_error(const LaunchCtx &ctx, uint32_t code) {
    atomicExch(ctx.err, code);
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- programmatic dependent launch ------------------------------------------
// Wait until the preceding kernel in the stream has completed and its memory
// is visible (no-op when the launch was not programmatic).
__device__ __forceinline__ void pdl_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Allow the next kernel in the stream to be scheduled.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- mbarrier ----------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile(
        "{ .reg .b64 st; mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1; }" ::"r"(
            smem_addr(bar)),
        "r"(bytes)
        : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("{ .reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0]; }" ::"r"(
                     smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar_addr, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; "
        "selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(bar_addr), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity to complete.  Returns
// false (and records a timeout) when the limit passes first.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity,
                                          const LaunchCtx &ctx) {
    const uint32_t a = smem_addr(bar);
    if (mbar_try_wait(a, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 0; it < (1u << 30); ++it) {
        if (mbar_try_wait(a, parity)) return true;
        if ((it & 15u) == 15u && global_timer_ns() - t0 > ctx.timeout_ns) break;
    }
    record_error(ctx, kDevErrTimeout);
    return false;
}

// ---- bulk copies (TMA engine, no tensor map) ---------------------------------
// Copies `bytes` (multiple of 16; both addresses 16-byte aligned) from global
// to this CTA's shared memory; completion is counted on `bar` in bytes.
__device__ __forceinline__ void bulk_g2s(void *dst_smem, const void *src_gmem, uint32_t bytes,
                                         uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, "
        "[%3];" ::"r"(smem_addr(dst_smem)),
        "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// ---- shared-memory loads --------------------------------------------------------
// Plain C++ accesses (not volatile asm), so the compiler may schedule them
// early; the "memory" clobber of every barrier wait keeps them after it.
__device__ __forceinline__ uint4 lds128(const void *p) {
    return *reinterpret_cast<const uint4 *>(p);
}

__device__ __forceinline__ float4 lds128f(const float *p) {
    return *reinterpret_cast<const float4 *>(p);
}

// binary16 bit pattern -> fp32 (exact for every pattern; hardware convert).
__device__ __forceinline__ float half_bits_to_float(uint32_t h16) {
    float f;
    asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"(static_cast<unsigned short>(h16)));
    return f;
}

}  // namespace qmm
