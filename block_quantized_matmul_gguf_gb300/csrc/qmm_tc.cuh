// qmm_tc.cuh -- inline-PTX wrappers shared by the tensor-core GEMM kernels:
// TMA tile loads, tensor-memory allocation and access, tcgen05 MMA and
// commit, shared-memory matrix descriptors, cluster barriers and the bounded
// mbarrier waits with a shared abort flag.
#pragma once

#include "qmm_internal.h"

namespace qmm {

// ---- PTX wrappers --------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, "
        "{%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// X tile load whose completion is counted on a barrier that may live in the
// peer CTA of the pair (the leader's).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *map, int x,
                                                 int y, uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster)
        : "memory");
}

// TMEM for the pair: executed by one warp in each CTA of the pair.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t slot_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// TMEM for one CTA (no pair): executed by one warp.
__device__ __forceinline__ void tmem_alloc_cta(uint32_t slot_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_cta(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// D (TMEM) += A (TMEM) x B (shared-memory descriptor), one CTA.
__device__ __forceinline__ void umma_bf16_cta_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                                 uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive (once) on this CTA's barrier when all previously issued MMAs of this
// thread complete.
__device__ __forceinline__ void umma_commit_cta(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// 16 consecutive 32-bit TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld_16cols(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 64 consecutive 32-bit TMEM columns of this thread's lane (waits for them).
__device__ __forceinline__ void tmem_ld_64cols(uint32_t taddr, uint32_t (&r)[64]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_nranks() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_barrier() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
                 ::: "memory");
}

// Address of the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}

// Arrive on a barrier of either CTA of the pair (CTA-scope release).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar_cluster) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}

// Bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned) from
// this CTA's shared memory to a cluster peer's, completing as transaction
// bytes on the peer's barrier.
__device__ __forceinline__ void bulk_s2cluster(uint32_t dst_cluster, uint32_t src_cta, uint32_t bytes,
                                               uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst_cluster),
        "r"(src_cta), "r"(bytes), "r"(bar_cluster)
        : "memory");
}

// Arrive on a cluster peer's barrier without ordering any data (a signal).
__device__ __forceinline__ void mbar_arrive_remote_relaxed(uint32_t bar_cluster) {
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster)
                 : "memory");
}

// Announces bytes a TMA load will deliver; publishes no data, so relaxed.
__device__ __forceinline__ void mbar_expect_tx_cluster(uint32_t bar_cluster, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.relaxed.cluster.shared::cluster.b64 _, [%0], %1;" ::"r"(
                     bar_cluster),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D (TMEM) += A (TMEM, both CTAs' halves) x B (shared-memory descriptor).
__device__ __forceinline__ void umma_bf16_pair_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                                  uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 16 consecutive 32-bit TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_st_16cols(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
        "r"(v[15])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Arrive (once each) on the barrier at this shared-memory offset in both CTAs
// of the pair when all previously issued MMAs of this thread complete.
__device__ __forceinline__ void umma_commit_pair(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
        "[%0], %1;" ::"r"(bar),
        "h"(static_cast<unsigned short>(3))
        : "memory");
}

__device__ __forceinline__ void tmem_ld_32cols(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows
// 128 bytes apart, 8-row groups 1024 bytes apart (SBO); LBO unused.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(1) << 16;             // LBO (ignored for swizzled K-major)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;     // SBO
    d |= static_cast<uint64_t>(1) << 46;             // descriptor version
    d |= static_cast<uint64_t>(2) << 61;             // 128-byte swizzle
    return d;
}

__device__ __forceinline__ bool abort_set(const int *flag) {
    return *reinterpret_cast<const volatile int *>(flag) != 0;
}

// try_wait with a suspend-time hint: the thread may sleep up to `ns`
// nanoseconds (instead of the system's default limit) unless the phase
// completes first, so that a waiting warp takes fewer issue slots.
__device__ __forceinline__ bool mbar_try_wait_hint(uint32_t bar_addr, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; "
        "selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(bar_addr), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}

#ifndef QMM_GEMM_SUSPEND_NS
#define QMM_GEMM_SUSPEND_NS 0      // suspend hint of the pipeline waits (0: default limit)
#endif
#ifndef QMM_GEMM_EPI_SUSPEND_NS
#define QMM_GEMM_EPI_SUSPEND_NS 0  // suspend hint of the epilogue's accumulator wait
#endif

// Bounded wait that also gives up as soon as another role has aborted.
template <uint32_t HINT = QMM_GEMM_SUSPEND_NS>
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, int *flag,
                                              const LaunchCtx &ctx) {
    auto try_once = [&]() {
        return HINT ? mbar_try_wait_hint(bar, parity, HINT) : mbar_try_wait(bar, parity);
    };
    if (try_once()) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 0; it < (1u << 30); ++it) {
        if (try_once()) return true;
        if ((it & 15u) == 15u) {
            if (abort_set(flag)) return false;
            if (global_timer_ns() - t0 > ctx.timeout_ns) break;
        }
    }
    *reinterpret_cast<volatile int *>(flag) = 1;
    record_error(ctx, kDevErrTimeout);
    return false;
}

// Wait whose acquire covers releases made by threads of the peer CTA.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar_addr, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2; "
        "selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(bar_addr), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool wait_or_abort_cluster(uint32_t bar, uint32_t parity, int *flag,
                                                      const LaunchCtx &ctx) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 0; it < (1u << 30); ++it) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if ((it & 15u) == 15u) {
            if (abort_set(flag)) return false;
            if (global_timer_ns() - t0 > ctx.timeout_ns) break;
        }
    }
    *reinterpret_cast<volatile int *>(flag) = 1;
    record_error(ctx, kDevErrTimeout);
    return false;
}

// Warp-wide form: every lane polls, and the warp agrees on the outcome so
// that the following __syncwarp / .sync.aligned instructions stay uniform.
template <uint32_t HINT = QMM_GEMM_SUSPEND_NS>
__device__ __forceinline__ bool warp_wait_or_abort(uint32_t bar, uint32_t parity, int *flag,
                                                   const LaunchCtx &ctx) {
    const bool ok = wait_or_abort<HINT>(bar, parity, flag, ctx);
    return __all_sync(0xFFFFFFFFu, ok);
}

// Bounded wait that ignores the abort flag (used to drain our own copies).
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity, const LaunchCtx &ctx) {
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 0; it < (1u << 30); ++it) {
        if (mbar_try_wait(bar, parity)) return;
        if ((it & 15u) == 15u && global_timer_ns() - t0 > ctx.timeout_ns) break;
    }
    record_error(ctx, kDevErrTimeout);
}

__device__ __forceinline__ void mbar_init_addr(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_addr(uint32_t bar) {
    asm volatile("{ .reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0]; }" ::"r"(bar)
                 : "memory");
}
__device__ __forceinline__ void mbar_expect_tx_addr(uint32_t bar, uint32_t bytes) {
    asm volatile("{ .reg .b64 st; mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1; }" ::"r"(
                     bar),
                 "r"(bytes)
                 : "memory");
}

// GELU, tanh form, as z * sigmoid(2a) with a = sqrt(2/pi) * (z + 0.044715 z^3)
// (equal to z/2 * (1 + tanh(a))).  The result is rounded to bf16, so the
// fast exponential and division are accurate enough; the exponent is
// clamped so that the divisor stays finite and in the fast division's range.
__device__ __forceinline__ float gelu_tanh_fast(float z) {
    const float a = 0.7978845608028654f * fmaf(0.044715f * z, z * z, z);
    return __fdividef(z, 1.0f + __expf(fminf(-2.0f * a, 80.0f)));
}

__device__ __forceinline__ uint16_t to_bf16(float v) {
    uint16_t r;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(v));
    return r;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// ---- weight decode to bf16 (exact fp32 product, one rounding) ---------------

// 2^23 + (v & mask) as a float.  `magic` (0x4B000000) comes from the kernel
// parameters so that it sits in a register: with the mask and the magic both
// immediates the compiler splits the extraction into two LOP3.
__device__ __forceinline__ float mag(uint32_t v, uint32_t mask, uint32_t magic) {
    return __uint_as_float((v & mask) | magic);
}

// bf16 pair (k, k+1) from two 2^23-magic nibble floats: exact (nibble-8)*2^s
// by one packed add, exact (nibble-8)*d by one packed multiply with d*2^-s,
// one rounding to bf16.
__device__ __forceinline__ uint32_t w_pair(float ma, float mb, float2 c, float2 ds) {
    const float2 f = __fadd2_rn(make_float2(ma, mb), c);
    const float2 w = __fmul2_rn(f, ds);
    return pack_bf16x2(w.x, w.y);
}

// Dequantise qs words [I0, I0 + NI) of Q4_0 block `b` (0..7) of a 144-byte
// row chunk held in wd[36].  Word i holds weights 4i..4i+3 (low nibbles) and
// 16+4i..19+4i (high nibbles); out[0..NI/2) are the low 16-byte chunks
// (K 8*I0/2 ..), out[NI/2..NI) the high ones (K 16 + ...).
template <int I0, int NI>
__device__ __forceinline__ void dequant_words_bf16(const uint32_t (&wd)[36], int b, uint32_t magic,
                                                   uint4 (&out)[NI]) {
    const int base = (18 * b) >> 2;
    uint32_t dbits, q[4];
    if ((b & 1) == 0) {
        dbits = wd[base] & 0xFFFFu;
#pragma unroll
        for (int i = 0; i < 4; ++i) q[i] = __byte_perm(wd[base + i], wd[base + i + 1], 0x5432);
    } else {
        dbits = wd[base] >> 16;
#pragma unroll
        for (int i = 0; i < 4; ++i) q[i] = wd[base + 1 + i];
    }
    const float d = half_bits_to_float(dbits);
    const float d4 = d * 0.0625f, d8 = d * 0.00390625f, d12 = d * 0.000244140625f,
                d16 = d * 1.52587890625e-05f;
    const float2 c08 = make_float2(-8388616.0f, -8390656.0f);  // s = 0, 8
    const float2 c168 = make_float2(-8912896.0f, -8390656.0f); // s = 16, 8
    const float2 c412 = make_float2(-8388736.0f, -8421376.0f); // s = 4, 12
    const float2 d08 = make_float2(d, d8), d168 = make_float2(d16, d8), d412 = make_float2(d4, d12);
    uint32_t lo[2 * NI], hi[2 * NI];
#pragma unroll
    for (int j = 0; j < NI; ++j) {
        const uint32_t v = q[I0 + j], u = v >> 16;
        // low nibbles: weights 4i .. 4i+3
        lo[2 * j + 0] = w_pair(mag(v, 0x0000000Fu, magic), mag(v, 0x00000F00u, magic), c08, d08);
        lo[2 * j + 1] = w_pair(mag(v, 0x000F0000u, magic), mag(u, 0x00000F00u, magic), c168, d168);
        // high nibbles: weights 16+4i .. 19+4i
        hi[2 * j + 0] = w_pair(mag(v, 0x000000F0u, magic), mag(v, 0x0000F000u, magic), c412, d412);
        hi[2 * j + 1] = w_pair(mag(u, 0x000000F0u, magic), mag(u, 0x0000F000u, magic), c412, d412);
    }
#pragma unroll
    for (int c = 0; c < NI / 2; ++c) {
        out[c] = make_uint4(lo[4 * c], lo[4 * c + 1], lo[4 * c + 2], lo[4 * c + 3]);
        out[NI / 2 + c] = make_uint4(hi[4 * c], hi[4 * c + 1], hi[4 * c + 2], hi[4 * c + 3]);
    }
}

// Q8_0 byte with its top bit flipped (q + 128) in the mantissa of 2^23;
// flip = 2^23's pattern with that byte's top bit set.  One LOP3.
__device__ __forceinline__ float mag8(uint32_t v, uint32_t mask, uint32_t flip) {
    return __uint_as_float((mask & (v ^ flip)) | (~mask & flip));
}

// Dequantise the Q8_0 block that starts `o` bytes into a window of row bytes
// held in wd[NW] (o % 4 is 0 or 2): d, then q[0..31] to 16 bf16 pairs in K order.
// (2^23 + (q+128)*2^s) - (2^23 + 128*2^s) is q*2^s exactly; times d*2^-s it
// is q*d exactly (an 8-bit by 11-bit product), rounded once to bf16.
template <int NW>
__device__ __forceinline__ void dequant_q8_block_bf16(const uint32_t (&wd)[NW], int o,
                                                      uint32_t flip0, uint32_t flip1,
                                                      uint32_t (&out)[16]) {
    const int base = o >> 2;
    uint32_t dbits, q[8];
    if ((o & 3) == 0) {  // d in the low half of word `base`, q from byte o + 2
        dbits = wd[base] & 0xFFFFu;
#pragma unroll
        for (int i = 0; i < 8; ++i) q[i] = __byte_perm(wd[base + i], wd[base + i + 1], 0x5432);
    } else {  // d in the high half, q word-aligned
        dbits = wd[base] >> 16;
#pragma unroll
        for (int i = 0; i < 8; ++i) q[i] = wd[base + 1 + i];
    }
    const float d = half_bits_to_float(dbits);
    const float2 c = make_float2(-8388736.0f, -8421376.0f);  // -(2^23 + 128*2^s), s = 0, 8
    const float2 ds = make_float2(d, d * 0.00390625f);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t v = q[i], u = v >> 16;
        out[2 * i + 0] = w_pair(mag8(v, 0x000000FFu, flip0), mag8(v, 0x0000FF00u, flip1), c, ds);
        out[2 * i + 1] = w_pair(mag8(u, 0x000000FFu, flip0), mag8(u, 0x0000FF00u, flip1), c, ds);
    }
}

}  // namespace qmm
