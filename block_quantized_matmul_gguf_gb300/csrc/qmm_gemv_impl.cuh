// qmm_gemv_impl.cuh -- decode GEMV y[m][n] = sum_k x[m][k] * w[n][k] for GGUF
// Q4_0 / Q8_0 weights and M = 1..16 fp32 activation rows.
//
// These are the 342 Q4_0 and one Q8_0 (LM head) dispatches per decode token
// counted in "Add generated quant-kernel JIT and accelerate Gemma4, BGE-M3,
// and GLiNER2", section "Validation"; M > 1 covers the batching named in its
// "Summary".  The work is a stream of weight bytes read once, so the design
// is about HBM and issue slots, not tensor cores.
//
// Streaming kernel (K % 256 == 0, 16-byte aligned w and x):
//  * A CTA owns 32 rows; lane r of every warp owns row r.  The K dimension is
//    cut into chunks of 256 weights (8 blocks: 144 bytes of Q4_0, 272 of
//    Q8_0), which keeps every row chunk 16-byte aligned.  Warps take chunks
//    round robin; small-N shapes also split K across a thread-block cluster
//    and reduce through distributed shared memory (no global scratch, fixed
//    summation order).
//  * Each warp runs its own ring of S shared-memory stages.  Every lane
//    issues one cp.async.bulk of its row's chunk; an mbarrier with a byte
//    count tracks the stage.  Shared-memory rows are 144 (272) bytes apart,
//    so the lanes' 16-byte reads hit distinct banks.
//  * Activations are staged once per CTA slice in shared memory, pre-scaled
//    by the power of two that matches where each nibble sits in its word
//    (see below), and read as warp-wide broadcasts.
//  * Decode without int->float conversions: OR-ing a nibble (or an offset
//    byte) into the mantissa of 2^23 gives 2^23 + v*2^s exactly; one FADD of
//    -(2^23 + 8*2^s) (Q4_0) or -(2^23 + 128*2^s) (Q8_0) leaves
//    (nibble-8)*2^s or q*2^s exactly, and the product with x*2^-s is the
//    exact w-free product (nibble-8)*x.  Adds and FMAs run as packed f32x2.
//  * Per block: acc = sum_j (nibble_j - 8) * x_j in fp32, then y += d * acc.
//
// Byte-wise kernel: any K % 32 == 0 and any alignment; a warp per row.
#pragma once

#include "qmm_internal.h"

#include <algorithm>

namespace qmm {
namespace {

constexpr int kRowsPerCta = 32;
constexpr int kChunkK = 256;
constexpr uint32_t kMagic = 0x4B000000u;  // 2^23

template <Fmt F>
struct StreamFmt;
template <>
struct StreamFmt<Fmt::Q4_0> {
    static constexpr int kChunkBytes = 144;
};
template <>
struct StreamFmt<Fmt::Q8_0> {
    static constexpr int kChunkBytes = 272;
};

// Power-of-two exponent s by which position j (0..31) of a block is
// pre-scaled (x' = x * 2^-s).  Q4_0: a qs word holds positions
// 4i..4i+3 (low nibbles, bits 0,8,16,24) and 16+4i..19+4i (high nibbles,
// bits 4,12,20,28); bits 0-19 are used in place, bits 20-31 after >> 16.
__device__ __forceinline__ int q4_0_shift(int j) {
    const int t = j & 3;
    if (j < 16) return t == 0 ? 0 : (t == 2 ? 16 : 8);
    return (t & 1) ? 12 : 4;
}
// Q8_0: bytes 0 and 2 of a word are used at bits 0-7 (s = 0), bytes 1 and 3
// at bits 8-15 (s = 8).

__device__ __forceinline__ float mag(uint32_t v, uint32_t mask) {
    return __uint_as_float((v & mask) | kMagic);
}
// Offset byte for Q8_0: ((v ^ 0x80 at the byte's top bit) & mask) | 2^23.
__device__ __forceinline__ float mag8(uint32_t v, uint32_t mask, uint32_t magic_flip) {
    return __uint_as_float((mask & (v ^ magic_flip)) | (~mask & magic_flip));
}

__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }

// Independent FMA chains per output row: at small M the rows alone do not
// give the scheduler enough independent work, so each block's sum is split.
template <int M>
struct Chains {
    static constexpr int value = M <= 2 ? 4 : (M <= 4 ? 2 : 1);
};

// One row chunk (8 Q4_0 blocks, 144 bytes at `src`) against the pre-scaled
// activations `xs` (position 0 of the chunk for row 0; rows XS apart).
template <int M>
__device__ __forceinline__ void q4_0_chunk(const uint8_t *src, const float *xs, int XS,
                                           float (&tot)[M]) {
    constexpr int CH = Chains<M>::value;
    uint32_t wd[36];
#pragma unroll
    for (int t = 0; t < 9; ++t) {
        const uint4 v = lds128(src + 16 * t);
        wd[4 * t + 0] = v.x;
        wd[4 * t + 1] = v.y;
        wd[4 * t + 2] = v.z;
        wd[4 * t + 3] = v.w;
    }
    const float2 c01 = f2(-8388616.0f, -8390656.0f);  // -(2^23 + 8*2^s), s = 0, 8
    const float2 c23 = f2(-8912896.0f, -8390656.0f);  // s = 16, 8
    const float2 c45 = f2(-8388736.0f, -8421376.0f);  // s = 4, 12
#pragma unroll
    for (int b = 0; b < 8; ++b) {
        const int base = (18 * b) >> 2;
        uint32_t dbits, q[4];
        if ((b & 1) == 0) {  // block starts on a word: d low half, qs shifted by 2 bytes
            dbits = wd[base] & 0xFFFFu;
#pragma unroll
            for (int i = 0; i < 4; ++i) q[i] = __byte_perm(wd[base + i], wd[base + i + 1], 0x5432);
        } else {  // block starts 2 bytes into a word: d high half, qs aligned
            dbits = wd[base] >> 16;
#pragma unroll
            for (int i = 0; i < 4; ++i) q[i] = wd[base + 1 + i];
        }
        const float d = half_bits_to_float(dbits);
        float2 acc[M][CH];
#pragma unroll
        for (int m = 0; m < M; ++m)
#pragma unroll
            for (int c = 0; c < CH; ++c) acc[m][c] = f2(0.0f, 0.0f);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t v = q[i], u = v >> 16;
            const float2 p01 = __fadd2_rn(f2(mag(v, 0x0000000Fu), mag(v, 0x00000F00u)), c01);
            const float2 p23 = __fadd2_rn(f2(mag(v, 0x000F0000u), mag(u, 0x00000F00u)), c23);
            const float2 p45 = __fadd2_rn(f2(mag(v, 0x000000F0u), mag(v, 0x0000F000u)), c45);
            const float2 p67 = __fadd2_rn(f2(mag(u, 0x000000F0u), mag(u, 0x0000F000u)), c45);
            const int c = i % CH;
#pragma unroll
            for (int m = 0; m < M; ++m) {
                const float4 xa = lds128f(xs + m * XS + 32 * b + 4 * i);
                const float4 xb = lds128f(xs + m * XS + 32 * b + 16 + 4 * i);
                acc[m][c] = __ffma2_rn(p01, f2(xa.x, xa.y), acc[m][c]);
                acc[m][c] = __ffma2_rn(p23, f2(xa.z, xa.w), acc[m][c]);
                acc[m][c] = __ffma2_rn(p45, f2(xb.x, xb.y), acc[m][c]);
                acc[m][c] = __ffma2_rn(p67, f2(xb.z, xb.w), acc[m][c]);
            }
        }
#pragma unroll
        for (int m = 0; m < M; ++m) {
            float2 a = acc[m][0];
#pragma unroll
            for (int c = 1; c < CH; ++c) a = __fadd2_rn(a, acc[m][c]);
            tot[m] = fmaf(d, a.x + a.y, tot[m]);
        }
    }
}

// One row chunk of 8 Q8_0 blocks (272 bytes).
template <int M>
__device__ __forceinline__ void q8_0_chunk(const uint8_t *src, const float *xs, int XS,
                                           float (&tot)[M]) {
    constexpr int CH = Chains<M>::value;
    uint32_t wd[68];
#pragma unroll
    for (int t = 0; t < 17; ++t) {
        const uint4 v = lds128(src + 16 * t);
        wd[4 * t + 0] = v.x;
        wd[4 * t + 1] = v.y;
        wd[4 * t + 2] = v.z;
        wd[4 * t + 3] = v.w;
    }
    const float2 c = f2(-8388736.0f, -8421376.0f);  // -(2^23 + 128*2^s), s = 0, 8
#pragma unroll
    for (int b = 0; b < 8; ++b) {
        const int base = (34 * b) >> 2;
        uint32_t dbits, q[8];
        if ((b & 1) == 0) {
            dbits = wd[base] & 0xFFFFu;
#pragma unroll
            for (int i = 0; i < 8; ++i) q[i] = __byte_perm(wd[base + i], wd[base + i + 1], 0x5432);
        } else {
            dbits = wd[base] >> 16;
#pragma unroll
            for (int i = 0; i < 8; ++i) q[i] = wd[base + 1 + i];
        }
        const float d = half_bits_to_float(dbits);
        float2 acc[M][CH];
#pragma unroll
        for (int m = 0; m < M; ++m)
#pragma unroll
            for (int h = 0; h < CH; ++h) acc[m][h] = f2(0.0f, 0.0f);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t v = q[i], u = v >> 16;
            const float2 p01 = __fadd2_rn(
                f2(mag8(v, 0x000000FFu, kMagic | 0x80u), mag8(v, 0x0000FF00u, kMagic | 0x8000u)), c);
            const float2 p23 = __fadd2_rn(
                f2(mag8(u, 0x000000FFu, kMagic | 0x80u), mag8(u, 0x0000FF00u, kMagic | 0x8000u)), c);
            const int h = i % CH;
#pragma unroll
            for (int m = 0; m < M; ++m) {
                const float4 xa = lds128f(xs + m * XS + 32 * b + 4 * i);
                acc[m][h] = __ffma2_rn(p01, f2(xa.x, xa.y), acc[m][h]);
                acc[m][h] = __ffma2_rn(p23, f2(xa.z, xa.w), acc[m][h]);
            }
        }
#pragma unroll
        for (int m = 0; m < M; ++m) {
            float2 a = acc[m][0];
#pragma unroll
            for (int h = 1; h < CH; ++h) a = __fadd2_rn(a, acc[m][h]);
            tot[m] = fmaf(d, a.x + a.y, tot[m]);
        }
    }
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
                 ::: "memory");
}
__device__ __forceinline__ float ld_dsmem_f32(const float *local, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                 : "=r"(remote)
                 : "r"(smem_addr(local)), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

struct StreamParams {
    const uint8_t *w;
    const float *x;
    float *y;
    int n;            // rows of W
    int k;            // columns (multiple of 256)
    int stages;       // ring depth per warp
    int cpc;          // chunks per CTA (the K range of one cluster rank)
    int xs_chunks;    // chunks per activation slice
    LaunchCtx ctx;
};

// Grid: blockIdx.x = group * ksplit + rank, with a cluster of ksplit CTAs
// along x.  Warp w of group g owns rows (g*nw + w)*32 .. +31; cluster rank r
// owns chunks [r*cpc, (r+1)*cpc) of K.  Every warp streams all chunks of its
// CTA's K range for its own rows.
template <Fmt F, int M>
__global__ void __launch_bounds__(128) gemv_stream_kernel(StreamParams p) {
    constexpr int CB = StreamFmt<F>::kChunkBytes;
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nw = blockDim.x >> 5;
    const int S = p.stages;
    const uint32_t rank = cluster_ctarank();
    const uint32_t ksplit = cluster_nctarank();
    const int group = static_cast<int>(blockIdx.x / ksplit);
    const int row0 = (group * nw + warp) * kRowsPerCta;
    const int row = row0 + lane;
    const bool row_ok = row < p.n;
    const int valid_rows = max(0, min(kRowsPerCta, p.n - row0));
    const int XS = p.xs_chunks * kChunkK;
    const size_t rowbytes = static_cast<size_t>(p.k / kChunkK) * CB;
    const int c_begin = static_cast<int>(rank) * p.cpc;
    const int cpc = p.cpc;

    // shared memory: ring [nw][S][32 rows][CB] | xs [M][XS] | part [nw][M][32] | bars [nw][S]
    uint8_t *my_ring = smem + static_cast<size_t>(warp) * S * kRowsPerCta * CB;
    float *xs = reinterpret_cast<float *>(smem + static_cast<size_t>(nw) * S * kRowsPerCta * CB);
    float *part = xs + M * XS;
    uint64_t *bars = reinterpret_cast<uint64_t *>(part + nw * M * kRowsPerCta);
    uint64_t *my_bars = bars + warp * S;

    if (lane == 0)
        for (int s = 0; s < S; ++s) mbar_init(&my_bars[s], 1);
    fence_mbar_init();
    __syncthreads();

    const uint8_t *my_src = p.w + static_cast<size_t>(row_ok ? row : 0) * rowbytes;
    auto issue = [&](int i) {  // chunk i of this CTA's K range into stage i % S
        const int st = i % S;
        if (lane == 0) mbar_arrive_expect_tx(&my_bars[st], valid_rows * CB);
        __syncwarp();
        if (row_ok)
            bulk_g2s(my_ring + (st * kRowsPerCta + lane) * CB,
                     my_src + static_cast<size_t>(c_begin + i) * CB, CB, &my_bars[st]);
    };
    // The weight prefetch may start before the preceding kernel in the stream
    // has finished (programmatic dependent launch): weights are read-only
    // model data that no kernel of this library writes.  Activations are read
    // and outputs written only after the wait below.
    int issued = 0;
    for (; issued < min(S, cpc); ++issued) issue(issued);
    pdl_wait();
    pdl_launch_dependents();

    float tot[M];
#pragma unroll
    for (int m = 0; m < M; ++m) tot[m] = 0.0f;

    bool failed = false;
    int consumed = 0;
    for (int s0 = 0; s0 < cpc; s0 += p.xs_chunks) {
        const int s1 = min(cpc, s0 + p.xs_chunks);
        if (s0 > 0) __syncthreads();  // the previous slice is no longer read
        {
            const int kx0 = (c_begin + s0) * kChunkK;
            const int nk4 = (s1 - s0) * (kChunkK / 4);
            for (int e = threadIdx.x; e < M * nk4; e += nw * 32) {
                const int m = e / nk4;
                const int kk = (e - m * nk4) * 4;
                float4 v = __ldg(reinterpret_cast<const float4 *>(
                    p.x + static_cast<size_t>(m) * p.k + kx0 + kk));
                const int j = (kx0 + kk) & 31;
                if constexpr (F == Fmt::Q4_0) {
                    v.x *= __int_as_float((127 - q4_0_shift(j + 0)) << 23);
                    v.y *= __int_as_float((127 - q4_0_shift(j + 1)) << 23);
                    v.z *= __int_as_float((127 - q4_0_shift(j + 2)) << 23);
                    v.w *= __int_as_float((127 - q4_0_shift(j + 3)) << 23);
                } else {
                    v.y *= 0.00390625f;  // 2^-8 for odd positions
                    v.w *= 0.00390625f;
                }
                *reinterpret_cast<float4 *>(xs + m * XS + kk) = v;
            }
        }
        __syncthreads();
        for (int i = s0; i < s1; ++i) {
            if (valid_rows == 0 || failed) continue;  // warp-uniform
            const int st = i % S;
            const uint32_t par = static_cast<uint32_t>(i / S) & 1u;
            if (!mbar_wait(&my_bars[st], par, p.ctx)) {
                failed = true;
                continue;
            }
            ++consumed;
            const uint8_t *src = my_ring + (st * kRowsPerCta + lane) * CB;
            const float *xc = xs + (i - s0) * kChunkK;
            if constexpr (F == Fmt::Q4_0)
                q4_0_chunk<M>(src, xc, XS, tot);
            else
                q8_0_chunk<M>(src, xc, XS, tot);
            __syncwarp();
            if (issued < cpc) {
                fence_proxy_async_smem();
                issue(issued);
                ++issued;
            }
        }
    }
    if (failed) {
        // Let copies still in flight land before the CTA's shared memory is
        // released; each wait is again bounded.
        for (int j = consumed; j < issued; ++j)
            mbar_wait(&my_bars[j % S], static_cast<uint32_t>(j / S) & 1u, p.ctx);
    }

    if (ksplit == 1) {
        if (row_ok) {
#pragma unroll
            for (int m = 0; m < M; ++m) p.y[static_cast<size_t>(m) * p.n + row] = tot[m];
        }
        return;
    }
    // partial sums of the cluster's K ranges, added in rank order by rank 0
    float *my_part = part + warp * M * kRowsPerCta;
#pragma unroll
    for (int m = 0; m < M; ++m) my_part[m * kRowsPerCta + lane] = tot[m];
    cluster_sync();
    if (rank == 0 && row_ok) {
#pragma unroll
        for (int m = 0; m < M; ++m) {
            float s = tot[m];
            for (uint32_t q = 1; q < ksplit; ++q) s += ld_dsmem_f32(&my_part[m * kRowsPerCta + lane], q);
            p.y[static_cast<size_t>(m) * p.n + row] = s;
        }
    }
    cluster_sync();  // peers keep their shared memory until rank 0 has read it
}

// Byte-wise fallback: one warp per row, lanes over blocks.
template <Fmt F, int M>
__global__ void __launch_bounds__(128) gemv_bytewise_kernel(const uint8_t *__restrict__ w,
                                                           const float *__restrict__ x,
                                                           float *__restrict__ y, int64_t n,
                                                           int64_t k, LaunchCtx ctx) {
    constexpr int kBB = F == Fmt::Q4_0 ? kQ4_0Bytes : kQ8_0Bytes;
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (row >= n) return;
    const int64_t nb = k / kQK;
    float acc[M];
#pragma unroll
    for (int m = 0; m < M; ++m) acc[m] = 0.0f;
    for (int64_t b = lane; b < nb; b += 32) {
        const uint8_t *blk = w + (row * nb + b) * kBB;
        const float d = half_bits_to_float(__ldg(blk) | (static_cast<uint32_t>(__ldg(blk + 1)) << 8));
        float part[M];
#pragma unroll
        for (int m = 0; m < M; ++m) part[m] = 0.0f;
        for (int j = 0; j < kQK; ++j) {
            float wq;
            if constexpr (F == Fmt::Q4_0) {
                const int byte = __ldg(blk + 2 + (j & 15));
                wq = static_cast<float>((j < 16 ? (byte & 15) : (byte >> 4)) - 8);
            } else {
                wq = static_cast<float>(static_cast<int8_t>(__ldg(blk + 2 + j)));
            }
#pragma unroll
            for (int m = 0; m < M; ++m) part[m] = fmaf(wq, __ldg(x + m * k + b * kQK + j), part[m]);
        }
#pragma unroll
        for (int m = 0; m < M; ++m) acc[m] = fmaf(d, part[m], acc[m]);
    }
#pragma unroll
    for (int m = 0; m < M; ++m) {
        float v = acc[m];
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
        if (lane == 0) y[m * n + row] = v;
    }
}

// Launch shape.  Units are (32-row tile, K range) pairs; the K dimension is
// split over a cluster (ksplit CTAs) until there are enough units to give
// every SM several resident warps, and warps per CTA share one activation
// slice.  Rings hold only as many stages as a warp has chunks.
struct StreamShape {
    int ksplit, nw, stages, cpc, xs_chunks;
    size_t smem;
};

template <Fmt F, int M>
StreamShape stream_shape(int64_t n, int64_t k, int sms) {
    constexpr int CB = StreamFmt<F>::kChunkBytes;
    StreamShape sh;
    const int64_t tiles = (n + kRowsPerCta - 1) / kRowsPerCta;
    const int C = static_cast<int>(k / kChunkK);
    const int64_t want_units = 8LL * sms;  // about eight resident row tiles per SM
    sh.ksplit = 1;
    while (sh.ksplit < 8 && tiles * sh.ksplit < want_units && C % (2 * sh.ksplit) == 0)
        sh.ksplit *= 2;
    sh.cpc = C / sh.ksplit;
    // several warps per CTA when there are plenty of tiles (they share x')
    const int64_t units = tiles * sh.ksplit;
    sh.nw = 1;
    while (sh.nw < 4 && units / (2 * sh.nw) >= 2LL * sms) sh.nw *= 2;
    sh.stages = std::min(sh.cpc, F == Fmt::Q4_0 ? 4 : 3);
    const int xs_budget = 32 * 1024;
    sh.xs_chunks = std::max(1, std::min(sh.cpc, xs_budget / (M * kChunkK * 4)));
    sh.smem = static_cast<size_t>(sh.nw) * sh.stages * kRowsPerCta * CB +
              sizeof(float) * (static_cast<size_t>(M) * sh.xs_chunks * kChunkK +
                               static_cast<size_t>(sh.nw) * M * kRowsPerCta) +
              sizeof(uint64_t) * sh.nw * sh.stages;
    return sh;
}

template <Fmt F, int M>
cudaError_t launch_stream(const uint8_t *w, const float *x, float *y, int64_t n, int64_t k,
                          cudaStream_t stream, const LaunchCtx &ctx) {
    const StreamShape sh = stream_shape<F, M>(n, k, device_sm_count());
    const int64_t tiles = (n + kRowsPerCta - 1) / kRowsPerCta;
    const int64_t groups = (tiles + sh.nw - 1) / sh.nw;
    StreamParams p;
    p.w = w;
    p.x = x;
    p.y = y;
    p.n = static_cast<int>(n);
    p.k = static_cast<int>(k);
    p.stages = sh.stages;
    p.cpc = sh.cpc;
    p.xs_chunks = sh.xs_chunks;
    p.ctx = ctx;
    auto kern = gemv_stream_kernel<F, M>;
    static int smem_limits[kMaxDevices] = {0};  // this instantiation's own cache
    const cudaError_t e = ensure_smem(kern, sh.smem, true, smem_limits);
    if (e != cudaSuccess) return e;
    return launch_kernel(kern, dim3(static_cast<unsigned>(groups * sh.ksplit)), dim3(sh.nw * 32),
                         sh.smem, stream, static_cast<unsigned>(sh.ksplit), p);
}

template <Fmt F, int M>
cudaError_t launch_m(const uint8_t *w, const float *x, float *y, int64_t n, int64_t k,
                     cudaStream_t stream, const LaunchCtx &ctx) {
    const bool aligned = ((reinterpret_cast<uintptr_t>(w) | reinterpret_cast<uintptr_t>(x)) & 15) == 0;
    if (k % kChunkK == 0 && aligned && n <= (1LL << 30) && k <= (1LL << 24))
        return launch_stream<F, M>(w, x, y, n, k, stream, ctx);
    const unsigned grid = static_cast<unsigned>((n + 3) / 4);
    return launch_kernel(gemv_bytewise_kernel<F, M>, dim3(grid), dim3(128), 0, stream, 1, w, x, y,
                         n, k, ctx);
}

template <Fmt F>
cudaError_t launch_fmt(const uint8_t *w, const float *x, float *y, int m, int64_t n, int64_t k,
                       cudaStream_t s, const LaunchCtx &ctx) {
    switch (m) {
#define QMM_CASE(MM) \
    case MM: return launch_m<F, MM>(w, x, y, n, k, s, ctx);
        QMM_CASE(1) QMM_CASE(2) QMM_CASE(3) QMM_CASE(4) QMM_CASE(5) QMM_CASE(6) QMM_CASE(7)
        QMM_CASE(8) QMM_CASE(9) QMM_CASE(10) QMM_CASE(11) QMM_CASE(12) QMM_CASE(13)
        QMM_CASE(14) QMM_CASE(15) QMM_CASE(16)
#undef QMM_CASE
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace
}  // namespace qmm
