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
//  * Lane r of a warp owns row r of a 32-row tile; for small problems (and,
//    at M = 1, where it needs a smaller cluster split) two lanes share a row
//    (half a chunk each), and at M <= 10 a lane owns two rows, so that each
//    activation load feeds both.  K is cut into chunks
//    of 256 weights (8 blocks: 144 bytes of Q4_0, 272 of Q8_0), which keeps
//    every row chunk 16-byte aligned.  A tile's K range is split over kw
//    warps of a CTA (partial sums added through shared memory) and, for
//    small N, over a thread-block cluster of ksplit CTAs (partials pushed
//    into rank 0's activation slice with remote stores once every rank is
//    done reading activations, then added in rank order by all of rank 0's
//    threads).  No global scratch; the summation order is fixed.
//  * Q4_0 at M >= 11 (the FMA pipe, not the loads, bounds it): the row-pair
//    form, four rows per lane, two lanes per row, two rows per packed FMA and
//    the block scale folded into the weights (q4_0_chunk_rp).
//  * A warp streams its chunks through its own ring of shared-memory stages.
//  * One 2-D TMA load moves a warp's 32 rows x one chunk (4.6 KB Q4_0,
//    8.7 KB Q8_0) and an mbarrier with a byte count tracks the stage (many
//    small per-row bulk copies would be limited by the copy engine's
//    per-request rate).  Rows sit 144 (272) bytes apart in shared memory, so
//    the lanes' 16-byte reads hit distinct banks.
//  * The CTA's slice of the activations (M rows x its K range) is copied
//    into shared memory by bulk copies issued by one thread after the
//    programmatic-launch wait; warps wait on its mbarrier and read x as
//    warp-wide broadcasts.  Q4_0 warps request one weight stage before that
//    wait and the rest after the copy, so that it does not queue behind them.
//  * Decode without int->float conversions: OR-ing a nibble (or an offset
//    byte) at bit s into the mantissa of 2^23 gives m = 2^23 + v*2^s exactly;
//    one FMA m*2^-s - (2^23 + 8*2^s)*2^-s (Q4_0; +128 for Q8_0) leaves the
//    exact integer nibble-8 (or q).  Both that FMA and the product with x run
//    as packed f32x2 instructions, one chain per block, row and token.
//  * Per block: acc = sum_j (nibble_j - 8) * x_j in fp32, then y += d * acc.
//
// Persistent kernel (one large matrix, M <= 10): one CTA per SM over an equal
// run of whole tiles, the CTA's warps splitting its (tile, chunk) units
// evenly; see gemv_persist_kernel.
//
// Byte-wise kernel: any K % 32 == 0 and any alignment, and the shapes whose
// activation slice does not fit shared memory at any cluster split; a warp
// per row.
#pragma once

#include "qmm_internal.h"

#include <algorithm>

// Launch-shape knobs (defaults; a build may override them with -D).
#ifndef QMM_GEMV_WARPS_PER_SM
#define QMM_GEMV_WARPS_PER_SM 10  // target resident warps per SM (work units)
#endif
#ifndef QMM_GEMV_MAX_KSPLIT
#define QMM_GEMV_MAX_KSPLIT 8     // largest cluster along K
#endif
#ifndef QMM_GEMV_MAX_KW
#define QMM_GEMV_MAX_KW 8         // largest K split across the warps of a CTA
#endif
#ifndef QMM_GEMV_MIN_WARPS
#define QMM_GEMV_MIN_WARPS 8      // warps per CTA when tiles allow
#endif
#ifndef QMM_GEMV_STAGES
#define QMM_GEMV_STAGES 4         // ring depth per warp
#endif
#ifndef QMM_GEMV_L2_UNITS
#define QMM_GEMV_L2_UNITS 1024    // (32-row tile x chunk) units up to which 2 lanes share a row
#endif

#ifndef QMM_GEMV_R2_MAX_M
#define QMM_GEMV_R2_MAX_M 4       // largest M at which a lane owns two weight rows
#endif
#ifndef QMM_GEMV_R_WIDE_MAX_M
#define QMM_GEMV_R_WIDE_MAX_M 10  // above R2_MAX_M, two rows per lane up to this M, then one
#endif
#ifndef QMM_GEMV_R_SMALL
#define QMM_GEMV_R_SMALL 1        // rows per lane for the small (two lanes per row) case
#endif
#ifndef QMM_GEMV_RP_MIN_M
#define QMM_GEMV_RP_MIN_M 11      // Q4_0: smallest M that takes the row-pair form
#endif
#ifndef QMM_GEMV_RP_L
#define QMM_GEMV_RP_L 2           // row-pair form: lanes per row (each half of the qs words)
#endif
#ifndef QMM_GEMV_RP_R
#define QMM_GEMV_RP_R 4           // row-pair form: rows per lane (two pairs)
#endif
// Ring stages a warp requests before the dependency wait, per format; the
// rest follow the activation copy, which would otherwise queue behind them
// (Q4_0 262144 x 2048: the copy's wait went from 4.9 us per CTA, and the
// launch from 98.5 to 90.4 us).  Q8_0 keeps its whole ring ahead: its LM
// head measured 10 % slower with one stage.
#ifndef QMM_GEMV_PREWAIT_Q4_0
#define QMM_GEMV_PREWAIT_Q4_0 1
#endif
#ifndef QMM_GEMV_PREWAIT_Q8_0
#define QMM_GEMV_PREWAIT_Q8_0 8
#endif
#ifndef QMM_GEMV_PERSIST
#define QMM_GEMV_PERSIST 1         // large single Q4_0 matrices at M <= 10: the persistent form
#endif
#ifndef QMM_GEMV_PERSIST_Q8_0
#define QMM_GEMV_PERSIST_Q8_0 1    // the same for Q8_0
#endif
#ifndef QMM_GEMV_PROXY_FENCE
#define QMM_GEMV_PROXY_FENCE 0    // 1: fence.proxy.async before refilling a stage (not needed)
#endif
#ifndef QMM_GEMV_X_BYTES
#define QMM_GEMV_X_BYTES 131072   // activation slice per CTA (shared memory)
#endif

namespace qmm {
namespace {

constexpr int kMaxGemvProblems = 4;
#ifndef QMM_GEMV_SMEM_CAP
#define QMM_GEMV_SMEM_CAP (224 * 1024)  // below the 227 KB per-CTA limit
#endif
constexpr size_t kGemvSmemCap = QMM_GEMV_SMEM_CAP;  // dynamic shared memory per CTA
// launch_stream's "no launch shape fits" answer (the caller falls back)
constexpr cudaError_t kShapeTooLarge = cudaErrorInvalidConfiguration;

static_assert((QMM_GEMV_MAX_KW & (QMM_GEMV_MAX_KW - 1)) == 0 &&
                  (QMM_GEMV_MAX_KSPLIT & (QMM_GEMV_MAX_KSPLIT - 1)) == 0,
              "K parts per CTA and per cluster are powers of two (the kernel shifts by them)");

constexpr int kChunkK = 256;
constexpr int kRpMaxProducts = 1024;  // row-pair form: products summed in one fp32 accumulator
constexpr uint32_t kMagic = 0x4B000000u;  // 2^23

// TMA view of the weight bytes: Q4_0 as uint8 (box 144 x 32), Q8_0 as
// uint16 pairs (box 136 x 32; a box row may hold at most 256 elements).
template <Fmt F>
struct StreamFmt;
template <>
struct StreamFmt<Fmt::Q4_0> {
    static constexpr int kChunkBytes = 144;
    static constexpr int kElemBytes = 1;
    static constexpr CUtensorMapDataType kType = CU_TENSOR_MAP_DATA_TYPE_UINT8;
};
template <>
struct StreamFmt<Fmt::Q8_0> {
    static constexpr int kChunkBytes = 272;
    static constexpr int kElemBytes = 2;
    static constexpr CUtensorMapDataType kType = CU_TENSOR_MAP_DATA_TYPE_UINT16;
};

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, "
        "{%2, %3}], [%4];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

// m = 2^23 + (v & mask) as a float: the nibble (byte) lands in the mantissa.
// `magic` is 2^23's bit pattern, passed in at run time: with the mask and the
// magic both compile-time immediates the compiler emits two LOP3 per
// extraction (a SASS LOP3 takes one immediate); with the magic in a register
// it is one.
#ifndef QMM_MAGIC_PARAM
#define QMM_MAGIC_PARAM 1
#endif
__device__ __forceinline__ float mag(uint32_t v, uint32_t mask, uint32_t magic) {
#if QMM_MAGIC_PARAM
    return __uint_as_float((v & mask) | magic);
#else
    (void)magic;
    return __uint_as_float((v & mask) | kMagic);
#endif
}
// Q8_0 byte with its sign bit flipped (q + 128) in the mantissa of 2^23;
// magic_flip = 2^23's pattern with the byte's top bit set.
__device__ __forceinline__ float mag8(uint32_t v, uint32_t mask, uint32_t magic_flip) {
    return __uint_as_float((mask & (v ^ magic_flip)) | (~mask & magic_flip));
}

__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }

// Loads this lane's share of a row chunk: `words` 32-bit words from a
// portion aligned to 16, 8 or 4 bytes (one, two or four lanes per row).
template <int L, int WORDS>
__device__ __forceinline__ void load_portion(const uint8_t *src, uint32_t (&wd)[WORDS]) {
    if constexpr (L == 1) {
#pragma unroll
        for (int t = 0; t < WORDS / 4; ++t) {
            const uint4 v = lds128(src + 16 * t);
            wd[4 * t + 0] = v.x;
            wd[4 * t + 1] = v.y;
            wd[4 * t + 2] = v.z;
            wd[4 * t + 3] = v.w;
        }
    } else if constexpr (L == 2) {
#pragma unroll
        for (int t = 0; t < WORDS / 2; ++t) {
            const uint2 v = *reinterpret_cast<const uint2 *>(src + 8 * t);
            wd[2 * t + 0] = v.x;
            wd[2 * t + 1] = v.y;
        }
    } else {
#pragma unroll
        for (int t = 0; t < WORDS; ++t) wd[t] = *reinterpret_cast<const uint32_t *>(src + 4 * t);
    }
}

// R rows' shares (8/L consecutive Q4_0 blocks, 144/L bytes each; row j at
// src + j*rstride) of a row chunk, against activations `xk` in shared memory
// (position 0 of the share for activation row 0; rows XS apart).  Each
// activation value is loaded once and used for all R weight rows.
//
// A qs word v holds weights 4i..4i+3 (low nibbles, bits 0,8,16,24) and
// 16+4i..19+4i (high nibbles, bits 4,12,20,28); bits 0-19 are used in place
// and bits 20-31 after u = v >> 16, so the nibble sits at s in {0,4,8,12,16}.
//
// Each block's sum runs as one packed FMA chain per row and token: splitting
// it into 2-4 independent chains (as at first, for latency) measured slower
// once the kernels were issue-bound (decode step 18.64 -> 18.03 us, Q8_0 LM
// head 97.3 -> 93.0 us, M = 2 at 8192 x 2048 5.12 -> 4.76 us with one chain):
// merging the chains cost more instructions than their overlap hid.
template <int M, int L, int R>
__device__ __forceinline__ void q4_0_chunk(const uint8_t *src, int rstride, const float *xk,
                                           int XS, uint32_t magic, float (&tot)[R][M]) {
    constexpr int NB = 8 / L;
    uint32_t wd[R][36 / L];
#pragma unroll
    for (int j = 0; j < R; ++j) load_portion<L>(src + j * rstride, wd[j]);
    // (m - (2^23 + 8*2^s)) * 2^-s = m*2^-s - (2^23*2^-s + 8): exact nibble-8
    const float2 s01 = f2(1.0f, 0.00390625f), b01 = f2(-8388616.0f, -32776.0f);           // s = 0, 8
    const float2 s23 = f2(1.52587890625e-05f, 0.00390625f), b23 = f2(-136.0f, -32776.0f); // s = 16, 8
    const float2 s45 = f2(0.0625f, 0.000244140625f), b45 = f2(-524296.0f, -2056.0f);      // s = 4, 12
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        const int base = (18 * b) >> 2;
        uint32_t q[R][4];
        float d[R];
#pragma unroll
        for (int j = 0; j < R; ++j) {
            uint32_t dbits;
            if ((b & 1) == 0) {  // block starts on a word: d low half, qs shifted by 2 bytes
                dbits = wd[j][base] & 0xFFFFu;
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    q[j][i] = __byte_perm(wd[j][base + i], wd[j][base + i + 1], 0x5432);
            } else {  // block starts 2 bytes into a word: d high half, qs aligned
                dbits = wd[j][base] >> 16;
#pragma unroll
                for (int i = 0; i < 4; ++i) q[j][i] = wd[j][base + 1 + i];
            }
            d[j] = half_bits_to_float(dbits);
        }
        float2 acc[R][M];
#pragma unroll
        for (int j = 0; j < R; ++j)
#pragma unroll
            for (int m = 0; m < M; ++m) acc[j][m] = f2(0.0f, 0.0f);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float4 xa[M], xb[M];
#pragma unroll
            for (int m = 0; m < M; ++m) {
                xa[m] = lds128f(xk + m * XS + 32 * b + 4 * i);
                xb[m] = lds128f(xk + m * XS + 32 * b + 16 + 4 * i);
            }
#pragma unroll
            for (int j = 0; j < R; ++j) {
                const uint32_t v = q[j][i], u = v >> 16;
                const float2 p01 = __ffma2_rn(f2(mag(v, 0x0000000Fu, magic), mag(v, 0x00000F00u, magic)), s01, b01);
                const float2 p23 = __ffma2_rn(f2(mag(v, 0x000F0000u, magic), mag(u, 0x00000F00u, magic)), s23, b23);
                const float2 p45 = __ffma2_rn(f2(mag(v, 0x000000F0u, magic), mag(v, 0x0000F000u, magic)), s45, b45);
                const float2 p67 = __ffma2_rn(f2(mag(u, 0x000000F0u, magic), mag(u, 0x0000F000u, magic)), s45, b45);
#pragma unroll
                for (int m = 0; m < M; ++m) {
                    acc[j][m] = __ffma2_rn(p01, f2(xa[m].x, xa[m].y), acc[j][m]);
                    acc[j][m] = __ffma2_rn(p23, f2(xa[m].z, xa[m].w), acc[j][m]);
                    acc[j][m] = __ffma2_rn(p45, f2(xb[m].x, xb[m].y), acc[j][m]);
                    acc[j][m] = __ffma2_rn(p67, f2(xb[m].z, xb[m].w), acc[j][m]);
                }
            }
        }
#pragma unroll
        for (int j = 0; j < R; ++j)
#pragma unroll
            for (int m = 0; m < M; ++m) tot[j][m] = fmaf(d[j], acc[j][m].x + acc[j][m].y, tot[j][m]);
    }
}

// R rows' shares (8/L consecutive Q8_0 blocks, 272/L bytes each) of a row
// chunk.  Bytes 0 and 2 of a word are used at bits 0-7 (s = 0), bytes 1 and
// 3 at bits 8-15 (s = 8).  One FMA chain per block, row and token, as in
// q4_0_chunk.
template <int M, int L, int R>
__device__ __forceinline__ void q8_0_chunk(const uint8_t *src, int rstride, const float *xk,
                                           int XS, uint32_t magic, float (&tot)[R][M]) {
    constexpr int NB = 8 / L;
    uint32_t wd[R][68 / L];
#pragma unroll
    for (int j = 0; j < R; ++j) load_portion<L>(src + j * rstride, wd[j]);
    // (m - (2^23 + 128*2^s)) * 2^-s: exact q
    const float2 sc = f2(1.0f, 0.00390625f), bc = f2(-8388736.0f, -32896.0f);
    // compile-time constants here: for the byte path the compiler's own
    // immediate form measured faster than a register operand
    (void)magic;
    constexpr uint32_t mf0 = kMagic | 0x80u, mf1 = kMagic | 0x8000u;
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        const int base = (34 * b) >> 2;
        float d[R];
#pragma unroll
        for (int j = 0; j < R; ++j)
            d[j] = half_bits_to_float((b & 1) == 0 ? (wd[j][base] & 0xFFFFu) : (wd[j][base] >> 16));
        float2 acc[R][M];
#pragma unroll
        for (int j = 0; j < R; ++j)
#pragma unroll
            for (int m = 0; m < M; ++m) acc[j][m] = f2(0.0f, 0.0f);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float4 xa[M];
#pragma unroll
            for (int m = 0; m < M; ++m) xa[m] = lds128f(xk + m * XS + 32 * b + 4 * i);
#pragma unroll
            for (int j = 0; j < R; ++j) {
                const uint32_t v = (b & 1) == 0 ? __byte_perm(wd[j][base + i], wd[j][base + i + 1], 0x5432)
                                                : wd[j][base + 1 + i];
                const uint32_t u = v >> 16;
                const float2 p01 = __ffma2_rn(
                    f2(mag8(v, 0x000000FFu, mf0), mag8(v, 0x0000FF00u, mf1)), sc, bc);
                const float2 p23 = __ffma2_rn(
                    f2(mag8(u, 0x000000FFu, mf0), mag8(u, 0x0000FF00u, mf1)), sc, bc);
#pragma unroll
                for (int m = 0; m < M; ++m) {
                    acc[j][m] = __ffma2_rn(p01, f2(xa[m].x, xa[m].y), acc[j][m]);
                    acc[j][m] = __ffma2_rn(p23, f2(xa[m].z, xa[m].w), acc[j][m]);
                }
            }
        }
#pragma unroll
        for (int j = 0; j < R; ++j)
#pragma unroll
            for (int m = 0; m < M; ++m) tot[j][m] = fmaf(d[j], acc[j][m].x + acc[j][m].y, tot[j][m]);
    }
}


// Wide-M forms (one lane per row, one row per lane): a runtime loop over
// block pairs, each pair's 36 (Q4_0) or 68 (Q8_0) bytes read from shared
// memory as words.  The arithmetic is that of q4_0_chunk / q8_0_chunk; the
// loop keeps the code (and build time) small where FMAs, not loads, bound
// the kernel.
template <int M, int R>
__device__ __forceinline__ void q4_0_chunk_wide(const uint8_t *src, int rstride, const float *xk,
                                                int XS, uint32_t magic, float (&tot)[R][M]) {
    const float2 s01 = f2(1.0f, 0.00390625f), b01 = f2(-8388616.0f, -32776.0f);
    const float2 s23 = f2(1.52587890625e-05f, 0.00390625f), b23 = f2(-136.0f, -32776.0f);
    const float2 s45 = f2(0.0625f, 0.000244140625f), b45 = f2(-524296.0f, -2056.0f);
#pragma unroll 1
    for (int bp = 0; bp < 4; ++bp) {
        uint32_t wd[R][9];
#pragma unroll
        for (int j = 0; j < R; ++j)
#pragma unroll
            for (int t = 0; t < 9; ++t)
                wd[j][t] = *reinterpret_cast<const uint32_t *>(src + j * rstride + 36 * bp + 4 * t);
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
            const int b = 2 * bp + hb;
            uint32_t q[R][4];
            float d[R];
#pragma unroll
            for (int j = 0; j < R; ++j) {
                uint32_t dbits;
                if (hb == 0) {
                    dbits = wd[j][0] & 0xFFFFu;
#pragma unroll
                    for (int i = 0; i < 4; ++i) q[j][i] = __byte_perm(wd[j][i], wd[j][i + 1], 0x5432);
                } else {
                    dbits = wd[j][4] >> 16;
#pragma unroll
                    for (int i = 0; i < 4; ++i) q[j][i] = wd[j][5 + i];
                }
                d[j] = half_bits_to_float(dbits);
            }
            float2 acc[R][M];
#pragma unroll
            for (int j = 0; j < R; ++j)
#pragma unroll
                for (int m = 0; m < M; ++m) acc[j][m] = f2(0.0f, 0.0f);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float2 p01[R], p23[R], p45[R], p67[R];
#pragma unroll
                for (int j = 0; j < R; ++j) {
                    const uint32_t v = q[j][i], u = v >> 16;
                    p01[j] = __ffma2_rn(f2(mag(v, 0x0000000Fu, magic), mag(v, 0x00000F00u, magic)), s01, b01);
                    p23[j] = __ffma2_rn(f2(mag(v, 0x000F0000u, magic), mag(u, 0x00000F00u, magic)), s23, b23);
                    p45[j] = __ffma2_rn(f2(mag(v, 0x000000F0u, magic), mag(v, 0x0000F000u, magic)), s45, b45);
                    p67[j] = __ffma2_rn(f2(mag(u, 0x000000F0u, magic), mag(u, 0x0000F000u, magic)), s45, b45);
                }
#pragma unroll
                for (int m = 0; m < M; ++m) {
                    // each activation load feeds all R rows
                    const float4 xa = lds128f(xk + m * XS + 32 * b + 4 * i);
                    const float4 xb = lds128f(xk + m * XS + 32 * b + 16 + 4 * i);
#pragma unroll
                    for (int j = 0; j < R; ++j) {
                        acc[j][m] = __ffma2_rn(p01[j], f2(xa.x, xa.y), acc[j][m]);
                        acc[j][m] = __ffma2_rn(p23[j], f2(xa.z, xa.w), acc[j][m]);
                        acc[j][m] = __ffma2_rn(p45[j], f2(xb.x, xb.y), acc[j][m]);
                        acc[j][m] = __ffma2_rn(p67[j], f2(xb.z, xb.w), acc[j][m]);
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < R; ++j)
#pragma unroll
                for (int m = 0; m < M; ++m) tot[j][m] = fmaf(d[j], acc[j][m].x + acc[j][m].y, tot[j][m]);
        }
    }
}

template <int M, int R>
__device__ __forceinline__ void q8_0_chunk_wide(const uint8_t *src, int rstride, const float *xk,
                                                int XS, uint32_t magic, float (&tot)[R][M]) {
    const float2 sc = f2(1.0f, 0.00390625f), bc = f2(-8388736.0f, -32896.0f);
    // compile-time constants here: for the byte path the compiler's own
    // immediate form measured faster than a register operand
    (void)magic;
    constexpr uint32_t mf0 = kMagic | 0x80u, mf1 = kMagic | 0x8000u;
#pragma unroll 1
    for (int bp = 0; bp < 4; ++bp) {
        uint32_t wd[R][17];
#pragma unroll
        for (int j = 0; j < R; ++j)
#pragma unroll
            for (int t = 0; t < 17; ++t)
                wd[j][t] = *reinterpret_cast<const uint32_t *>(src + j * rstride + 68 * bp + 4 * t);
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
            const int b = 2 * bp + hb;
            float d[R];
#pragma unroll
            for (int j = 0; j < R; ++j)
                d[j] = half_bits_to_float(hb == 0 ? (wd[j][0] & 0xFFFFu) : (wd[j][8] >> 16));
            float2 acc[R][M];
#pragma unroll
            for (int j = 0; j < R; ++j)
#pragma unroll
                for (int m = 0; m < M; ++m) acc[j][m] = f2(0.0f, 0.0f);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float2 p01[R], p23[R];
#pragma unroll
                for (int j = 0; j < R; ++j) {
                    const uint32_t v = hb == 0 ? __byte_perm(wd[j][i], wd[j][i + 1], 0x5432) : wd[j][9 + i];
                    const uint32_t u = v >> 16;
                    p01[j] = __ffma2_rn(f2(mag8(v, 0x000000FFu, mf0), mag8(v, 0x0000FF00u, mf1)), sc, bc);
                    p23[j] = __ffma2_rn(f2(mag8(u, 0x000000FFu, mf0), mag8(u, 0x0000FF00u, mf1)), sc, bc);
                }
#pragma unroll
                for (int m = 0; m < M; ++m) {
                    const float4 xa = lds128f(xk + m * XS + 32 * b + 4 * i);
#pragma unroll
                    for (int j = 0; j < R; ++j) {
                        acc[j][m] = __ffma2_rn(p01[j], f2(xa.x, xa.y), acc[j][m]);
                        acc[j][m] = __ffma2_rn(p23[j], f2(xa.z, xa.w), acc[j][m]);
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < R; ++j)
#pragma unroll
                for (int m = 0; m < M; ++m) tot[j][m] = fmaf(d[j], acc[j][m].x + acc[j][m].y, tot[j][m]);
        }
    }
}

// Row-pair form for wide M (Q4_0; the FMA pipe, not the loads, bounds it).
// A packed FMA carries two weight rows of one activation value,
//   acc[p][m] += (w[2p][k], w[2p+1][k]) * (x[m][k], x[m][k]),
// so each activation read from shared memory feeds R rows and the
// accumulators take R*M registers (the k-pair form above needs 2*R*M for the
// same reuse).  The block scale is folded into the weights: (nibble-8)*d is
// exact in fp32 (a 4-bit integer times an 11-bit significand), so acc is a
// plain fp32 sum of the products w*x over the lane's share of K.
//
// Lane h of the L lanes of a row decodes qs words i = h, h+L, ... of every
// block of the chunk.  The L lanes then read activations 4i..4i+3 and
// 16+4i..19+4i: distinct banks, so one shared-memory pass serves all of them.
// `row` is the row's chunk in shared memory (rows rstride bytes apart).
template <int M, int L, int R>
__device__ __forceinline__ void q4_0_chunk_rp(const uint8_t *row, int rstride, const float *xk,
                                              int XS, int h, uint32_t magic,
                                              float2 (&acc)[R / 2][M]) {
    static_assert(R % 2 == 0 && 4 % L == 0, "rows come in pairs; L divides the 4 qs words");
    constexpr int NW = 4 / L;
    // m * 2^-s - (2^(23-s) + 8) turns 2^23's float with nibble v at bit s
    // into v - 8, exactly
    const float2 S0 = f2(1.0f, 1.0f), B0 = f2(-8388616.0f, -8388616.0f);
    const float2 S4 = f2(0.0625f, 0.0625f), B4 = f2(-524296.0f, -524296.0f);
    const float2 S8 = f2(0.00390625f, 0.00390625f), B8 = f2(-32776.0f, -32776.0f);
    const float2 S12 = f2(0.000244140625f, 0.000244140625f), B12 = f2(-2056.0f, -2056.0f);
    const float2 S16 = f2(1.52587890625e-05f, 1.52587890625e-05f), B16 = f2(-136.0f, -136.0f);
#pragma unroll 1
    for (int bp = 0; bp < 4; ++bp) {  // block pairs: 36 bytes, 4-byte aligned
        const uint8_t *pb = row + 36 * bp;
        float2 dd[2][R / 2];  // (d of row 2p, d of row 2p+1) for the pair's two blocks
#pragma unroll
        for (int p = 0; p < R / 2; ++p) {
            const uint8_t *r0 = pb + 2 * p * rstride, *r1 = r0 + rstride;
            const uint32_t a0 = *reinterpret_cast<const uint32_t *>(r0);
            const uint32_t a1 = *reinterpret_cast<const uint32_t *>(r1);
            const uint32_t c0 = *reinterpret_cast<const uint32_t *>(r0 + 16);
            const uint32_t c1 = *reinterpret_cast<const uint32_t *>(r1 + 16);
            dd[0][p] = f2(half_bits_to_float(a0 & 0xFFFFu), half_bits_to_float(a1 & 0xFFFFu));
            dd[1][p] = f2(half_bits_to_float(c0 >> 16), half_bits_to_float(c1 >> 16));
        }
#pragma unroll 1
        for (int wi = 0; wi < NW; ++wi) {
            const int i = h + L * wi;  // qs word of each block
            const uint8_t *pw = pb + 4 * i;
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {
                const int b = 2 * bp + hb;
                float2 w[R / 2][8];  // weights 4i..4i+3 and 16+4i..19+4i of both rows
#pragma unroll
                for (int p = 0; p < R / 2; ++p) {
                    const uint8_t *q0 = pw + 2 * p * rstride, *q1 = q0 + rstride;
                    uint32_t v0, v1;
                    if (hb == 0) {  // even block: qs starts 2 bytes into a word
                        v0 = __byte_perm(*reinterpret_cast<const uint32_t *>(q0),
                                         *reinterpret_cast<const uint32_t *>(q0 + 4), 0x5432);
                        v1 = __byte_perm(*reinterpret_cast<const uint32_t *>(q1),
                                         *reinterpret_cast<const uint32_t *>(q1 + 4), 0x5432);
                    } else {
                        v0 = *reinterpret_cast<const uint32_t *>(q0 + 20);
                        v1 = *reinterpret_cast<const uint32_t *>(q1 + 20);
                    }
                    const uint32_t u0 = v0 >> 16, u1 = v1 >> 16;
                    const float2 d = dd[hb][p];
                    w[p][0] = __fmul2_rn(__ffma2_rn(f2(mag(v0, 0x0000000Fu, magic), mag(v1, 0x0000000Fu, magic)), S0, B0), d);
                    w[p][1] = __fmul2_rn(__ffma2_rn(f2(mag(v0, 0x00000F00u, magic), mag(v1, 0x00000F00u, magic)), S8, B8), d);
                    w[p][2] = __fmul2_rn(__ffma2_rn(f2(mag(v0, 0x000F0000u, magic), mag(v1, 0x000F0000u, magic)), S16, B16), d);
                    w[p][3] = __fmul2_rn(__ffma2_rn(f2(mag(u0, 0x00000F00u, magic), mag(u1, 0x00000F00u, magic)), S8, B8), d);
                    w[p][4] = __fmul2_rn(__ffma2_rn(f2(mag(v0, 0x000000F0u, magic), mag(v1, 0x000000F0u, magic)), S4, B4), d);
                    w[p][5] = __fmul2_rn(__ffma2_rn(f2(mag(v0, 0x0000F000u, magic), mag(v1, 0x0000F000u, magic)), S12, B12), d);
                    w[p][6] = __fmul2_rn(__ffma2_rn(f2(mag(u0, 0x000000F0u, magic), mag(u1, 0x000000F0u, magic)), S4, B4), d);
                    w[p][7] = __fmul2_rn(__ffma2_rn(f2(mag(u0, 0x0000F000u, magic), mag(u1, 0x0000F000u, magic)), S12, B12), d);
                }
#pragma unroll
                for (int m = 0; m < M; ++m) {
                    const float4 xa = lds128f(xk + m * XS + 32 * b + 4 * i);
                    const float4 xb = lds128f(xk + m * XS + 32 * b + 16 + 4 * i);
                    const float xv[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
                    for (int p = 0; p < R / 2; ++p)
#pragma unroll
                        for (int t = 0; t < 8; ++t)
                            acc[p][m] = __ffma2_rn(w[p][t], f2(xv[t], xv[t]), acc[p][m]);
                }
            }
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
// The two halves of cluster_sync, for work in between.
__device__ __forceinline__ void gemv_cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void gemv_cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void st_dsmem_f32(const float *local, uint32_t rank, float v) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                 : "=r"(remote)
                 : "r"(smem_addr(local)), "r"(rank));
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}

// Up to kMaxGemvProblems weight matrices that share the activations x (and
// K), e.g. the q/k/v or gate/up projections of a decode layer, in one launch.
struct StreamMaps {
    CUtensorMap m[kMaxGemvProblems];
};

struct StreamParams {
    const float *x;
    float *y[kMaxGemvProblems];
    int n[kMaxGemvProblems];                  // rows of each W
    int group_begin[kMaxGemvProblems + 1];    // first CTA group of each problem
    int count;                                // problems
    int k;            // columns (multiple of 256)
    int rw;           // row tiles per CTA
    int kw;           // warps sharing one row tile (K split inside the CTA)
    int cpw;          // chunks per warp
    int stages;       // ring depth per warp
    uint32_t magic;   // 0x4B000000 (2^23), kept in a register by the kernel
    LaunchCtx ctx;
};

// GeGLU feed-forward input h = gelu(g) * u, g = x.Wg^T, u = x.Wu^T (the
// tanh form of the GELU, evaluated as z * sigmoid(2a) with
// a = sqrt(2/pi) * (z + 0.044715 z^3), which equals z/2 * (1 + tanh(a))
// and has no cancellation for negative z).
__device__ __forceinline__ float gelu_tanh(float z) {
    const float a = 0.7978845608028654f * fmaf(0.044715f * z, z * z, z);
    return z / (1.0f + expf(-2.0f * a));
}

// Grid: blockIdx.x = group * ksplit + rank (cluster of ksplit CTAs along x).
// Warp w of a CTA owns row tile group*rw + w / kw and the (w % kw)-th part of
// the CTA's K range; cluster rank r owns the r-th part of K.
//
// G (GeGLU): one problem whose gate and up weights are maps.m[0] and
// maps.m[1].  A lane's two rows (R == 2) are gate row and up row of the same
// output: a stage holds the gate box (32/L rows) followed by the up box, the
// lane's two sums meet in registers and the writer stores gelu(g) * u.
#ifndef QMM_GEMV_MAX_THREADS
#define QMM_GEMV_MAX_THREADS 256
#endif
// Register budget hint (CTAs of QMM_GEMV_MAX_THREADS per SM that it must
// allow).  Without one, ptxas kept the M <= 4 kernels near 80 registers;
// allowing two CTAs' worth (up to 128) took the decode step from 19.0 to
// 18.05 us.  The row-pair form needs more than 128 and the per-block forms of
// M 5..9 measured 1-2 % faster with more: both get one CTA's worth.
#ifndef QMM_GEMV_MB_L1
#define QMM_GEMV_MB_L1 2
#endif
#ifndef QMM_GEMV_MB_L2
#define QMM_GEMV_MB_L2 2
#endif
#ifndef QMM_GEMV_MB_WIDE
#define QMM_GEMV_MB_WIDE 1
#endif
template <int M, int L, bool RP>
struct StreamMinBlocks {
    static constexpr int value =
        RP ? 1 : (M <= QMM_GEMV_R2_MAX_M ? (L == 1 ? QMM_GEMV_MB_L1 : QMM_GEMV_MB_L2) : QMM_GEMV_MB_WIDE);
};
template <Fmt F, int M, int L, int R, bool G = false, bool RP = false>
__global__ void __launch_bounds__(QMM_GEMV_MAX_THREADS, (StreamMinBlocks<M, L, RP>::value))
    gemv_stream_kernel(const __grid_constant__ StreamMaps maps, StreamParams p) {
    static_assert(!G || R == 2, "GeGLU pairs the gate and up rows of one output in a lane");
    static_assert(!RP || (F == Fmt::Q4_0 && !G && R % 2 == 0), "row-pair form: Q4_0 row pairs");
    constexpr int CB = StreamFmt<F>::kChunkBytes;
    constexpr int kLaneRows = 32 / L;                 // rows covered by one pass of the lanes
    constexpr int kRowsPerWarp = kLaneRows * R;       // L lanes share a row; a lane owns R rows
    constexpr int kTileRows = G ? kLaneRows : kRowsPerWarp;  // output rows of a warp's tile
    extern __shared__ __align__(128) uint8_t smem_dyn[];
    // TMA destinations: 128-byte aligned (the launch adds 128 bytes of slack)
    uint8_t *smem = smem_dyn + ((128u - (smem_addr(smem_dyn) & 127u)) & 127u);
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nw = blockDim.x >> 5;
    const int S = p.stages;
    const int kw = p.kw, cpw = p.cpw;
    const uint32_t rank = cluster_ctarank();
    const uint32_t ksplit = cluster_nctarank();
    // kw and ksplit are powers of two: shifts instead of run-time divisions
    const int gg = static_cast<int>(blockIdx.x >> (__ffs(static_cast<int>(ksplit)) - 1));  // CTA group
    // this CTA's problem, picked with unrolled selects (indexing the
    // parameter arrays with a run-time index would copy them to local memory)
    int prob = 0, gbegin = p.group_begin[0], n_rows = p.n[0];
    float *y = p.y[0];
#pragma unroll
    for (int i = 1; i < kMaxGemvProblems; ++i) {
        if (i < p.count && gg >= p.group_begin[i]) {
            prob = i;
            gbegin = p.group_begin[i];
            n_rows = p.n[i];
            y = p.y[i];
        }
    }
    const int group = gg - gbegin;
    const CUtensorMap *wmap = &maps.m[prob];
    const int tile_in_cta = warp >> (__ffs(kw) - 1);
    const int kpart = warp & (kw - 1);
    const int row0 = (group * p.rw + tile_in_cta) * kTileRows;
    const int r = lane / L;  // rows r, r + 32/L, ... of the warp's tile
    const int h = lane % L;  // this lane's share of each chunk
    const bool warp_active = row0 < n_rows;  // warp-uniform
    const int cta_chunks = kw * cpw;
    const int cta_c0 = static_cast<int>(rank) * cta_chunks;  // first chunk of the CTA
    const int w_c0 = kpart * cpw;                            // first chunk of the warp, CTA-relative
    const int XS = cta_chunks * kChunkK;  // activation floats per row in shared memory

    // shared memory: ring [nw][S][rows][CB] | xs [M][XS] | (part) | bars [nw][S] | xbar
    // A warp's K-part sums for the in-CTA reduction ([M][rows] floats) go to
    // the start of its own ring once its last stage has been read.  The
    // cluster's K-part sums, part [ksplit][rw][M][rows] (rank 0 only), reuse
    // the activation slice when they fit in it (all ranks are done reading
    // activations by then), else follow it.
    static_assert(4 * M <= CB, "a warp's partial sums fit one ring stage");
    const size_t ring_bytes = static_cast<size_t>(S) * kRowsPerWarp * CB;  // per warp
    uint8_t *my_ring = smem + warp * ring_bytes;
    auto red_of = [&](int w_) { return reinterpret_cast<float *>(smem + w_ * ring_bytes); };
    float *xs = reinterpret_cast<float *>(smem + nw * ring_bytes);
    const int part_floats = static_cast<int>(ksplit) * p.rw * M * kRowsPerWarp;
    const bool part_in_xs = part_floats <= M * XS;
    float *part = part_in_xs ? xs : xs + M * XS;
    uint64_t *bars = reinterpret_cast<uint64_t *>(xs + M * XS + (part_in_xs ? 0 : part_floats));
    uint64_t *my_bars = bars + warp * S;
    uint64_t *xbar = bars + nw * S;

    if (lane == 0) {
        if (warp == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(wmap)) : "memory");
            if constexpr (G)
                asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&maps.m[1]))
                             : "memory");
            mbar_init(xbar, 1);
        }
        for (int s = 0; s < S; ++s) mbar_init(&my_bars[s], 1);
        fence_mbar_init();
    }
    __syncthreads();  // barriers initialised before any thread waits on them

    auto issue = [&](int st, int i) {  // chunk i of this warp into stage st (= i % S)
        if (lane == 0) {
            // full box bytes: rows past N are zero-filled and still counted
            mbar_arrive_expect_tx(&my_bars[st], kRowsPerWarp * CB);
            const int cx = (cta_c0 + w_c0 + i) * (CB / StreamFmt<F>::kElemBytes);
            tma_load_2d(my_ring + st * kRowsPerWarp * CB, wmap, cx, row0, &my_bars[st]);
            if constexpr (G)  // the up rows of the same outputs, after the gate box
                tma_load_2d(my_ring + (st * kRowsPerWarp + kLaneRows) * CB, &maps.m[1], cx, row0,
                            &my_bars[st]);
        }
    };
    // The weight prefetch may start before the preceding kernel in the stream
    // has finished (programmatic dependent launch): weights are read-only
    // model data that no kernel of this library writes.  Activations are read
    // and outputs written only after the wait below.
    constexpr int kPrewait = F == Fmt::Q4_0 ? QMM_GEMV_PREWAIT_Q4_0 : QMM_GEMV_PREWAIT_Q8_0;
    int issued = 0;
    if (warp_active)
        for (; issued < min(min(S, cpw), kPrewait); ++issued) issue(issued, issued);
    pdl_wait();
    if (threadIdx.x == 0) {  // activations: one bulk copy per row m of the CTA's K range
        mbar_arrive_expect_tx(xbar, static_cast<uint32_t>(M * XS * sizeof(float)));
#pragma unroll
        for (int m = 0; m < M; ++m)
            bulk_g2s(xs + m * XS, p.x + static_cast<size_t>(m) * p.k + cta_c0 * kChunkK,
                     static_cast<uint32_t>(XS * sizeof(float)), xbar);
    }
    pdl_launch_dependents();
    if (kPrewait < min(S, cpw)) {  // (the same in every warp) the rest of the ring, after the
        __syncthreads();           // activation copy
        if (warp_active)
            for (; issued < min(S, cpw); ++issued) issue(issued, issued);
    }

    float tot[R][M];
#pragma unroll
    for (int j = 0; j < R; ++j)
#pragma unroll
        for (int m = 0; m < M; ++m) tot[j][m] = 0.0f;
    float2 acc[RP ? R / 2 : 1][RP ? M : 1];  // row-pair sums (RP)
#pragma unroll
    for (int j = 0; j < (RP ? R / 2 : 1); ++j)
#pragma unroll
        for (int m = 0; m < (RP ? M : 1); ++m) acc[j][m] = f2(0.0f, 0.0f);

    int consumed = 0;
    // every warp waits for the activations (so none exits with the copy in flight)
    const bool x_ok = __all_sync(0xFFFFFFFFu, mbar_wait(xbar, 0, p.ctx));
    bool failed = !x_ok;
    if (warp_active) {
        int st = 0;         // i % S, kept incrementally (S is a run-time value)
        uint32_t par = 0;   // (i / S) & 1
        for (int i = 0; i < cpw && !failed; ++i) {
            // a lane's wait can give up while another's succeeds: the warp decides together
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&my_bars[st], par, p.ctx))) {
                failed = true;
                break;
            }
            ++consumed;
            const uint8_t *src = my_ring + (st * kRowsPerWarp + r) * CB + h * (CB / L);
            const float *xk = xs + (w_c0 + i) * kChunkK + h * (kChunkK / L);
            if constexpr (RP) {  // the lane picks its qs words itself: row and chunk starts
                q4_0_chunk_rp<M, L, R>(my_ring + (st * kRowsPerWarp + r) * CB, kLaneRows * CB,
                                       xs + (w_c0 + i) * kChunkK, XS, h, p.magic, acc);
            } else if constexpr (M > QMM_GEMV_R2_MAX_M && L == 1) {
                if constexpr (F == Fmt::Q4_0)
                    q4_0_chunk_wide<M, R>(src, kLaneRows * CB, xk, XS, p.magic, tot);
                else
                    q8_0_chunk_wide<M, R>(src, kLaneRows * CB, xk, XS, p.magic, tot);
            } else if constexpr (F == Fmt::Q4_0) {
                q4_0_chunk<M, L, R>(src, kLaneRows * CB, xk, XS, p.magic, tot);
            } else {
                q8_0_chunk<M, L, R>(src, kLaneRows * CB, xk, XS, p.magic, tot);
            }
            __syncwarp();  // every lane is done reading the stage
            if (issued < cpw) {
#if QMM_GEMV_PROXY_FENCE
                fence_proxy_async_smem();
#endif
                // The stage was only read (its values are already in registers
                // and used), so the TMA write that refills it needs no proxy
                // fence: a write-after-read through the async proxy is ordered
                // by the warp's own program order and __syncwarp.
                issue(st, issued);  // issued == i + S: the stage just read
                ++issued;
            }
            if (++st == S) {
                st = 0;
                par ^= 1u;
            }
        }
    }
    if (failed) {
        // Let copies still in flight land before the CTA's shared memory is
        // released; each wait is again bounded.
        if (!x_ok) mbar_wait(xbar, 0, p.ctx);
        for (int j = consumed; j < issued; ++j)
            mbar_wait(&my_bars[j % S], static_cast<uint32_t>(j / S) & 1u, p.ctx);
    }

    // this CTA reads no more activations: its slice may take the cluster's sums
    if (ksplit > 1) gemv_cluster_arrive();
    if constexpr (RP) {  // pair p holds rows 2p and 2p+1 of the lane
#pragma unroll
        for (int j = 0; j < R / 2; ++j)
#pragma unroll
            for (int m = 0; m < M; ++m) {
                tot[2 * j][m] = acc[j][m].x;
                tot[2 * j + 1][m] = acc[j][m].y;
            }
    }
    // 0) the L lanes of a row add their shares (every lane ends with the sum)
#pragma unroll
    for (int off = 1; off < L; off <<= 1) {
#pragma unroll
        for (int j = 0; j < R; ++j)
#pragma unroll
            for (int m = 0; m < M; ++m) tot[j][m] += __shfl_xor_sync(0xFFFFFFFFu, tot[j][m], off);
    }
    const bool writer = h == 0;
    // 1) K parts inside the CTA: warps kpart > 0 hand their sums to kpart 0
    if (kw > 1) {
        if (kpart > 0 && writer) {
#pragma unroll
            for (int j = 0; j < R; ++j)
#pragma unroll
                for (int m = 0; m < M; ++m)
                    red_of(warp)[m * kRowsPerWarp + j * kLaneRows + r] = tot[j][m];
        }
        __syncthreads();
        if (kpart == 0) {
#pragma unroll
            for (int q = 1; q < QMM_GEMV_MAX_KW; ++q) {
                if (q < kw) {
#pragma unroll
                    for (int j = 0; j < R; ++j)
#pragma unroll
                        for (int m = 0; m < M; ++m)
                            tot[j][m] += red_of(warp + q)[m * kRowsPerWarp + j * kLaneRows + r];
                }
            }
        }
    }
    // 2) K parts across the cluster: ranks push into rank 0, which adds in rank order
    if (ksplit == 1) {
        if (kpart == 0 && writer) {
            if constexpr (G) {
                const int row = row0 + r;
                if (row < n_rows) {
#pragma unroll
                    for (int m = 0; m < M; ++m)
                        y[static_cast<size_t>(m) * n_rows + row] = gelu_tanh(tot[0][m]) * tot[1][m];
                }
            } else {
#pragma unroll
                for (int j = 0; j < R; ++j) {
                    const int row = row0 + j * kLaneRows + r;
                    if (row < n_rows) {
#pragma unroll
                        for (int m = 0; m < M; ++m)
                            y[static_cast<size_t>(m) * n_rows + row] = tot[j][m];
                    }
                }
            }
        }
        return;
    }
    gemv_cluster_wait();  // every CTA of the cluster is done with its activations
    if (kpart == 0 && writer) {
        float *slot = part + ((rank * p.rw + tile_in_cta) * M) * kRowsPerWarp;
#pragma unroll
        for (int j = 0; j < R; ++j)
#pragma unroll
            for (int m = 0; m < M; ++m)
                st_dsmem_f32(slot + m * kRowsPerWarp + j * kLaneRows + r, 0, tot[j][m]);
    }
    cluster_sync();
    if (rank == 0) {
        // every thread of rank 0 adds the ranks' sums of some outputs, in rank
        // order (the same order for every output); consecutive threads take
        // consecutive rows.  The rank loop is unrolled to the largest cluster
        // with a guard: a run-time loop measured about 100 ns per partial.
        const int total = p.rw * M * kTileRows;
        const int qstride = p.rw * M * kRowsPerWarp;
        for (int o = threadIdx.x; o < total; o += blockDim.x) {
            const int rt = o % kTileRows;  // row within the tile
            const int mt = o / kTileRows;
            const int m = mt % M;
            const int tile = mt / M;
            const int row = (group * p.rw + tile) * kTileRows + rt;
            if (row >= n_rows) continue;
            const float *pp = part + (tile * M + m) * kRowsPerWarp + rt;
            float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
            for (uint32_t q = 0; q < QMM_GEMV_MAX_KSPLIT; ++q) {
                if (q < ksplit) {
                    s0 += pp[q * qstride];
                    if constexpr (G) s1 += pp[q * qstride + kLaneRows];  // the up row
                }
            }
            if constexpr (G)
                y[static_cast<size_t>(m) * n_rows + row] = gelu_tanh(s0) * s1;
            else
                y[static_cast<size_t>(m) * n_rows + row] = s0;
        }
    }
}

// ---- Persistent form: large N at M <= 10 (one launch that spans many waves) ----
// One CTA per SM.  CTA c owns whole tiles [c*T/G, (c+1)*T/G) of the T row
// tiles (G CTAs), so every SM gets the same work to within one tile; its nw
// warps split the CTA's (tile, chunk) units evenly, in order.  A warp streams
// its units through its ring without a break at tile boundaries and keeps one
// set of sums per tile: a tile it covers whole it writes out, a tile it shares
// with the previous or the next warp goes to a shared-memory slot, and after
// one CTA barrier the two halves are added, earlier chunks first.  The
// activations are copied once per CTA.  Each warp covers at least one tile's
// worth of units (the launcher requires T/G >= nw), so a tile is shared by at
// most two warps.
struct PersistParams {
    const float *x;
    float *y;
    int n;          // rows
    int tiles;      // row tiles (32 * R rows each)
    int chunks;     // K / 256
    int stages;     // ring depth per warp
    uint32_t magic;  // 0x4B000000 (2^23), kept in a register by the kernel
    LaunchCtx ctx;
};

template <Fmt F, int M, int R>
__global__ void __launch_bounds__(QMM_GEMV_MAX_THREADS, 1)  // one CTA per SM
    gemv_persist_kernel(const __grid_constant__ CUtensorMap wmap, PersistParams p) {
    static_assert(M <= QMM_GEMV_R_WIDE_MAX_M, "the per-block chunk forms");
    constexpr int CB = StreamFmt<F>::kChunkBytes;
    constexpr int EB = StreamFmt<F>::kElemBytes;
    constexpr int kRows = 32 * R;  // lane r owns rows r, r + 32, ... of a tile
    extern __shared__ __align__(128) uint8_t smem_dyn[];
    uint8_t *smem = smem_dyn + ((128u - (smem_addr(smem_dyn) & 127u)) & 127u);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int S = p.stages, C = p.chunks, XS = C * kChunkK;
    const int G = gridDim.x;
    const int t0 = static_cast<int>(static_cast<int64_t>(blockIdx.x) * p.tiles / G);
    const int t1 = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * p.tiles / G);
    const int uc = (t1 - t0) * C;  // the CTA's units, tile-major
    const int u0 = static_cast<int>(static_cast<int64_t>(warp) * uc / nw);
    const int nu = static_cast<int>(static_cast<int64_t>(warp + 1) * uc / nw) - u0;

    // shared memory: ring [nw][S][kRows][CB] | xs [M][XS] | slots [nw][2][M][kRows] |
    //                bars [nw][S] | xbar
    const size_t ring_bytes = static_cast<size_t>(S) * kRows * CB;  // per warp
    uint8_t *my_ring = smem + warp * ring_bytes;
    float *xs = reinterpret_cast<float *>(smem + nw * ring_bytes);
    float *slots = xs + M * XS;  // [warp][0]: a tile's later chunks, [warp][1]: its earlier ones
    uint64_t *bars = reinterpret_cast<uint64_t *>(slots + nw * 2 * M * kRows);
    uint64_t *my_bars = bars + warp * S;
    uint64_t *xbar = bars + nw * S;

    if (lane == 0) {
        if (warp == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&wmap)) : "memory");
            mbar_init(xbar, 1);
        }
        for (int s = 0; s < S; ++s) mbar_init(&my_bars[s], 1);
        fence_mbar_init();
    }
    __syncthreads();  // barriers initialised before any thread waits on them

    int it = t0 + u0 / C, ic = u0 % C;  // next unit to request (every lane keeps the count)
    auto issue = [&](int st) {
        if (lane == 0) {
            mbar_arrive_expect_tx(&my_bars[st], kRows * CB);
            tma_load_2d(my_ring + st * kRows * CB, &wmap, ic * (CB / EB), it * kRows, &my_bars[st]);
        }
        if (++ic == C) {
            ic = 0;
            ++it;
        }
    };
    // weights before the dependency wait (read-only model data), activations after
    constexpr int kPrewait = F == Fmt::Q4_0 ? QMM_GEMV_PREWAIT_Q4_0 : QMM_GEMV_PREWAIT_Q8_0;
    int issued = 0;
    for (; issued < min(min(S, nu), kPrewait); ++issued) issue(issued);
    pdl_wait();
    if (threadIdx.x == 0) {  // activations: one bulk copy per row m
        mbar_arrive_expect_tx(xbar, static_cast<uint32_t>(M * XS * sizeof(float)));
#pragma unroll
        for (int m = 0; m < M; ++m)
            bulk_g2s(xs + m * XS, p.x + static_cast<size_t>(m) * XS,
                     static_cast<uint32_t>(XS * sizeof(float)), xbar);
    }
    pdl_launch_dependents();
    if (kPrewait < S) {  // (the same in every warp) the rest of the ring, after the activations
        __syncthreads();
        for (; issued < min(S, nu); ++issued) issue(issued);
    }

    float tot[R][M];
#pragma unroll
    for (int j = 0; j < R; ++j)
#pragma unroll
        for (int m = 0; m < M; ++m) tot[j][m] = 0.0f;
    // every warp waits for the activations (so none exits with the copy in flight)
    const bool x_ok = __all_sync(0xFFFFFFFFu, mbar_wait(xbar, 0, p.ctx));
    bool failed = !x_ok;
    int consumed = 0;
    int tc = t0 + u0 / C, cc = u0 % C;  // the unit being added
    bool head = cc != 0;                // the first tile began in the previous warp's units
    int st = 0;
    uint32_t par = 0;
    for (int i = 0; i < nu && !failed; ++i) {
        // a lane's wait can give up while another's succeeds: the warp decides together
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&my_bars[st], par, p.ctx))) {
            failed = true;
            break;
        }
        ++consumed;
        const uint8_t *src = my_ring + (st * kRows + lane) * CB;
        const float *xk = xs + cc * kChunkK;
        if constexpr (M > QMM_GEMV_R2_MAX_M) {
            if constexpr (F == Fmt::Q4_0)
                q4_0_chunk_wide<M, R>(src, 32 * CB, xk, XS, p.magic, tot);
            else
                q8_0_chunk_wide<M, R>(src, 32 * CB, xk, XS, p.magic, tot);
        } else if constexpr (F == Fmt::Q4_0) {
            q4_0_chunk<M, 1, R>(src, 32 * CB, xk, XS, p.magic, tot);
        } else {
            q8_0_chunk<M, 1, R>(src, 32 * CB, xk, XS, p.magic, tot);
        }
        __syncwarp();  // every lane is done reading the stage before it is refilled
        if (issued < nu) {
            issue(st);
            ++issued;
        }
        if (++st == S) {
            st = 0;
            par ^= 1u;
        }
        if (cc == C - 1 || i == nu - 1) {  // this warp's share of tile tc ends here
            float *slot = head ? slots + (warp * 2 + 0) * M * kRows
                               : (cc != C - 1 ? slots + (warp * 2 + 1) * M * kRows : nullptr);
            if (slot) {
#pragma unroll
                for (int j = 0; j < R; ++j)
#pragma unroll
                    for (int m = 0; m < M; ++m) slot[m * kRows + j * 32 + lane] = tot[j][m];
            } else {
#pragma unroll
                for (int j = 0; j < R; ++j) {
                    const int row = tc * kRows + j * 32 + lane;
                    if (row < p.n) {
#pragma unroll
                        for (int m = 0; m < M; ++m)
                            p.y[static_cast<size_t>(m) * p.n + row] = tot[j][m];
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < R; ++j)
#pragma unroll
                for (int m = 0; m < M; ++m) tot[j][m] = 0.0f;
            head = false;
        }
        if (++cc == C) {
            cc = 0;
            ++tc;
        }
    }
    if (failed) {
        // Let copies still in flight land before the CTA's shared memory is
        // released; each wait is again bounded.
        if (!x_ok) mbar_wait(xbar, 0, p.ctx);
        for (int j = consumed; j < issued; ++j)
            mbar_wait(&my_bars[j % S], static_cast<uint32_t>(j / S) & 1u, p.ctx);
    }
    __syncthreads();
    // a tile shared with the previous warp: its earlier chunks (that warp's
    // last slot) plus the later ones (this warp's first slot)
    if (warp > 0 && u0 % C != 0) {
        const int t = t0 + u0 / C;
        const float *early = slots + ((warp - 1) * 2 + 1) * M * kRows;
        const float *late = slots + (warp * 2 + 0) * M * kRows;
#pragma unroll
        for (int j = 0; j < R; ++j) {
            const int row = t * kRows + j * 32 + lane;
            if (row < p.n) {
#pragma unroll
                for (int m = 0; m < M; ++m)
                    p.y[static_cast<size_t>(m) * p.n + row] =
                        early[m * kRows + j * 32 + lane] + late[m * kRows + j * 32 + lane];
            }
        }
    }
}

// Byte-wise fallback: one warp per row, lanes over blocks.
template <Fmt F, int M>
__device__ __forceinline__ void bytewise_row(const uint8_t *__restrict__ w,
                                             const float *__restrict__ x, int64_t row, int64_t k,
                                             int lane, float (&acc)[M]) {
    constexpr int kBB = F == Fmt::Q4_0 ? kQ4_0Bytes : kQ8_0Bytes;
    const int64_t nb = k / kQK;
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
    for (int m = 0; m < M; ++m)
        for (int off = 16; off > 0; off >>= 1) acc[m] += __shfl_xor_sync(0xFFFFFFFFu, acc[m], off);
}

// y[m][row] = x[m] . w[row]; G (GeGLU): y[m][row] = gelu(x[m] . w[row]) * (x[m] . w2[row]).
template <Fmt F, int M, bool G = false>
__global__ void __launch_bounds__(128) gemv_bytewise_kernel(const uint8_t *__restrict__ w,
                                                           const uint8_t *__restrict__ w2,
                                                           const float *__restrict__ x,
                                                           float *__restrict__ y, int64_t n,
                                                           int64_t k, LaunchCtx ctx) {
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (row >= n) return;
    float acc[M];
    bytewise_row<F, M>(w, x, row, k, lane, acc);
    if constexpr (G) {
        float up[M];
        bytewise_row<F, M>(w2, x, row, k, lane, up);
#pragma unroll
        for (int m = 0; m < M; ++m) acc[m] = gelu_tanh(acc[m]) * up[m];
    }
    if (lane == 0) {
#pragma unroll
        for (int m = 0; m < M; ++m) y[m * n + row] = acc[m];
    }
}

// Launch shape.  g = kw * ksplit K parts per 32-row tile, the smallest
// power of two giving about QMM_GEMV_WARPS_PER_SM warps per SM (at most one
// part per chunk).  Parts go to warps of one CTA first (cheap reduction),
// then to a cluster; CTAs hold rw tiles when kw alone gives few warps.  The
// CTA's activation slice must fit its shared-memory budget.
struct StreamShape {
    int ksplit, kw, rw, cpw, stages;
    size_t smem;
};

template <Fmt F, int M, int L, int R>
StreamShape stream_shape(int64_t tiles, int64_t k, int sms) {
    constexpr int CB = StreamFmt<F>::kChunkBytes;
    constexpr int kRowsPerWarp = 32 / L * R;
    StreamShape sh;
    const int C = static_cast<int>(k / kChunkK);
    const int64_t want = static_cast<int64_t>(QMM_GEMV_WARPS_PER_SM) * sms;
    int g = 1;
    while (g < C && C % (2 * g) == 0 && tiles * g < want &&
           g < QMM_GEMV_MAX_KW * QMM_GEMV_MAX_KSPLIT)
        g *= 2;
    sh.kw = std::min(g, QMM_GEMV_MAX_KW);
    sh.ksplit = g / sh.kw;
    // the CTA's activation slice (M rows x its K range) must fit the budget
    while (sh.ksplit < QMM_GEMV_MAX_KSPLIT && (C / sh.ksplit) % 2 == 0 && sh.kw > 1 &&
           static_cast<int64_t>(M) * (k / sh.ksplit) * 4 > QMM_GEMV_X_BYTES) {
        sh.ksplit *= 2;
        sh.kw /= 2;
    }
    while (sh.ksplit < QMM_GEMV_MAX_KSPLIT && (C / sh.ksplit) % 2 == 0 &&
           static_cast<int64_t>(M) * (k / sh.ksplit) * 4 > QMM_GEMV_X_BYTES)
        sh.ksplit *= 2;
    sh.cpw = C / (sh.kw * sh.ksplit);
    sh.rw = 1;
    while (sh.rw * sh.kw < QMM_GEMV_MIN_WARPS && tiles >= 2LL * sh.rw * sms) sh.rw *= 2;
    sh.stages = std::min(sh.cpw, QMM_GEMV_STAGES);
    auto smem_of = [&](const StreamShape &t) {
        const int nw = t.rw * t.kw;
        const int cta_chunks = t.kw * t.cpw;
        return static_cast<size_t>(nw) * t.stages * kRowsPerWarp * CB +
               sizeof(float) * (static_cast<size_t>(M) * cta_chunks * kChunkK +
                                (static_cast<size_t>(t.ksplit) * t.rw * kRowsPerWarp <=
                                         static_cast<size_t>(cta_chunks) * kChunkK
                                     ? 0
                                     : static_cast<size_t>(t.ksplit) * t.rw * M * kRowsPerWarp)) +
               sizeof(uint64_t) * (nw * t.stages + 1) + 128;
    };
    // fit the shared-memory budget: shallower rings, then fewer tiles per CTA,
    // then a wider cluster split (halves the activation slice), then K parts
    // moved from the CTA's warps to the cluster (halves the ring as well)
    while (smem_of(sh) > kGemvSmemCap && sh.stages > 2) --sh.stages;
    while (smem_of(sh) > kGemvSmemCap && sh.rw > 1) sh.rw /= 2;
    while (smem_of(sh) > kGemvSmemCap && sh.stages > 1) --sh.stages;
    while (smem_of(sh) > kGemvSmemCap && sh.ksplit < QMM_GEMV_MAX_KSPLIT &&
           C % (2 * sh.kw * sh.ksplit) == 0) {
        sh.ksplit *= 2;
        sh.cpw = C / (sh.kw * sh.ksplit);
        sh.stages = std::min(sh.stages, sh.cpw);
    }
    while (smem_of(sh) > kGemvSmemCap && sh.kw > 1 && sh.ksplit < QMM_GEMV_MAX_KSPLIT) {
        sh.kw /= 2;
        sh.ksplit *= 2;
    }
    sh.smem = smem_of(sh);
    return sh;
}

// One launch over `count` problems sharing x: problem i has weights
// probs[i].w (probs[i].n rows) and output probs[i].y.  G (GeGLU): count == 2,
// probs[0] the gate weights and the output h, probs[1] the up weights (same
// n); one problem of n outputs whose tiles read both.
template <Fmt F, int M, int L, int R, bool G = false, bool RP = false>
cudaError_t launch_stream(const GemvProblem *probs, int count, const float *x, int64_t k,
                          cudaStream_t stream, const LaunchCtx &ctx) {
    constexpr int kRowsPerWarp = 32 / L * R;
    constexpr int kTileRows = G ? 32 / L : kRowsPerWarp;  // output rows of a tile
    constexpr int kBoxRows = G ? 32 / L : kRowsPerWarp;   // rows of one TMA box
    int64_t tiles = 0;
    for (int i = 0; i < (G ? 1 : count); ++i) tiles += (probs[i].n + kTileRows - 1) / kTileRows;
    const StreamShape sh = stream_shape<F, M, L, R>(tiles, k, device_sm_count());
    if (sh.smem > kGemvSmemCap) return kShapeTooLarge;  // nothing launched
    // the row-pair form sums at most 1024 products per fp32 accumulator (a
    // lane's share of each of its chunks is 256 / L weights)
    if (RP && sh.cpw * (kChunkK / L) > kRpMaxProducts) return kShapeTooLarge;
    StreamMaps maps;
    StreamParams p;
    p.x = x;
    p.k = static_cast<int>(k);
    p.count = G ? 1 : count;
    p.rw = sh.rw;
    p.kw = sh.kw;
    p.cpw = sh.cpw;
    p.stages = sh.stages;
    p.magic = kMagic;
    p.ctx = ctx;
    const uint64_t rowbytes = static_cast<uint64_t>(k / kChunkK) * StreamFmt<F>::kChunkBytes;
    constexpr int EB = StreamFmt<F>::kElemBytes;
    int64_t groups = 0;
    for (int i = 0; i < kMaxGemvProblems; ++i) {
        if (i < count) {
            if (!encode_tmap_2d(&maps.m[i], StreamFmt<F>::kType, probs[i].w, rowbytes / EB,
                                probs[i].n, rowbytes, StreamFmt<F>::kChunkBytes / EB, kBoxRows))
                return cudaErrorInvalidValue;
        } else {
            maps.m[i] = maps.m[0];
        }
        if (i < p.count) {
            p.y[i] = probs[i].y;
            p.n[i] = static_cast<int>(probs[i].n);
            p.group_begin[i] = static_cast<int>(groups);
            const int64_t t = (probs[i].n + kTileRows - 1) / kTileRows;
            groups += (t + sh.rw - 1) / sh.rw;
        } else {
            p.y[i] = nullptr;
            p.n[i] = 0;
            p.group_begin[i] = static_cast<int>(groups);
        }
    }
    p.group_begin[kMaxGemvProblems] = static_cast<int>(groups);
    auto kern = gemv_stream_kernel<F, M, L, R, G, RP>;
    static int smem_limits[kMaxDevices] = {0};  // this instantiation's own cache
    const cudaError_t e = ensure_smem(kern, sh.smem, true, smem_limits);
    if (e != cudaSuccess) return e;
    return launch_kernel(kern, dim3(static_cast<unsigned>(groups * sh.ksplit)),
                         dim3(sh.rw * sh.kw * 32), sh.smem, stream,
                         static_cast<unsigned>(sh.ksplit), maps, p);
}


// The persistent form (one problem): one CTA per SM, warps and ring depth
// chosen for the shared-memory budget.  kShapeTooLarge when the matrix has
// too few tiles for every warp to hold one, or nothing fits.
template <Fmt F, int M, int R>
cudaError_t launch_persist(const GemvProblem &pr, const float *x, int64_t k, cudaStream_t stream,
                           const LaunchCtx &ctx) {
    constexpr int CB = StreamFmt<F>::kChunkBytes;
    constexpr int EB = StreamFmt<F>::kElemBytes;
    constexpr int kRows = 32 * R;
    const int sms = device_sm_count();
    const int64_t tiles = (pr.n + kRows - 1) / kRows;
    const int64_t C = k / kChunkK;
    auto smem_of = [&](int nw, int S) {
        return static_cast<size_t>(nw) * S * kRows * CB +
               sizeof(float) * (static_cast<size_t>(M) * C * kChunkK + static_cast<size_t>(nw) * 2 * M * kRows) +
               sizeof(uint64_t) * (nw * S + 1) + 128;
    };
    // 8 warps with at least two stages each, else 4 warps with the deepest ring that fits
    int nw = 0, S = 0;
    for (int w : {8, 4}) {
        for (int s = QMM_GEMV_STAGES; s >= 2 && nw == 0; --s)
            if (smem_of(w, s) <= kGemvSmemCap) nw = w, S = s;
        if (nw != 0) break;
    }
    if (nw == 0) return kShapeTooLarge;
    const size_t smem = smem_of(nw, S);
    if (smem > kGemvSmemCap || tiles < static_cast<int64_t>(nw) * sms) return kShapeTooLarge;
    CUtensorMap map;
    const uint64_t rowbytes = static_cast<uint64_t>(C) * CB;
    if (!encode_tmap_2d(&map, StreamFmt<F>::kType, pr.w, rowbytes / EB, pr.n, rowbytes, CB / EB, kRows))
        return cudaErrorInvalidValue;
    PersistParams p;
    p.x = x;
    p.y = pr.y;
    p.n = static_cast<int>(pr.n);
    p.tiles = static_cast<int>(tiles);
    p.chunks = static_cast<int>(C);
    p.stages = S;
    p.magic = kMagic;
    p.ctx = ctx;
    auto kern = gemv_persist_kernel<F, M, R>;
    static int smem_limits[kMaxDevices] = {0};
    const cudaError_t e = ensure_smem(kern, smem, false, smem_limits);
    if (e != cudaSuccess) return e;
    return launch_kernel(kern, dim3(static_cast<unsigned>(sms)), dim3(nw * 32), smem, stream, 1, map, p);
}

// Whether two lanes per row (QMM_GEMV_R_SMALL rows each) need a smaller
// cluster split along K than one lane per row with two rows.
template <Fmt F, int M>
bool two_lanes_split_less(const GemvProblem *probs, int count, int64_t k) {
    int64_t t1 = 0, t2 = 0;
    for (int i = 0; i < count; ++i) {
        t1 += (probs[i].n + 63) / 64;
        t2 += (probs[i].n + 16 * QMM_GEMV_R_SMALL - 1) / (16 * QMM_GEMV_R_SMALL);
    }
    const int sms = device_sm_count();
    return stream_shape<F, M, 2, QMM_GEMV_R_SMALL>(t2, k, sms).ksplit <
           stream_shape<F, M, 1, 2>(t1, k, sms).ksplit;
}

template <Fmt F, int M, bool G = false>
cudaError_t launch_m(const GemvProblem *probs, int count, const float *x, int64_t k,
                     cudaStream_t stream, const LaunchCtx &ctx) {
    bool aligned = (reinterpret_cast<uintptr_t>(x) & 15) == 0;
    int64_t units = 0;
    for (int i = 0; i < count; ++i) {
        aligned = aligned && (reinterpret_cast<uintptr_t>(probs[i].w) & 15) == 0 &&
                  probs[i].n <= (1LL << 30);
        units += ((probs[i].n + 31) / 32) * (k / kChunkK);
    }
    if (k % kChunkK == 0 && aligned && k <= (1LL << 24)) {
        // Lanes per row: small problems at small M are latency bound, so more
        // lanes share each row chunk; large or wide-M problems keep one.
        // Rows per lane: at small M each activation load feeds two weight rows.
        // A shape whose activation slice cannot fit shared memory even at the
        // largest cluster split (very large K at large M) is refused before
        // any launch and takes the byte-wise kernel below.
        cudaError_t e;
        if constexpr (G) {
            // GeGLU: a lane always owns the gate row and the up row of an output
            if constexpr (M <= QMM_GEMV_R2_MAX_M) {
                if (units <= QMM_GEMV_L2_UNITS)
                    e = launch_stream<F, M, 2, 2, true>(probs, count, x, k, stream, ctx);
                else
                    e = launch_stream<F, M, 1, 2, true>(probs, count, x, k, stream, ctx);
            } else {
                e = launch_stream<F, M, 1, 2, true>(probs, count, x, k, stream, ctx);
            }
        } else if constexpr (F == Fmt::Q4_0 && M >= QMM_GEMV_RP_MIN_M) {
            // wide M: row pairs (the FMA pipe bounds it); a K share too long
            // for one accumulator takes the per-block form below
            e = launch_stream<F, M, QMM_GEMV_RP_L, QMM_GEMV_RP_R, false, true>(probs, count, x, k,
                                                                              stream, ctx);
            if (e == kShapeTooLarge) {
                if constexpr (M <= QMM_GEMV_R_WIDE_MAX_M) {
                    e = launch_stream<F, M, 1, 2>(probs, count, x, k, stream, ctx);
                    if (e == kShapeTooLarge) e = launch_stream<F, M, 1, 1>(probs, count, x, k, stream, ctx);
                } else {
                    e = launch_stream<F, M, 1, 1>(probs, count, x, k, stream, ctx);
                }
            }
        } else if constexpr (M <= QMM_GEMV_R2_MAX_M) {
            if (units <= QMM_GEMV_L2_UNITS) {
                e = launch_stream<F, M, 2, QMM_GEMV_R_SMALL>(probs, count, x, k, stream, ctx);
            } else {
                // one large matrix: the persistent form when every warp gets a tile
                constexpr bool kPersist = F == Fmt::Q4_0 ? QMM_GEMV_PERSIST : QMM_GEMV_PERSIST_Q8_0;
                e = count == 1 && kPersist ? launch_persist<F, M, 2>(probs[0], x, k, stream, ctx)
                                           : kShapeTooLarge;
                // M = 1, few rows and a long K (2048 x 8192): two lanes a row give
                // four times the tiles, so K spreads over clusters of 2 CTAs instead
                // of 4 (5.97 -> 5.27 us).  Where both forms need the same cluster, one
                // lane a row (two rows each) is faster (8192 x 2048: 3.99 against
                // 4.57 us), and so it is at M = 2..4 on any shape (2048 x 8192 at
                // M = 3: 6.85 against 10.43 us)
                if (M == 1 && e == kShapeTooLarge && two_lanes_split_less<F, M>(probs, count, k))
                    e = launch_stream<F, M, 2, QMM_GEMV_R_SMALL>(probs, count, x, k, stream, ctx);
                if (e == kShapeTooLarge) e = launch_stream<F, M, 1, 2>(probs, count, x, k, stream, ctx);
            }
        } else {
            // the activation loads bound wide M; two rows per lane halve them per
            // FMA until the accumulators crowd the registers (M > 10); where
            // their shared memory does not fit, one row per lane
            if constexpr (M <= QMM_GEMV_R_WIDE_MAX_M) {
                constexpr bool kPersist = F == Fmt::Q4_0 ? QMM_GEMV_PERSIST : QMM_GEMV_PERSIST_Q8_0;
                e = count == 1 && kPersist ? launch_persist<F, M, 2>(probs[0], x, k, stream, ctx)
                                           : kShapeTooLarge;
                if (e == kShapeTooLarge) e = launch_stream<F, M, 1, 2>(probs, count, x, k, stream, ctx);
                if (e == kShapeTooLarge) e = launch_stream<F, M, 1, 1>(probs, count, x, k, stream, ctx);
            } else {
                e = launch_stream<F, M, 1, 1>(probs, count, x, k, stream, ctx);
            }
        }
        if (e != kShapeTooLarge) return e;
    }
    if constexpr (G) {  // byte-wise GeGLU: both rows of an output in one warp
        const unsigned grid = static_cast<unsigned>((probs[0].n + 3) / 4);
        return launch_kernel(gemv_bytewise_kernel<F, M, true>, dim3(grid), dim3(128), 0, stream, 1,
                             static_cast<const uint8_t *>(probs[0].w),
                             static_cast<const uint8_t *>(probs[1].w), x, probs[0].y, probs[0].n,
                             k, ctx);
    } else {
        for (int i = 0; i < count; ++i) {  // byte-wise kernel, one launch per problem
            const unsigned grid = static_cast<unsigned>((probs[i].n + 3) / 4);
            const cudaError_t e = launch_kernel(
                gemv_bytewise_kernel<F, M>, dim3(grid), dim3(128), 0, stream, 1,
                static_cast<const uint8_t *>(probs[i].w), static_cast<const uint8_t *>(nullptr), x,
                probs[i].y, probs[i].n, k, ctx);
            if (e != cudaSuccess) return e;
        }
        return cudaSuccess;
    }
}

// Dispatch of m in [LO, HI] (one translation unit per range builds in
// parallel with the others).
template <Fmt F, int LO, int HI, bool G = false>
cudaError_t launch_m_range(const GemvProblem *probs, int count, const float *x, int m, int64_t k,
                           cudaStream_t s, const LaunchCtx &ctx) {
    if constexpr (LO > HI) {
        return cudaErrorInvalidValue;
    } else {
        if (m == LO) return launch_m<F, LO, G>(probs, count, x, k, s, ctx);
        return launch_m_range<F, LO + 1, HI, G>(probs, count, x, m, k, s, ctx);
    }
}

}  // namespace
}  // namespace qmm
