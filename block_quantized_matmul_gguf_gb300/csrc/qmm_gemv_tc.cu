// qmm_gemv_tc.cu -- batched decode GEMV y[m][n] = sum_k x[m][k] * w[n][k] for
// Q4_0 weights and M = 1..16 fp32 activation rows on the tensor cores
// (tcgen05, sm_103a), with the accuracy of the fp32 GEMV.
//
// Batches of a few tokens (the batching and MTP verify steps of "Add
// generated quant-kernel JIT and accelerate Gemma4, BGE-M3, and GLiNER2",
// "Summary" and "Benchmarks") make the CUDA-core GEMV spend M FMAs per weight;
// here one MMA row does all M tokens.
//
// Arithmetic.  Per 32-weight block b of row n:
//   S_b[t] = sum_j (nibble_j - 8) * x[t][32b + j],   y[t][n] = sum_b d_b * S_b[t].
// (nibble - 8) is an integer in [-8, 7], exact in bf16: it is the A operand.
// Each activation is split as x = x_hi + x_lo, x_hi = bf16(x), x_lo =
// bf16(x - x_hi) (x - x_hi is exact in fp32), leaving |x - x_hi - x_lo| <=
// 2^-16 |x|; B holds x_hi for the M tokens and x_lo for the same tokens in
// the next Mp rows (N = 2 Mp columns of D, Mp = 8 or 16).  Every product
// (nibble-8) * x_part is exact in the fp32 tensor-memory accumulation; one
// MMA pair (K = 16 each) gives S_b's hi and lo parts for all tokens, and the
// epilogue forms d_b * (hi + lo) in fp32.  The error is at most about
// 2^-16 sum |w x| plus fp32 rounding: inside the fp32 GEMV's bound of
// 1e-4 sum |w x| + 1e-6.
//
// A operand without conversion instructions.  OR-ing a nibble (moved to bits
// 0-3 of a 16-bit half) into the mantissa of bf16 128.0 (0x4300) gives
// 128 + v exactly, two weights per 32-bit word (one LOP3, after a shift for
// all but the first pair); one packed bf16 FMA subtracts 136, exactly.  A
// word of qs bytes (L0 H0)(L1 H1)(L2 H2)(L3 H3) thus yields the column pairs
// (L0, L2), (L1, L3), (H0, H2), (H1, H3): the block's K order is permuted,
// and the B operand is written with the same permutation.
//
// Structure: one CTA per SM (512 TMEM columns), 448 threads, persistent over
// 128-row tiles; the K range is split over a thread-block cluster of ks CTAs
// (partial sums pushed to rank 0's shared memory and added in rank order).
//   warp 0      producer: TMA of raw Q4_0 stages (128 rows x 144 bytes = 256
//               weights per row), from the first instruction after barrier
//               set-up and before the programmatic-launch wait (weights are
//               read-only model data).
//   warp 1      TMEM allocation and the MMA thread: per group of 64 D columns
//               (2 blocks at N = 32, 4 at N = 16), two tcgen05.mma.cta_group::1
//               .kind::f16 (M = 128, N = 2 Mp, K = 16) per block into its own
//               D slot, then one commit for the group (a commit costs about
//               as much issue time as an MMA of these shapes).
//   warps 2-9   dequantisers: lane quarter q = warp % 4, one weight row per
//               lane, half of a stage's 8 blocks per warp; write A with
//               tcgen05.st and the blocks' d (fp32) to shared memory.
//   warps 10-13 epilogue: one tcgen05.ld of a group's D slots, y[t] +=
//               d*(hi+lo); at the end of a tile the K parts are added and y
//               stored (with one tile per cluster, after the final cluster
//               barrier, so that no per-tile cluster handshake is needed).
//   warps 2-13 first convert the CTA's activation slice to B (bf16 hi/lo,
//   128-byte swizzle, K-major) in shared memory.
// Every wait is bounded; a timeout sets the CTA's abort flag and records the
// error; the kernel drains its own copies and MMAs and frees TMEM.
#include "qmm_internal.h"
#include "qmm_tc.cuh"

#include <algorithm>

namespace qmm {
namespace {

constexpr int TW = 128;               // weight rows per tile (MMA M)
constexpr int TCK = 256;              // weights per row per raw stage (8 blocks)
constexpr int TC_ROW_BYTES = 144;     // Q4_0 bytes of one row per raw stage
constexpr int TC_RAW_STAGE = TW * TC_ROW_BYTES;  // 18432
constexpr int TC_AS = 2;              // A slots in TMEM (one raw stage each)
constexpr int TC_DS = 8;              // D slots in TMEM (one block each)
constexpr uint32_t TC_A_COLS = TCK / 2;          // 128 columns per A slot
constexpr uint32_t TC_D_COL0 = TC_AS * TC_A_COLS;  // 256
constexpr uint32_t TC_TMEM_COLS = 512;
constexpr int TC_WARP_PROD = 0, TC_WARP_MMA = 1, TC_WARP_DEQ0 = 2;
constexpr int TC_DEQ_WARPS = 8;       // two per TMEM lane quarter, four blocks of a stage each
constexpr int TC_WARP_EPI0 = TC_WARP_DEQ0 + TC_DEQ_WARPS;  // 10
constexpr int TC_WARP_MMA2 = TC_WARP_EPI0 + 4;             // 14: the second MMA thread
constexpr int TC_THREADS = (TC_WARP_MMA2 + 1) * 32;        // 480
constexpr int TC_CONVERTERS = 4 * 32 * 3;                  // warps 2-13
static_assert(TC_DEQ_WARPS == 8, "dequantiser warp w takes lane quarter w % 4, half (w - 2) / 4");
constexpr int TC_MAX_KS = 8;
// one CTA per SM: every CTA takes more than half of the SM's shared memory,
// so that a second CTA (which would wait for the TMEM this one holds) never
// shares the SM
constexpr size_t TC_MIN_SMEM = 120 * 1024;

struct TcParams {
    float *y;
    int m, n;
    int cta_chunks;   // raw stages (256 weights) per row per CTA: K / (256 ks)
    int tiles;        // 128-row tiles
    int clusters;     // clusters in the grid (each loops over tiles)
    int raw_stages;   // TMA ring depth
    uint32_t off_raw, off_dsm, off_part, off_bars;  // shared-memory offsets (B at 0)
    LaunchCtx ctx;
};

// kind::f16, D fp32, A and B bf16, K-major, M = 128, N = n_cols.
constexpr uint32_t tc_idesc(int n_cols) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n_cols >> 3) << 17) |
           (static_cast<uint32_t>(TW >> 4) << 24);
}

__device__ __forceinline__ uint32_t bf16x2_fma(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Remote (cluster) release arrive and acquire wait, for the K-part reduction.
__device__ __forceinline__ bool mbar_try_wait_acq_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2; "
        "selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// B (activations) in shared memory: rows j < Mp hold x_hi of token j, rows
// Mp + j its x_lo; K-major, 128-byte swizzle: 64-element K slices of N rows
// (N * 128 bytes each), 8-row groups of 1024 bytes, 16-byte chunk c of row r
// stored at chunk c ^ (r & 7).  Within each 32-weight block, K slot s holds
// weight perm(s) (see the file comment): s = 8i + 2t + h holds weight
// 16 (t >> 1) + 4i + (t & 1) + 2h.
template <int MP>
__device__ __forceinline__ void convert_activations(const float *__restrict__ x, int m, int k,
                                                    int k0, int cta_k, uint8_t *b_smem, int tid) {
    constexpr int N = 2 * MP;
    constexpr int U = 4;  // units per thread whose loads are in flight together
    const int cpt = cta_k >> 3;    // 16-byte chunks (8 K slots) per token
    const int units = MP * cpt;    // (token, chunk)
    for (int u0 = tid; u0 < units; u0 += U * TC_CONVERTERS) {
        float4 ld[U][2];
#pragma unroll
        for (int j = 0; j < U; ++j) {
            const int u = u0 + j * TC_CONVERTERS;
            const int t = u / cpt;
            ld[j][0] = ld[j][1] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (u < units && t < m) {
                // slots 8i..8i+7 of block ch/4 (i = ch % 4): weights 4i + {0,2,1,3}
                // and 16 + 4i + {0,2,1,3}
                const int ch = u - t * cpt;
                const float *src = x + static_cast<size_t>(t) * k + k0 + 32 * (ch >> 2) + 4 * (ch & 3);
                ld[j][0] = *reinterpret_cast<const float4 *>(src);
                ld[j][1] = *reinterpret_cast<const float4 *>(src + 16);
            }
        }
#pragma unroll
        for (int j = 0; j < U; ++j) {
            const int u = u0 + j * TC_CONVERTERS;
            if (u >= units) break;
            const int t = u / cpt;
            const int ch = u - t * cpt;
            const float4 a = ld[j][0], c = ld[j][1];
            const float v[8] = {a.x, a.z, a.y, a.w, c.x, c.z, c.y, c.w};
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                hi[q] = pack_bf16x2(v[2 * q], v[2 * q + 1]);
                const float h0 = __uint_as_float(hi[q] << 16), h1 = __uint_as_float(hi[q] & 0xFFFF0000u);
                lo[q] = pack_bf16x2(v[2 * q] - h0, v[2 * q + 1] - h1);
            }
            const int sl = ch >> 3, c16 = ch & 7;
#pragma unroll
            for (int part = 0; part < 2; ++part) {
                const int row = t + part * MP;
                const uint32_t off = static_cast<uint32_t>(sl) * (N * 128) + (row >> 3) * 1024 +
                                     (row & 7) * 128 + ((c16 ^ (row & 7)) << 4);
                *reinterpret_cast<uint4 *>(b_smem + off) =
                    part == 0 ? make_uint4(hi[0], hi[1], hi[2], hi[3]) : make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
        }
    }
}

// Split cluster barrier: arrive early, wait only where it matters.
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}
// Named barrier over the warps after the producer (TMEM address handed out).
__device__ __forceinline__ void sync_after_producer() {
    asm volatile("bar.sync 1, %0;" ::"r"(TC_THREADS - 32) : "memory");
}

// Dequantiser half H (blocks 4H .. 4H+3) of one row's 256-weight stage, held
// in wd[36]: (nibble - 8) as bf16 pairs into TMEM columns a_col + 16 b, and
// the blocks' d (fp32) into dsm_row[b * TW].
template <int H>
__device__ __forceinline__ void dequant_half(const uint32_t (&wd)[36], uint32_t taddr_slot,
                                             float *dsm_row) {
    const uint32_t M128 = 0x43004300u;                       // bf16 128.0, 128.0
    const uint32_t ONE = 0x3F803F80u, NEG136 = 0xC308C308u;  // 1, -136
#pragma unroll
    for (int bb = 0; bb < 4; ++bb) {
        const int b = 4 * H + bb;
        const int base = (18 * b) >> 2;
        uint32_t dbits, qw[4];
        if ((b & 1) == 0) {
            dbits = wd[base] & 0xFFFFu;
#pragma unroll
            for (int i = 0; i < 4; ++i) qw[i] = __byte_perm(wd[base + i], wd[base + i + 1], 0x5432);
        } else {
            dbits = wd[base] >> 16;
#pragma unroll
            for (int i = 0; i < 4; ++i) qw[i] = wd[base + 1 + i];
        }
        dsm_row[b * TW] = half_bits_to_float(dbits);
        uint32_t cols[16];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            // every nibble is moved to bits 0-3 of its 16-bit half first: bf16
            // has 7 mantissa bits, so bits 4-7 would reach the exponent
            const uint32_t v = qw[i];
            cols[4 * i + 0] = bf16x2_fma((v & 0x000F000Fu) | M128, ONE, NEG136);
            cols[4 * i + 1] = bf16x2_fma(((v >> 8) & 0x000F000Fu) | M128, ONE, NEG136);
            cols[4 * i + 2] = bf16x2_fma(((v >> 4) & 0x000F000Fu) | M128, ONE, NEG136);
            cols[4 * i + 3] = bf16x2_fma(((v >> 12) & 0x000F000Fu) | M128, ONE, NEG136);
        }
        tmem_st_16cols(taddr_slot + b * 16, cols);
    }
}

template <int MP>
__global__ void __launch_bounds__(TC_THREADS, 1)
    gemv_tc_kernel(const __grid_constant__ CUtensorMap tmap_w, const float *__restrict__ x, int k,
                   TcParams p) {
    constexpr int N = 2 * MP;
    constexpr uint32_t kIdesc = tc_idesc(N);
    constexpr int BPW = 64 / N;  // blocks per D group: 64 TMEM columns, one commit, one load
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_addr(smem_raw);
    const uint32_t sbase = (raw_base + 1023u) & ~1023u;  // 1024-byte aligned (swizzle atoms)
    uint8_t *sgen = smem_raw + (sbase - raw_base);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const LaunchCtx ctx = p.ctx;
    const uint32_t rank = cluster_rank();
    const uint32_t ks = cluster_nranks();
    const int cluster = static_cast<int>(blockIdx.x / ks);
    const int RS = p.raw_stages;
    const int C = p.cta_chunks;
    // every cluster handles at most one tile: the K parts are then added after
    // the final cluster barrier instead of through per-tile handshakes
    const bool single_tile = p.tiles <= p.clusters;

    // barriers: raw_full[RS], raw_empty[RS], a_full[AS], a_empty[AS],
    // d_full[DS], d_empty[DS] (the first slot of each D group is used),
    // red_full[4], red_empty[4], b_ready, final[2] (one per MMA thread)
    const uint32_t bars = sbase + p.off_bars;
    auto raw_full = [&](int r) { return bars + 8u * r; };
    auto raw_empty = [&](int r) { return bars + 8u * (RS + r); };
    const uint32_t a_full0 = bars + 8u * (2 * RS);
    const uint32_t a_empty0 = a_full0 + 8u * TC_AS;
    const uint32_t d_full0 = a_empty0 + 8u * TC_AS;
    const uint32_t d_empty0 = d_full0 + 8u * TC_DS;
    const uint32_t red_full0 = d_empty0 + 8u * TC_DS;
    const uint32_t red_empty0 = red_full0 + 8u * 4;
    const uint32_t b_ready = red_empty0 + 8u * 4;
    const uint32_t final_bar0 = b_ready + 8u;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sgen + p.off_bars + 8 * (2 * RS + 2 * TC_AS + 2 * TC_DS + 11));
    int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);
    float *dsm = reinterpret_cast<float *>(sgen + p.off_dsm);    // [AS][8 blocks][128 rows]
    float *part = reinterpret_cast<float *>(sgen + p.off_part);  // [ks-1][128 rows][MP+1]

    if (threadIdx.x == 0) {
        // the weight tensor map's first fetch overlaps the barrier set-up
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_w)) : "memory");
        for (int r = 0; r < RS; ++r) {
            mbar_init_addr(raw_full(r), 1);
            mbar_init_addr(raw_empty(r), TC_DEQ_WARPS);
        }
        for (int a = 0; a < TC_AS; ++a) {
            mbar_init_addr(a_full0 + 8u * a, TC_DEQ_WARPS);
            mbar_init_addr(a_empty0 + 8u * a, 2 + 4);  // 2 MMA-thread commits + 4 epilogue warps
        }
        for (int d = 0; d < TC_DS; ++d) {
            mbar_init_addr(d_full0 + 8u * d, 1);
            mbar_init_addr(d_empty0 + 8u * d, 4);
        }
        for (int q = 0; q < 4; ++q) {
            // one tile per cluster: rank 0's warp q expects the peers' partial
            // sums as bulk-copy bytes (one arrival), and each peer waits for
            // one acknowledgement; otherwise per-lane handshakes per tile
            mbar_init_addr(red_full0 + 8u * q, single_tile ? 1u : 32u * (ks > 1 ? ks - 1 : 1));
            mbar_init_addr(red_empty0 + 8u * q, single_tile ? 1u : 32u);
        }
        mbar_init_addr(b_ready, TC_CONVERTERS);
        mbar_init_addr(final_bar0, 1);
        mbar_init_addr(final_bar0 + 8u, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    // this CTA's barriers exist: announce it to the cluster now, wait for the
    // peers only before the first access to their shared memory
    if (ks > 1) cluster_arrive_relaxed();
    bool cluster_waited = false;

    const int my_tiles = cluster < p.tiles ? (p.tiles - cluster + p.clusters - 1) / p.clusters : 0;
    const uint32_t total_stages = static_cast<uint32_t>(my_tiles) * static_cast<uint32_t>(C);
    const int chunk0 = static_cast<int>(rank) * C;  // first raw stage of this CTA's K range

    uint32_t tmem_base = 0;
    float y[MP];
#pragma unroll
    for (int t = 0; t < MP; ++t) y[t] = 0.0f;

    if (warp == TC_WARP_PROD) {
        // weight stages from the start: they need neither TMEM nor the activations
        if (lane == 0) {
            uint32_t it = 0;
            int r = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int i = 0; ok && i < my_tiles; ++i) {
                const int row0 = (cluster + i * p.clusters) * TW;
                for (int c = 0; c < C; ++c) {
                    if (!wait_or_abort(raw_empty(r), ph ^ 1u, abort_flag, ctx)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx_addr(raw_full(r), TC_RAW_STAGE);
                    tma_load_2d(sbase + p.off_raw + r * TC_RAW_STAGE, &tmap_w,
                                (chunk0 + c) * TC_ROW_BYTES, row0, raw_full(r));
                    ++it;
                    if (++r == RS) {
                        r = 0;
                        ph ^= 1u;
                    }
                }
            }
            // every copy lands before the CTA's shared memory is released
            for (int q = 0; q < RS; ++q) {
                if (it > static_cast<uint32_t>(q)) {
                    const uint32_t last = it - 1 - ((it - 1 - q) % RS);
                    wait_drain(raw_full(q), (last / RS) & 1u, ctx);
                }
            }
        }
        __syncwarp();
    } else {
        if (warp == TC_WARP_MMA) tmem_alloc_cta(smem_addr(tmem_slot), TC_TMEM_COLS);
        tc_fence_before();
        sync_after_producer();
        tc_fence_after();
        tmem_base = *reinterpret_cast<volatile uint32_t *>(tmem_slot);
    }

    if (warp == TC_WARP_MMA || warp == TC_WARP_MMA2) {
        // two MMA threads on different schedulers take alternate D groups:
        // one thread issuing every MMA was slowed by the busy warps sharing its
        // scheduler; each commits (and drains) only its own MMAs
        const uint32_t mine = warp == TC_WARP_MMA ? 0u : 1u;
        if (lane == 0) {
            bool ok = total_stages == 0 || wait_or_abort(b_ready, 0, abort_flag, ctx);
            const uint64_t bdesc0 = sw128_desc(sbase);
            bool issued = false;
            uint32_t g = 0;  // blocks of all groups so far
            int a = 0;
            uint32_t aph = 0;
            int c = 0;
            for (uint32_t it = 0; ok && it < total_stages; ++it) {
                if (!wait_or_abort(a_full0 + 8u * a, aph, abort_flag, ctx)) break;
                tc_fence_after();
#pragma unroll 1
                for (int b0 = 0; b0 < 8; b0 += BPW, g += BPW) {
                    if (((g / BPW) & 1u) != mine) continue;
                    const uint32_t ds0 = g % TC_DS;
                    if (!wait_or_abort(d_empty0 + 8u * ds0, ((g / TC_DS) & 1u) ^ 1u, abort_flag, ctx)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int j = 0; j < BPW; ++j) {
                        const int b = b0 + j;
                        // K slots of block b of chunk c: slice (4c + b/2), 64 bytes in for odd b
                        const uint64_t bdesc =
                            bdesc0 + ((static_cast<uint64_t>(4 * c + (b >> 1)) * (N * 128) + (b & 1) * 64) >> 4);
                        const uint32_t a_tmem = tmem_base + a * TC_A_COLS + b * 16;
                        const uint32_t d_tmem = tmem_base + TC_D_COL0 + (ds0 + j) * N;
                        umma_bf16_cta_ta(d_tmem, a_tmem, bdesc, kIdesc, 0u);
                        umma_bf16_cta_ta(d_tmem, a_tmem + 8, bdesc + 2, kIdesc, 1u);  // +16 K: 32 bytes
                    }
                    issued = true;
                    umma_commit_cta(d_full0 + 8u * ds0);
                }
                if (!ok) break;
                umma_commit_cta(a_empty0 + 8u * a);
                if (++a == TC_AS) {
                    a = 0;
                    aph ^= 1u;
                }
                if (++c == C) c = 0;
            }
            if (issued) {  // this thread's MMAs complete before TMEM is freed
                umma_commit_cta(final_bar0 + 8u * mine);
                wait_drain(final_bar0 + 8u * mine, 0, ctx);
            }
        }
        __syncwarp();
    } else if (warp >= TC_WARP_DEQ0) {
        // warps 2-13: the activation slice -> B (after the programmatic-launch
        // wait: x is written by the preceding kernel)
        pdl_wait();
        convert_activations<MP>(x, p.m, k, chunk0 * TCK, C * TCK, sgen, threadIdx.x - 64);
        fence_proxy_async_smem();  // generic writes -> tensor-core reads
        mbar_arrive_addr(b_ready);
        pdl_launch_dependents();

        const int q = warp & 3;           // TMEM lane quarter this warp may access
        const int row = 32 * q + lane;    // weight row within the tile (TMEM lane)
        const uint32_t lane_off = static_cast<uint32_t>(32 * q) << 16;
        if (warp < TC_WARP_EPI0) {
            // ---- dequantisers: two warps per lane quarter, four blocks each ----
            const int half = (warp - TC_WARP_DEQ0) >> 2;
            int r = 0, a = 0;
            uint32_t rph = 0, aph = 0;
            for (uint32_t it = 0; it < total_stages; ++it) {
                if (!warp_wait_or_abort(raw_full(r), rph, abort_flag, ctx)) break;
                uint32_t wd[36];
                const uint8_t *src = sgen + p.off_raw + r * TC_RAW_STAGE + row * TC_ROW_BYTES;
#pragma unroll
                for (int t = 0; t < 9; ++t) {
                    const uint4 v = lds128(src + 16 * t);
                    wd[4 * t + 0] = v.x;
                    wd[4 * t + 1] = v.y;
                    wd[4 * t + 2] = v.z;
                    wd[4 * t + 3] = v.w;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive_addr(raw_empty(r));
                if (++r == RS) {
                    r = 0;
                    rph ^= 1u;
                }
                if (!warp_wait_or_abort(a_empty0 + 8u * a, aph ^ 1u, abort_flag, ctx)) break;
                tc_fence_after();
                const uint32_t taddr = tmem_base + lane_off + a * TC_A_COLS;
                float *dsm_row = dsm + a * 8 * TW + row;
                if (half == 0)
                    dequant_half<0>(wd, taddr, dsm_row);
                else
                    dequant_half<1>(wd, taddr, dsm_row);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_addr(a_full0 + 8u * a);
                if (++a == TC_AS) {
                    a = 0;
                    aph ^= 1u;
                }
            }
        } else {
            // ---- epilogue ----
            uint32_t g = 0;
            int a = 0, c = 0, tile_i = 0;
            uint32_t aph = 0;
            bool ok = true;
            for (uint32_t it = 0; ok && it < total_stages; ++it) {
                if (!warp_wait_or_abort(a_full0 + 8u * a, aph, abort_flag, ctx)) break;
#pragma unroll 1
                for (int b0 = 0; b0 < 8; b0 += BPW, g += BPW) {
                    const uint32_t ds0 = g % TC_DS;
                    if (!warp_wait_or_abort(d_full0 + 8u * ds0, (g / TC_DS) & 1u, abort_flag, ctx)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // the group's D slots are 64 consecutive TMEM columns
                    uint32_t v[64];
                    tmem_ld_64cols(tmem_base + lane_off + TC_D_COL0 + ds0 * N, v);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_addr(d_empty0 + 8u * ds0);
#pragma unroll
                    for (int j = 0; j < BPW; ++j) {
                        const float d = dsm[(a * 8 + b0 + j) * TW + row];
#pragma unroll
                        for (int t = 0; t < MP; ++t)
                            y[t] = fmaf(d, __uint_as_float(v[j * N + t]) + __uint_as_float(v[j * N + MP + t]),
                                        y[t]);
                    }
                }
                if (!ok) break;
                __syncwarp();
                if (lane == 0) mbar_arrive_addr(a_empty0 + 8u * a);
                if (++a == TC_AS) {
                    a = 0;
                    aph ^= 1u;
                }
                if (++c < C) continue;
                // ---- end of a tile: add the K parts, store ----
                c = 0;
                const int n_row = (cluster + tile_i * p.clusters) * TW + row;
                const uint32_t tpar = static_cast<uint32_t>(tile_i) & 1u;
                if (ks > 1 && !cluster_waited) {  // the peers are running: their shared memory exists
                    cluster_wait();
                    cluster_waited = true;
                }
                if (ks > 1 && single_tile) {
                    if (rank != 0) {
                        // partial sums staged in this CTA's own buffer, then one
                        // bulk copy into rank 0's, completing as bytes on rank
                        // 0's barrier (no cluster-scope release needed)
                        float *stage = part + (q * 32 + lane) * MP;
#pragma unroll
                        for (int t = 0; t < MP; ++t) stage[t] = y[t];
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            const uint32_t dst = map_to_rank(
                                smem_addr(part + ((rank - 1) * 4 + q) * 32 * MP), 0);
                            bulk_s2cluster(dst, smem_addr(part + q * 32 * MP), 32 * MP * 4,
                                           map_to_rank(red_full0 + 8u * q, 0));
                        }
                        // rank 0 acknowledges once it has the bytes: this CTA's
                        // buffer (the copy's source) stays until then
                        if (!warp_wait_or_abort(red_empty0 + 8u * q, 0, abort_flag, ctx)) break;
                    } else {
                        if (lane == 0)
                            mbar_expect_tx_addr(red_full0 + 8u * q, (ks - 1) * 32 * MP * 4);
                        if (!warp_wait_or_abort(red_full0 + 8u * q, 0, abort_flag, ctx)) break;
                        for (uint32_t rr = 1; rr < ks; ++rr) {
                            const float *pp = part + (((rr - 1) * 4 + q) * 32 + lane) * MP;
#pragma unroll
                            for (int t = 0; t < MP; ++t) y[t] += pp[t];
                        }
                        __syncwarp();
                        if (lane == 0)
                            for (uint32_t rr = 1; rr < ks; ++rr)
                                mbar_arrive_remote_relaxed(map_to_rank(red_empty0 + 8u * q, rr));
                        if (n_row < p.n) {
#pragma unroll
                            for (int t = 0; t < MP; ++t)
                                if (t < p.m) p.y[static_cast<size_t>(t) * p.n + n_row] = y[t];
                        }
                    }
                    ++tile_i;
                    continue;  // the only tile
                }
                if (ks > 1 && rank != 0) {
                    if (!warp_wait_or_abort(red_empty0 + 8u * q, tpar ^ 1u, abort_flag, ctx)) break;
                    const uint32_t dst = map_to_rank(
                        smem_addr(part + ((rank - 1) * TW + row) * (MP + 1)), 0);
#pragma unroll
                    for (int t = 0; t < MP; ++t) st_cluster_f32(dst + 4u * t, y[t]);
                    mbar_arrive_cluster(map_to_rank(red_full0 + 8u * q, 0));
                } else {
                    if (ks > 1) {
                        // acquire at cluster scope: the peers' partial sums are visible
                        bool got = mbar_try_wait_acq_cluster(red_full0 + 8u * q, tpar);
                        if (!got) {
                            const uint64_t t0 = global_timer_ns();
                            for (uint32_t spin = 0; spin < (1u << 30) && !got; ++spin) {
                                got = mbar_try_wait_acq_cluster(red_full0 + 8u * q, tpar);
                                if (!got && (spin & 15u) == 15u &&
                                    (abort_set(abort_flag) || global_timer_ns() - t0 > ctx.timeout_ns))
                                    break;
                            }
                        }
                        if (!__all_sync(0xFFFFFFFFu, got)) {
                            if (!abort_set(abort_flag)) {
                                *reinterpret_cast<volatile int *>(abort_flag) = 1;
                                record_error(ctx, kDevErrTimeout);
                            }
                            break;
                        }
                        for (uint32_t rr = 1; rr < ks; ++rr) {
                            const float *pp = part + ((rr - 1) * TW + row) * (MP + 1);
#pragma unroll
                            for (int t = 0; t < MP; ++t) y[t] += pp[t];
                        }
                        for (uint32_t rr = 1; rr < ks; ++rr)
                            mbar_arrive_cluster(map_to_rank(red_empty0 + 8u * q, rr));
                    }
                    if (n_row < p.n) {
#pragma unroll
                        for (int t = 0; t < MP; ++t)
                            if (t < p.m) p.y[static_cast<size_t>(t) * p.n + n_row] = y[t];
                    }
                }
#pragma unroll
                for (int t = 0; t < MP; ++t) y[t] = 0.0f;
                ++tile_i;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (ks > 1) {
        if (!cluster_waited) cluster_wait();  // the start-up phase of the cluster barrier
        // several tiles per cluster: no peer may still write this CTA's shared
        // memory (with one tile, every transfer was waited for above)
        if (!single_tile) cluster_barrier();
    }
    tc_fence_after();
    if (warp == TC_WARP_MMA) tmem_dealloc_cta(tmem_base, TC_TMEM_COLS);
}

struct TcShape {
    int ks, clusters, tiles, raw_stages;
    size_t smem, off_raw, off_dsm, off_part, off_bars;
};

constexpr size_t kTcSmemCap = 227 * 1024;

// Shared-memory layout for ks K parts and rs raw stages: B (the CTA's
// activation slice, hi and lo), the raw ring, the block scales, the K-part
// buffer (rank 0 receives ks - 1 partial tiles) and the barriers.
template <int MP>
TcShape tc_layout(int64_t k, int ks, int rs) {
    constexpr int N = 2 * MP;
    TcShape sh{};
    const int C_cta = static_cast<int>(k / TCK) / ks;
    const size_t b_bytes = static_cast<size_t>(C_cta) * TCK * N * 2;
    const size_t dsm_bytes = static_cast<size_t>(TC_AS) * 8 * TW * 4;
    const size_t part_bytes = static_cast<size_t>(std::max(ks - 1, 1)) * TW * (MP + 1) * 4;
    const int nbars = 2 * rs + 2 * TC_AS + 2 * TC_DS + 11;
    sh.ks = ks;
    sh.raw_stages = rs;
    sh.off_raw = b_bytes;
    sh.off_dsm = sh.off_raw + static_cast<size_t>(rs) * TC_RAW_STAGE;
    sh.off_part = sh.off_dsm + dsm_bytes;
    sh.off_bars = (sh.off_part + part_bytes + 15) & ~size_t(15);
    sh.smem = std::max(sh.off_bars + 8 * nbars + 16 + 1024, TC_MIN_SMEM);  // + alignment slack
    return sh;
}

// K parts ks (cluster size): among the splits whose layout fits with at
// least two raw stages, the one that keeps the most SMs busy over whole
// rounds of tiles (ties: fewer parts); then the deepest ring (up to 8) that
// fits.  max_clusters(ks) is how many clusters of ks CTAs (one per SM) can
// be resident at once: with 8-CTA clusters that is fewer than SMs / 8, and
// launching more would run them in a second wave.  ks == 0: no split fits.
template <int MP, typename MaxClusters>
TcShape tc_shape(int64_t n, int64_t k, int sms, MaxClusters max_clusters) {
    TcShape best{};
    const int tiles = static_cast<int>((n + TW - 1) / TW);
    const int C = static_cast<int>(k / TCK);
    double best_eff = -1.0;
    for (int ks = 1; ks <= TC_MAX_KS && C % ks == 0; ks *= 2) {
        if (tc_layout<MP>(k, ks, 2).smem > kTcSmemCap) continue;
        const int clusters = std::max(1, std::min(tiles, std::min(sms / ks, max_clusters(ks))));
        const int rounds = (tiles + clusters - 1) / clusters;
        const double eff = static_cast<double>(tiles) * ks / (static_cast<double>(rounds) * sms);
        if (eff > best_eff + 1e-9) {
            best_eff = eff;
            int rs = 8;
            while (rs > 2 && tc_layout<MP>(k, ks, rs).smem > kTcSmemCap) --rs;
            best = tc_layout<MP>(k, ks, rs);
            best.clusters = clusters;
        }
    }
    best.tiles = tiles;
    return best;
}

template <int MP>
cudaError_t launch_tc(const uint8_t *w, const float *x, float *y, int m, int64_t n, int64_t k,
                      cudaStream_t stream, const LaunchCtx &ctx) {
    // resident clusters per cluster size, queried once per device and size
    static int max_active[kMaxDevices][TC_MAX_KS + 1] = {};
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    static int smem_limits[kMaxDevices] = {0};
    cudaError_t e = ensure_smem(gemv_tc_kernel<MP>, kTcSmemCap, true, smem_limits);
    if (e != cudaSuccess) return e;
    auto max_clusters = [&](int ks) {
        int &cached = max_active[dev][ks];
        if (__atomic_load_n(&cached, __ATOMIC_ACQUIRE) > 0) return cached;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(ks));
        cfg.blockDim = dim3(TC_THREADS);
        cfg.dynamicSmemBytes = TC_MIN_SMEM;  // every layout is at least this (one CTA per SM)
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = static_cast<unsigned>(ks);
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int num = 0;
        if (cudaOccupancyMaxActiveClusters(&num, gemv_tc_kernel<MP>, &cfg) != cudaSuccess || num < 1)
            num = std::max(1, device_sm_count() / (2 * ks));  // conservative if the query fails
        __atomic_store_n(&cached, num, __ATOMIC_RELEASE);
        return num;
    };
    const TcShape sh = tc_shape<MP>(n, k, device_sm_count(), max_clusters);
    if (sh.ks == 0 || sh.smem > kTcSmemCap) return cudaErrorInvalidValue;
    CUtensorMap tw;
    const uint64_t rowbytes = static_cast<uint64_t>(k / TCK) * TC_ROW_BYTES;
    if (!encode_tmap_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, rowbytes, n, rowbytes, TC_ROW_BYTES, TW))
        return cudaErrorInvalidValue;
    TcParams p;
    p.y = y;
    p.m = m;
    p.n = static_cast<int>(n);
    p.cta_chunks = static_cast<int>(k / TCK) / sh.ks;
    p.tiles = sh.tiles;
    p.clusters = sh.clusters;
    p.raw_stages = sh.raw_stages;
    p.off_raw = static_cast<uint32_t>(sh.off_raw);
    p.off_dsm = static_cast<uint32_t>(sh.off_dsm);
    p.off_part = static_cast<uint32_t>(sh.off_part);
    p.off_bars = static_cast<uint32_t>(sh.off_bars);
    p.ctx = ctx;
    return launch_kernel(gemv_tc_kernel<MP>, dim3(static_cast<unsigned>(sh.clusters * sh.ks)),
                         dim3(TC_THREADS), sh.smem, stream, static_cast<unsigned>(sh.ks), tw, x,
                         static_cast<int>(k), p);
}

}  // namespace

bool gemv_tc_shape_ok(int m, int64_t n, int64_t k) {
    if (m < 1 || m > 16 || k < TCK || k % TCK != 0 || n < 1 || n > (int64_t(1) << 30) ||
        k > (int64_t(1) << 24))
        return false;
    // whether some cluster split fits does not depend on the SM count
    auto any = [](int) { return 1; };
    return (m <= 8 ? tc_shape<8>(n, k, 152, any).ks : tc_shape<16>(n, k, 152, any).ks) > 0;
}

cudaError_t launch_gemv_tc_q4_0(const uint8_t *w, const float *x, float *y, int m, int64_t n,
                                int64_t k, cudaStream_t stream, const LaunchCtx &ctx) {
    return m <= 8 ? launch_tc<8>(w, x, y, m, n, k, stream, ctx)
                  : launch_tc<16>(w, x, y, m, n, k, stream, ctx);
}

}  // namespace qmm
