// qmm_gemm.cu -- prefill GEMM Y[m][n] = sum_k X[m][k] * w[n][k] with bf16
// activations X and GGUF Q4_0 weights W, on the 5th-generation tensor cores
// (tcgen05, sm_103a).
//
// Prefill is the TTFT side of the Gemma4 rows in "Add generated quant-kernel
// JIT and accelerate Gemma4, BGE-M3, and GLiNER2" ("Benchmarks": Gemma4 E2B
// TTFT on M4 and L4); the products are the same Q4_0 dispatches as decode
// ("Validation"), with M = prompt tokens.
//
// Per weight: w = (nibble - 8) * d is formed exactly in fp32 and rounded once
// to bf16 (round to nearest even); products are summed in fp32 in tensor
// memory.
//
// Structure: persistent CTA pairs (thread-block clusters of 2), one CTA per
// SM, 576 threads each, warp-specialised.  A pair computes a tile of
// 256 weight rows x 256 tokens as Y^T = W . X^T with
// tcgen05.mma.cta_group::2 (M=256 weight rows, N=256 tokens, K=16): the A
// operand (dequantised W, bf16) is in tensor memory, written there by the
// dequantiser warps with tcgen05.st straight from registers; the B operand
// (X, bf16) is in shared memory, loaded by TMA.  Each CTA holds 128 weight
// rows in its TMEM and 128 tokens of X in its shared memory.  Writing the
// weights to tensor memory instead of shared memory avoids both the shared-
// memory traffic of a dequantised B tile and the generic-to-async proxy
// fence that shared-memory writes need before the tensor core may read
// them (about 1.6k cycles per fence and warp on this part).
//   warp 0      producers (both CTAs): lane 0 loads X tiles (128 tokens x
//               64 bf16, 128-byte swizzle; completion counted on the leader
//               CTA's barrier), lane 1 loads raw Q4_0 tiles (128 rows x 144
//               bytes = 8 blocks per row).
//   warps 2-9   dequantisers (both CTAs): warp w owns TMEM lanes (weight
//               rows) 32*(w%4)..+31 and one of the two 32-weight blocks of
//               each 64-wide K stage; it forms bf16((nibble-8)*d) and writes
//               16 columns of the stage's A slot with tcgen05.st.
//   warp 1      MMA issuer (leader CTA): one thread issues the pair's MMAs
//               into the 256-column accumulator and releases X stages, A
//               slots and the accumulator with multicast tcgen05.commit.
//               X stages and A slots are announced to it per group of four
//               K stages (one wait per 16 MMAs): under the dequantisers'
//               integer load a per-stage wait delayed the issue stream.
//               Every dequantiser warp of both CTAs reports a written A slot
//               on the leader's barrier with a CTA-scope (not cluster-scope)
//               release arrive: the TMEM data is complete once tcgen05.wait::st
//               returns, and a cluster-scope release costs about 1k cycles per
//               arrive on this part, which serialised the pipeline when one
//               peer thread forwarded every stage.
//   warps 10-17 epilogue (both CTAs): tcgen05.ld of the CTA's 128 x 256 fp32
//               accumulator, two warps per lane quarter (half the columns
//               each); lane i holds weight row i, so each store of a warp
//               writes 32 consecutive outputs of one token (coalesced).
// Every wait is bounded (GPU global timer).  On a timeout the CTA records the
// error, sets a shared abort flag that makes its other waits give up at once,
// lets its own TMA copies and MMAs finish (bounded waits), keeps its shared
// memory until the peer has drained (cluster barrier), frees TMEM and exits.
#include "qmm_internal.h"
#include "qmm_tc.cuh"

#include <algorithm>

namespace qmm {
namespace {

#ifndef QMM_GEMM_STAGES
#define QMM_GEMM_STAGES 8
#endif
#ifndef QMM_GEMM_LOOKAHEAD_KK
#define QMM_GEMM_LOOKAHEAD_KK 1
#endif
#ifndef QMM_GEMM_GROUP
#define QMM_GEMM_GROUP 4
#endif
#ifndef QMM_GEMM_RAW_STAGES
#define QMM_GEMM_RAW_STAGES 3
#endif
constexpr int BW = 128;              // weight rows per CTA (MMA M = 2 * BW per pair)
constexpr int BT = 256;              // tokens per pair tile (MMA N); 128 per CTA
constexpr int BT_CTA = BT / 2;
constexpr int BK = 64;               // K per stage (one 128-byte swizzle row of X)
constexpr int UMMA_K = 16;           // K per tcgen05.mma (kind::f16)
constexpr int RAW_K = 256;           // K per raw stage (8 blocks)
constexpr int STAGES = QMM_GEMM_STAGES;  // K stages in flight (X in shared memory, A in TMEM)
constexpr int LOOKAHEAD_KK = QMM_GEMM_LOOKAHEAD_KK;
// Stages are announced to the MMA thread in groups: one "full" barrier per
// GROUP consecutive stages, so the issuing thread waits once per 4*GROUP MMAs.
// Under the integer/fp32 load of the dequantiser warps on the same SM, each
// wait delays the issue stream by a couple of hundred cycles; one wait per
// 16 MMAs hides that behind the MMAs still queued.  Slots are still released
// one stage at a time.
constexpr int GROUP = QMM_GEMM_GROUP;
constexpr int NGROUPS = STAGES / GROUP;
static_assert(STAGES % GROUP == 0, "whole groups in the ring");
// the MMA thread waits for the next group's first stage while the current
// group's slots are still held: one group in the ring would wait forever
static_assert(NGROUPS >= 2, "at least two groups in the ring");
static_assert((256 / BK) % GROUP == 0, "k % 256 == 0 makes every tile a whole number of groups");
constexpr int X_STAGE_BYTES = BT_CTA * BK * 2;           // 16 KB

// Raw weight stages: 128 rows x 256 weights of block bytes, one TMA box.
// Q4_0: 144-byte rows (18 KB a stage, three stages).  Q8_0: 272-byte rows
// (34 KB, two stages, so that the CTA's shared memory still fits), loaded as
// uint16 elements because a box dimension holds at most 256 elements.
template <Fmt F>
struct RawFmt;
template <>
struct RawFmt<Fmt::Q4_0> {
    static constexpr int kRowBytes = 8 * kQ4_0Bytes;  // 144
    static constexpr int kStages = QMM_GEMM_RAW_STAGES;
    static constexpr int kElemBytes = 1;
    static constexpr CUtensorMapDataType kType = CU_TENSOR_MAP_DATA_TYPE_UINT8;
};
template <>
struct RawFmt<Fmt::Q8_0> {
    static constexpr int kRowBytes = 8 * kQ8_0Bytes;  // 272
    static constexpr int kStages = 2;
    static constexpr int kElemBytes = 2;
    static constexpr CUtensorMapDataType kType = CU_TENSOR_MAP_DATA_TYPE_UINT16;
};
constexpr uint32_t D_COLS = BT;                          // fp32 accumulator columns
constexpr uint32_t A_COLS = BK / 2;                      // bf16 pairs per row per stage
constexpr uint32_t TMEM_COLS = 512;
static_assert(D_COLS + STAGES * A_COLS <= TMEM_COLS, "tensor memory budget");
static_assert(LOOKAHEAD_KK >= 0 && LOOKAHEAD_KK < BK / 16, "look-ahead point within a stage");

constexpr int WARP_PRODUCER = 0;
constexpr int WARP_MMA = 1;
constexpr int WARP_DEQ0 = 2;
constexpr int DEQ_PER_STAGE = 8;  // warps writing one K stage: 4 lane quarters x 2 blocks
#ifndef QMM_GEMM_DEQ_PHASES
#define QMM_GEMM_DEQ_PHASES 1
#endif
// 1: one set of dequantiser warps writes every K stage; 2: two sets take
// alternate K stages, so that one set's latency overlaps the other's work
constexpr int DEQ_PHASES = QMM_GEMM_DEQ_PHASES;
static_assert(DEQ_PHASES == 1 || DEQ_PHASES == 2, "dequantiser phases");
constexpr int NUM_DEQ_WARPS = DEQ_PER_STAGE * DEQ_PHASES;
constexpr int WARP_EPI0 = WARP_DEQ0 + NUM_DEQ_WARPS;  // 10 or 18
#ifndef QMM_GEMM_EPI_WARPS
#define QMM_GEMM_EPI_WARPS 8
#endif
constexpr int NUM_EPI_WARPS = QMM_GEMM_EPI_WARPS;  // 4 or 8: one or two per lane quarter
static_assert(NUM_EPI_WARPS == 4 || NUM_EPI_WARPS == 8, "epilogue warps");
constexpr int NUM_THREADS = (WARP_EPI0 + NUM_EPI_WARPS) * 32;  // 448 .. 832

static_assert(RAW_K % BK == 0 && BK == 2 * 32, "a K stage is two blocks");

template <Fmt F>
struct SmemLayout {
    static constexpr int raw_stages = RawFmt<F>::kStages;
    static constexpr int raw_stage_bytes = BW * RawFmt<F>::kRowBytes;
    static constexpr int x = 0;
    static constexpr int raw = x + STAGES * X_STAGE_BYTES;
    static constexpr int bars = raw + raw_stages * raw_stage_bytes;
    // barriers: full [NGROUPS], empty [STAGES]; raw_full, raw_empty
    // [raw_stages]; d_full, d_empty, final
    static constexpr int nbars = NGROUPS + STAGES + 2 * raw_stages + 3;
    static constexpr int tmem_slot = bars + nbars * 8;
    static constexpr int abort_flag = tmem_slot + 4;
    static constexpr int total = abort_flag + 4;
    static constexpr size_t smem_bytes = total + 1024;  // + alignment slack
};
static_assert(SmemLayout<Fmt::Q4_0>::smem_bytes <= 232448, "shared memory per CTA");
static_assert(SmemLayout<Fmt::Q8_0>::smem_bytes <= 232448, "shared memory per CTA");

struct GemmParams {
    float *y;     // plain GEMM: fp32 [m][n]
    uint16_t *h;  // GeGLU form: bf16 [m][n] (n = rows of each of the two weights)
    float *part;  // K split (ksplit > 1): fp32 [ksplit][m][n] partial products
    int m, n, k;
    int num_t_blocks;  // token blocks of BT
    int num_tiles;     // pair tiles
    int ksplit;        // K parts per tile (plain GEMM only); a work item is (tile, part)
    uint32_t magic;    // 0x4B000000 (2^23)
    LaunchCtx ctx;
};

// Instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major,
// N = 256 tokens, M = 256 weight rows (the pair).
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) |
                            (static_cast<uint32_t>(BT >> 3) << 17) |
                            (static_cast<uint32_t>((2 * BW) >> 4) << 24);

#ifndef QMM_GEMM_WAIT_CLUSTER
#define QMM_GEMM_WAIT_CLUSTER 0
#endif
#if QMM_GEMM_WAIT_CLUSTER
#define MMA_WAIT wait_or_abort_cluster
#else
#define MMA_WAIT wait_or_abort
#endif

// G (GeGLU): tmap_w holds the gate weights and tmap_w2 the up weights (64-row
// boxes).  A CTA's 128 accumulator rows are 64 features: in lane quarter q,
// lanes 0-15 hold the gate rows of features 16q..16q+15 and lanes 16-31 the
// up rows of the same features, so lane l and lane l ^ 16 of an epilogue warp
// meet with one shuffle and write h = gelu(g) * u as bf16.  A pair tile is
// 128 features x 256 tokens.
template <Fmt F, bool G>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmap_x,
                const __grid_constant__ CUtensorMap tmap_w,
                const __grid_constant__ CUtensorMap tmap_w2, GemmParams p) {
    static_assert(!G || F == Fmt::Q4_0, "the GeGLU form is built for Q4_0 weights");
    using SL = SmemLayout<F>;
    constexpr int RAW_STAGES = SL::raw_stages;
    constexpr int RAW_STAGE_BYTES = SL::raw_stage_bytes;
    constexpr int RAW_ROW_BYTES = RawFmt<F>::kRowBytes;
    constexpr int RAW_X = RAW_ROW_BYTES / RawFmt<F>::kElemBytes;  // TMA x extent of a raw stage
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_addr(smem_raw);
    const uint32_t sbase = (raw_base + 1023u) & ~1023u;  // 1024-byte aligned (swizzle atoms)
    uint8_t *sgen = smem_raw + (sbase - raw_base);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const LaunchCtx ctx = p.ctx;
    const uint32_t rank = cluster_rank();  // 0 = leader of the pair
    const bool leader = rank == 0;
    const int pair = static_cast<int>(blockIdx.x >> 1);
    const int num_pairs = static_cast<int>(gridDim.x >> 1);

    auto bar = [&](int i) -> uint32_t { return sbase + SL::bars + 8u * i; };
    // full(g): leader only; for each stage of group g, both X producers
    // (expect_tx + bytes) and the 16 dequantiser warps of the pair.
    // empty(s): both CTAs; multicast commit once the stage's MMAs are done.
    // Stage index i (counted over the pair's whole sequence) uses slot
    // i % STAGES and group barrier (i / GROUP) % NGROUPS, whose phase is
    // i / STAGES.
    auto full = [&](uint32_t i) { return bar(static_cast<int>((i / GROUP) % NGROUPS)); };
    auto empty = [&](int s) { return bar(NGROUPS + s); };
    auto raw_full = [&](int r) { return bar(NGROUPS + STAGES + r); };
    auto raw_empty = [&](int r) { return bar(NGROUPS + STAGES + RAW_STAGES + r); };
    const uint32_t d_full = bar(NGROUPS + STAGES + 2 * RAW_STAGES);       // both
    const uint32_t d_empty = bar(NGROUPS + STAGES + 2 * RAW_STAGES + 1);  // leader: 8
    const uint32_t final_bar = bar(NGROUPS + STAGES + 2 * RAW_STAGES + 2);
    int *abort_flag = reinterpret_cast<int *>(sgen + SL::abort_flag);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sgen + SL::tmem_slot);

    if (threadIdx.x == 0) {
        for (int g = 0; g < NGROUPS; ++g) mbar_init_addr(bar(g), GROUP * (2 + 2 * DEQ_PER_STAGE));
        for (int s = 0; s < STAGES; ++s) mbar_init_addr(empty(s), 1);
        for (int r = 0; r < RAW_STAGES; ++r) {
            mbar_init_addr(raw_full(r), 1);
            mbar_init_addr(raw_empty(r), NUM_DEQ_WARPS);
        }
        mbar_init_addr(d_full, 1);
        mbar_init_addr(d_empty, 2 * NUM_EPI_WARPS);
        mbar_init_addr(final_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == WARP_MMA) tmem_alloc_pair(sbase + SL::tmem_slot, TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    cluster_barrier();  // the peer's barriers exist before anyone signals them
    tc_fence_after();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t *>(tmem_slot);
    const uint32_t a_col0 = D_COLS;  // A slots follow the accumulator

    pdl_wait();

    // Work items: (pair tile t, K part s), item = t * ksplit + s; an item
    // covers K stages [s * KB, (s + 1) * KB).
    const int KB = p.k / BK / p.ksplit;     // K stages per item
    const int KR = p.k / RAW_K / p.ksplit;  // raw stages per item
    const int num_items = p.num_tiles * p.ksplit;

    if (warp == WARP_PRODUCER) {
        if (lane == 0) {
            // X tiles: this CTA's 128 tokens of the pair tile
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_x)) : "memory");
            uint32_t it = 0;
            bool ok = true;
            for (int item = pair; ok && item < num_items; item += num_pairs) {
                const int t = item / p.ksplit;
                const int kb0 = (item - t * p.ksplit) * KB;
                const int tb = t % p.num_t_blocks;
                const int xrow = tb * BT + static_cast<int>(rank) * BT_CTA;
                for (int kb = 0; kb < KB; ++kb) {
                    const int s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1u;
                    if (!wait_or_abort(empty(s), ph ^ 1u, abort_flag, ctx)) { ok = false; break; }
                    const uint32_t xf = map_to_rank(full(it), 0);
                    mbar_expect_tx_cluster(xf, X_STAGE_BYTES);
                    tma_load_2d_pair(sbase + SL::x + s * X_STAGE_BYTES, &tmap_x, (kb0 + kb) * BK, xrow, xf);
                    ++it;
                }
            }
            if (leader) {  // X copies of both CTAs complete on the leader's barriers
                for (int s = 0; s < STAGES; ++s) {
                    if (it > static_cast<uint32_t>(s)) {
                        const uint32_t last = it - 1 - ((it - 1 - s) % STAGES);
                        wait_drain(full(last), (last / STAGES) & 1u, ctx);
                    }
                }
            }
        } else if (lane == 1) {
            // raw weight tiles: this CTA's 128 weight rows
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_w)) : "memory");
            if constexpr (G)
                asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_w2))
                             : "memory");
            uint32_t rit = 0;
            bool ok = true;
            for (int item = pair; ok && item < num_items; item += num_pairs) {
                const int t = item / p.ksplit;
                const int kr0 = (item - t * p.ksplit) * KR;
                const int wb = t / p.num_t_blocks;
                // G: this CTA's 64 features, gate rows then up rows
                const int wrow = G ? wb * BW + static_cast<int>(rank) * (BW / 2)
                                   : wb * 2 * BW + static_cast<int>(rank) * BW;
                for (int kr = 0; kr < KR; ++kr) {
                    const int r = rit % RAW_STAGES;
                    const uint32_t ph = (rit / RAW_STAGES) & 1u;
                    if (!wait_or_abort(raw_empty(r), ph ^ 1u, abort_flag, ctx)) { ok = false; break; }
                    mbar_expect_tx_addr(raw_full(r), RAW_STAGE_BYTES);
                    tma_load_2d(sbase + SL::raw + r * RAW_STAGE_BYTES, &tmap_w, (kr0 + kr) * RAW_X,
                                wrow, raw_full(r));
                    if constexpr (G)
                        tma_load_2d(sbase + SL::raw + r * RAW_STAGE_BYTES +
                                        (BW / 2) * RAW_ROW_BYTES,
                                    &tmap_w2, (kr0 + kr) * RAW_X, wrow, raw_full(r));
                    ++rit;
                }
            }
            for (int r = 0; r < RAW_STAGES; ++r) {
                if (rit > static_cast<uint32_t>(r)) {
                    const uint32_t last = rit - 1 - ((rit - 1 - r) % RAW_STAGES);
                    wait_drain(raw_full(r), (last / RAW_STAGES) & 1u, ctx);
                }
            }
        }
    } else if (warp == WARP_MMA) {
        if (leader && lane == 0) {
            // one flat sequence of K stages over this pair's tiles; the wait
            // for stage g+1 is placed after MMA LOOKAHEAD_KK of stage g, so
            // that its latency overlaps the MMAs still queued in the pipe.
            // This thread shares its scheduler with two dequantiser warps, so
            // its path between MMAs is kept short: the K stage, ring slot,
            // descriptors and barrier addresses are advanced incrementally
            // (no run-time division), which measured as the pipeline's pace.
            const uint32_t my_items =
                pair < num_items ? static_cast<uint32_t>((num_items - pair + num_pairs - 1) / num_pairs) : 0u;
            const uint32_t total = my_items * static_cast<uint32_t>(KB);
            const uint64_t bdesc0 = sw128_desc(sbase + SL::x);
            const uint32_t a0 = tmem_base + a_col0;
            const uint32_t empty0 = empty(0);
            uint32_t tiles_done = 0;
            bool issued = false;
            bool ok = total == 0 || MMA_WAIT(full(0u), 0u, abort_flag, ctx);
            uint32_t kb = 0, s = 0;   // K stage within the tile, ring slot
            uint64_t bdesc = bdesc0;  // B (X) descriptor of slot s
            uint32_t a_tmem = a0;     // A columns of slot s
            for (uint32_t g = 0; ok && g < total; ++g) {
                if (kb == 0 && !wait_or_abort_cluster(d_empty, (tiles_done & 1u) ^ 1u, abort_flag, ctx))
                    break;
                tc_fence_after();
                const bool group_end = (g & (GROUP - 1)) == GROUP - 1 && g + 1 < total;
#pragma unroll
                for (int kk = 0; kk < BK / UMMA_K; ++kk) {
                    // K step kk: 8 TMEM columns of A, 32 bytes along the swizzle row of B
                    umma_bf16_pair_ta(tmem_base, a_tmem + (UMMA_K / 2) * kk, bdesc + 2 * kk, kIdesc,
                                      (kk != 0 || kb != 0) ? 1u : 0u);
                    if (kk == LOOKAHEAD_KK && group_end) {
                        const uint32_t g1 = g + 1;  // first stage of the next group
                        ok = MMA_WAIT(full(g1), (g1 / STAGES) & 1u, abort_flag, ctx);
                    }
                }
                issued = true;
                umma_commit_pair(empty0 + 8u * s);
                if (++kb == static_cast<uint32_t>(KB)) {
                    umma_commit_pair(d_full);
                    ++tiles_done;
                    kb = 0;
                }
                if (++s == STAGES) {
                    s = 0;
                    bdesc = bdesc0;
                    a_tmem = a0;
                } else {
                    bdesc += X_STAGE_BYTES >> 4;  // descriptor start address in 16-byte units
                    a_tmem += A_COLS;
                }
            }
            if (issued) {  // all MMAs of the pair complete before TMEM is freed
                umma_commit_pair(final_bar);
                wait_drain(final_bar, 0, ctx);
            }
        }
    } else if (warp < WARP_EPI0) {
        // dequantisers: warp w writes TMEM lanes 32*(w%4)..+31 (its weight rows)
        // and block `half` (K 32*half..+31) of every 64-wide K stage of its
        // phase (every stage, or every other with two sets of warps); `it`
        // counts all K stages, so that slots and parities match the MMA's
        const int q = warp & 3;
        const int half = ((warp - WARP_DEQ0) >> 2) & 1;            // warp-uniform
        const int phase = (warp - WARP_DEQ0) / DEQ_PER_STAGE;        // K stages it % DEQ_PHASES
        // weight row of the raw stage written to TMEM lane 32q + lane; G: gate
        // rows of features 16q.. in lanes 0-15, their up rows (stage rows
        // 64..) in lanes 16-31 (each 8-lane phase of the 16-byte reads still
        // covers 8 consecutive 144-byte rows: no bank conflicts)
        const int row = G ? (lane >> 4) * (BW / 2) + q * 16 + (lane & 15) : q * 32 + lane;
        const uint32_t full_leader0 = map_to_rank(bar(0), 0);
        const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + a_col0 +
                                   static_cast<uint32_t>(half * 16);
        const uint32_t flip0 = p.magic | 0x80u, flip1 = p.magic | 0x8000u;  // Q8_0 decode
        (void)flip0;
        (void)flip1;
        uint32_t it = 0, rit = 0;
        bool ok = true;
        for (int item = pair; ok && item < num_items; item += num_pairs) {
            for (int kr = 0; ok && kr < KR; ++kr) {
                const int r = rit % RAW_STAGES;
                if (!warp_wait_or_abort(raw_full(r), (rit / RAW_STAGES) & 1u, abort_flag, ctx)) {
                    ok = false;
                    break;
                }
                // the row's block bytes in windows of 144 bytes (nine 16-byte
                // reads; rows 144 or 272 bytes apart, so each 8-lane phase
                // hits 32 distinct banks): Q4_0 one window for the four K
                // stages, Q8_0 two (bytes 0..143 for K stages 0-1, 128..271
                // for K stages 2-3)
                constexpr int WINDOWS = F == Fmt::Q4_0 ? 1 : 2;
                constexpr int SUBS = (RAW_K / BK) / WINDOWS;  // K stages per window
                const uint8_t *src = sgen + SL::raw + r * RAW_STAGE_BYTES + row * RAW_ROW_BYTES;
#pragma unroll
                for (int win = 0; win < WINDOWS; ++win) {
                    uint32_t wd[36];
#pragma unroll
                    for (int qq = 0; qq < 9; ++qq) {
                        const uint4 v = lds128(src + 128 * win + 16 * qq);
                        wd[4 * qq + 0] = v.x;
                        wd[4 * qq + 1] = v.y;
                        wd[4 * qq + 2] = v.z;
                        wd[4 * qq + 3] = v.w;
                    }
                    if (win == WINDOWS - 1) {  // the raw stage is in registers
                        __syncwarp();
                        if (lane == 0) mbar_arrive_addr(raw_empty(r));
                        ++rit;
                    }
#pragma unroll
                    for (int sub2 = 0; sub2 < SUBS; ++sub2) {
                        const int sub = win * SUBS + sub2;
                        if (DEQ_PHASES > 1 && (sub & (DEQ_PHASES - 1)) != phase) {
                            ++it;  // K stage written by the other set of warps
                            continue;
                        }
                        const int s = it % STAGES;
                        if (!warp_wait_or_abort(empty(s), ((it / STAGES) & 1u) ^ 1u, abort_flag, ctx)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        uint32_t v[16];
                        if constexpr (F == Fmt::Q4_0) {
                            uint4 ch[4];
                            if (half == 0)
                                dequant_words_bf16<0, 4>(wd, 2 * sub, p.magic, ch);
                            else
                                dequant_words_bf16<0, 4>(wd, 2 * sub + 1, p.magic, ch);
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                v[4 * c + 0] = ch[c].x;
                                v[4 * c + 1] = ch[c].y;
                                v[4 * c + 2] = ch[c].z;
                                v[4 * c + 3] = ch[c].w;
                            }
                        } else {
                            // block 2*sub + half starts 34*(2*sub + half) - 128*win
                            // bytes into the window (a constant in each branch)
                            const int o = 68 * sub - 128 * win;
                            if (half == 0)
                                dequant_q8_block_bf16(wd, o, flip0, flip1, v);
                            else
                                dequant_q8_block_bf16(wd, o + 34, flip0, flip1, v);
                        }
                        tmem_st_16cols(lane_base + s * A_COLS, v);
                        tmem_wait_st();
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive_remote(full_leader0 + 8u * ((it / GROUP) % NGROUPS));
                        ++it;
                    }
                    if (!ok) break;
                }
            }
        }
    } else {
        // epilogue: lane i of warp quarter q holds weight row 32q+i; columns are tokens
        const int q = warp & 3;
        constexpr int CPW = (BT / 32) / (NUM_EPI_WARPS / 4);    // 32-column chunks per warp
        const int c0 = ((warp - WARP_EPI0) >> 2) * CPW;
        const uint32_t d_empty_leader = map_to_rank(d_empty, 0);
        uint32_t tiles_done = 0;
        for (int item = pair; item < num_items; item += num_pairs) {
            const int t = item / p.ksplit;
            const int tb = t % p.num_t_blocks, wb = t / p.num_t_blocks;
            if (!warp_wait_or_abort<QMM_GEMM_EPI_SUSPEND_NS>(d_full, tiles_done & 1u, abort_flag, ctx)) break;
            tc_fence_after();
            if constexpr (G) {
                const bool upper = lane >= 16;  // holds the up row; takes columns 16..31
                const int f = wb * BW + static_cast<int>(rank) * (BW / 2) + q * 16 + (lane & 15);
                const bool f_ok = f < p.n;
#pragma unroll 1
                for (int c = c0; c < c0 + CPW; ++c) {
                    uint32_t v[32];
                    tmem_ld_32cols(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + c * 32, v);
                    const int m0 = tb * BT + c * 32 + (upper ? 16 : 0);
                    uint16_t hv[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        // the lower lane passes g of column 16+j, the upper lane u of column j
                        const float other =
                            __shfl_xor_sync(0xFFFFFFFFu, __uint_as_float(upper ? v[j] : v[16 + j]), 16);
                        const float g = upper ? other : __uint_as_float(v[j]);
                        const float u = upper ? __uint_as_float(v[16 + j]) : other;
                        hv[j] = to_bf16(gelu_tanh_fast(g) * u);
                    }
                    if (f_ok) {
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            if (m0 + j < p.m) p.h[static_cast<size_t>(m0 + j) * p.n + f] = hv[j];
                    }
                }
            } else {
                // the whole product, or this item's K part of it
                float *yo = p.ksplit > 1 ? p.part + static_cast<size_t>(item - t * p.ksplit) * p.m * p.n
                                         : p.y;
                const int n = wb * 2 * BW + static_cast<int>(rank) * BW + q * 32 + lane;
                const bool n_ok = n < p.n;
#pragma unroll 1
                for (int c = c0; c < c0 + CPW; ++c) {
                    uint32_t v[32];
                    tmem_ld_32cols(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + c * 32, v);
                    // column j of the accumulator is token tb*BT + j: the leader's 128 tokens
                    // then the peer's 128
                    const int m0 = tb * BT + c * 32;
                    if (n_ok) {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (m0 + j < p.m)
                                yo[static_cast<size_t>(m0 + j) * p.n + n] = __uint_as_float(v[j]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(d_empty_leader);
            ++tiles_done;
        }
    }

    pdl_launch_dependents();
    tc_fence_before();
    __syncthreads();
    cluster_barrier();  // the leader has drained; the peer's shared memory may go
    tc_fence_after();
    if (warp == WARP_MMA) tmem_dealloc_pair(tmem_base, TMEM_COLS);
}

// y = sum of the K parts, in part order (the same order for every output).
// V: 16-byte accesses (y 16-byte aligned and mn % 4 == 0; the parts always
// are), so that each thread has a whole part's float4 of every part in
// flight; otherwise 4-byte ones.
template <bool V>
__global__ void __launch_bounds__(256) splitk_sum_kernel(const float *__restrict__ part,
                                                         float *__restrict__ y, int64_t mn, int ks) {
    pdl_wait();
    pdl_launch_dependents();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t start = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if constexpr (V) {
        const float4 *p4 = reinterpret_cast<const float4 *>(part);
        float4 *y4 = reinterpret_cast<float4 *>(y);
        const int64_t n4 = mn / 4;
        for (int64_t i = start; i < n4; i += stride) {
            float4 v[8];  // ks <= 8: every part's load issued before the adds
#pragma unroll
            for (int s = 0; s < 8; ++s)
                if (s < ks) v[s] = __ldcg(p4 + static_cast<int64_t>(s) * n4 + i);
            float4 acc = v[0];
#pragma unroll
            for (int s = 1; s < 8; ++s) {
                if (s < ks) {
                    acc.x += v[s].x;
                    acc.y += v[s].y;
                    acc.z += v[s].z;
                    acc.w += v[s].w;
                }
            }
            y4[i] = acc;
        }
    } else {
        for (int64_t i = start; i < mn; i += stride) {
            float v[8];
#pragma unroll
            for (int s = 0; s < 8; ++s)
                if (s < ks) v[s] = __ldcg(part + static_cast<int64_t>(s) * mn + i);
            float acc = v[0];
#pragma unroll
            for (int s = 1; s < 8; ++s)
                if (s < ks) acc += v[s];
            y[i] = acc;
        }
    }
}

// K parts for a plain GEMM whose tiles leave most pairs idle: the split (1,
// 2, 4 or 8, dividing the raw stages) that best fills the pairs, if its
// partial products fit `part_bytes`, each part keeps at least four raw stages
// (1024 of K), all its items run in one round, and it fills the pairs
// clearly better than no split.  Shorter parts do not pay back the second
// pass: at 256 x 8192 x 1024 two parts of two stages took 15.9 us against
// 14.0 unsplit.  An item of a split tile is
// its K part (fewer stages, same work per stage), so the fill is the share of
// pair rounds that are busy.  Splits over several rounds would only trim the
// last round's idle pairs, for twice the partial-product traffic: at
// 512 x 8192 x 8192 eight parts took 101 us against 61 us unsplit.
int choose_ksplit(int64_t m, int64_t n, int64_t k, int num_tiles, int pairs, size_t part_bytes) {
    if (num_tiles >= pairs) return 1;
    auto fill = [&](int ks) {
        const int64_t items = static_cast<int64_t>(num_tiles) * ks;
        const int64_t rounds = (items + pairs - 1) / pairs;
        return static_cast<double>(items) / static_cast<double>(rounds * pairs);
    };
    int best = 1;
    double best_fill = fill(1);
    for (int ks = 2; ks <= 8; ks *= 2) {
        if ((k / RAW_K) % ks != 0 || (k / RAW_K) / ks < 4 ||
            static_cast<int64_t>(num_tiles) * ks > pairs)
            break;
        if (static_cast<size_t>(ks) * static_cast<size_t>(m) * static_cast<size_t>(n) * sizeof(float) > part_bytes)
            break;
        const double f = fill(ks);
        if (f > best_fill + 0.05) {
            best = ks;
            best_fill = f;
        }
    }
    return best;
}

// One launch: plain GEMM (w2 == nullptr: y fp32) or the GeGLU form (w gate,
// w2 up: h bf16).  part (plain GEMM, may be null): room for K-split partial
// products; with a split, a second kernel adds them into y.
template <Fmt F, bool G>
cudaError_t launch(const uint8_t *w, const uint8_t *w2, const uint16_t *x, float *y, uint16_t *h,
                   int64_t m, int64_t n, int64_t k, cudaStream_t stream, const LaunchCtx &ctx,
                   float *part = nullptr, size_t part_bytes = 0) {
    if (m > (1 << 30) || n > (1 << 30) || k > (1 << 24)) return cudaErrorInvalidValue;
    CUtensorMap tx, tw, tw2;
    if (!encode_tmap_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, k, m, k * 2, BK, BT_CTA,
                        CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    using RF = RawFmt<F>;
    const uint64_t rowbytes = static_cast<uint64_t>(k / RAW_K) * RF::kRowBytes;
    constexpr uint32_t box_rows = G ? BW / 2 : BW;
    constexpr uint32_t box_x = RF::kRowBytes / RF::kElemBytes;
    if (!encode_tmap_2d(&tw, RF::kType, w, rowbytes / RF::kElemBytes, n, rowbytes, box_x, box_rows))
        return cudaErrorInvalidValue;
    if (G) {
        if (!encode_tmap_2d(&tw2, RF::kType, w2, rowbytes / RF::kElemBytes, n, rowbytes, box_x,
                            box_rows))
            return cudaErrorInvalidValue;
    } else {
        tw2 = tw;
    }
    GemmParams p;
    p.y = y;
    p.h = h;
    p.m = static_cast<int>(m);
    p.n = static_cast<int>(n);
    p.k = static_cast<int>(k);
    p.num_t_blocks = static_cast<int>((m + BT - 1) / BT);
    // weight rows of a pair tile: 256 rows, or 128 features (gate + up rows)
    const int64_t tile_rows = G ? BW : 2 * BW;
    const int nwb = static_cast<int>((n + tile_rows - 1) / tile_rows);
    p.num_tiles = p.num_t_blocks * nwb;
    const int all_pairs = std::max(1, device_sm_count() / 2);
    p.ksplit = (!G && part != nullptr) ? gemm_fused_ksplit(m, n, k, part_bytes) : 1;
    p.part = p.ksplit > 1 ? part : nullptr;
    p.magic = 0x4B000000u;
    p.ctx = ctx;
    constexpr size_t smem = SmemLayout<F>::smem_bytes;
    static int smem_limits[kMaxDevices] = {0};
    cudaError_t e = ensure_smem(gemm_kernel<F, G>, smem, true, smem_limits);
    if (e != cudaSuccess) return e;
    const int pairs = std::min(p.num_tiles * p.ksplit, all_pairs);
    e = launch_kernel(gemm_kernel<F, G>, dim3(2 * pairs), dim3(NUM_THREADS), smem, stream, 2,
                      tx, tw, tw2, p);
    if (e != cudaSuccess || p.ksplit == 1) return e;
    const int64_t mn = m * n;
    const bool vec = mn % 4 == 0 && (reinterpret_cast<uintptr_t>(y) & 15) == 0;
    const int64_t threads = vec ? mn / 4 : mn;
    const unsigned blocks = static_cast<unsigned>(
        std::min<int64_t>((threads + 255) / 256, static_cast<int64_t>(device_sm_count()) * 8));
    return vec ? launch_kernel(splitk_sum_kernel<true>, dim3(blocks), dim3(256), 0, stream, 1,
                               static_cast<const float *>(p.part), y, mn, p.ksplit)
               : launch_kernel(splitk_sum_kernel<false>, dim3(blocks), dim3(256), 0, stream, 1,
                               static_cast<const float *>(p.part), y, mn, p.ksplit);
}

}  // namespace

int gemm_fused_ksplit(int64_t m, int64_t n, int64_t k, size_t part_bytes) {
    if (part_bytes == 0) return 1;
    const int64_t tiles = (m + BT - 1) / BT * ((n + 2 * BW - 1) / (2 * BW));
    return choose_ksplit(m, n, k, static_cast<int>(tiles), std::max(1, device_sm_count() / 2),
                         part_bytes);
}

bool use_two_phase_gemm(int64_t m, int64_t n, int64_t k) {
    const int64_t blocks = (m + BT - 1) / BT;
    if (blocks <= 2) return false;
    return !(blocks <= 4 && gemm_fused_ksplit(m, n, k, fused_part_budget(n, k)) > 1);
}

cudaError_t launch_gemm_q4_0(const uint8_t *w, const uint16_t *x, float *y, int64_t m, int64_t n,
                             int64_t k, cudaStream_t stream, const LaunchCtx &ctx, float *part,
                             size_t part_bytes) {
    return launch<Fmt::Q4_0, false>(w, nullptr, x, y, nullptr, m, n, k, stream, ctx, part, part_bytes);
}

cudaError_t launch_gemm_q8_0(const uint8_t *w, const uint16_t *x, float *y, int64_t m, int64_t n,
                             int64_t k, cudaStream_t stream, const LaunchCtx &ctx, float *part,
                             size_t part_bytes) {
    return launch<Fmt::Q8_0, false>(w, nullptr, x, y, nullptr, m, n, k, stream, ctx, part, part_bytes);
}

cudaError_t launch_gemm_q4_0_geglu(const uint8_t *wg, const uint8_t *wu, const uint16_t *x,
                                   uint16_t *h, int64_t m, int64_t n, int64_t k,
                                   cudaStream_t stream, const LaunchCtx &ctx) {
    return launch<Fmt::Q4_0, true>(wg, wu, x, nullptr, h, m, n, k, stream, ctx);
}

}  // namespace qmm
