// qmm_gemm_ss.cu -- prefill GEMM in two phases for long prompts: the weights
// are dequantised once into a caller-provided bf16 workspace, then a
// tensor-core GEMM reads both operands from shared memory.
//
// Why: the fused kernel (qmm_gemm.cu) dequantises a weight tile again for
// every 256-token block, so at M = 2048 each weight is decoded eight times
// and that integer/fp32 load on the MMA's SMs sets the pipeline's pace (a
// per-role clock trace showed the MMA-issuing thread slowed by it).  Here the
// decode runs once per call (an HBM-bound pass: 0.5625 bytes read and 2
// bytes written per weight, the written copy mostly staying in L2), and the
// GEMM SMs only move tiles and issue MMAs.
//
// Phase 1, dequant_bf16_kernel: one thread per 32-weight block writes
// bf16((nibble-8)*d) (Q4_0) or bf16(q*d) (Q8_0), each the exact fp32 product
// rounded once to nearest even -- the same weights the fused kernel forms.
// GeGLU form: workspace rows are ordered so that each 128-row CTA tile holds,
// per 32-row lane quarter, 16 gate rows then the 16 up rows of the same
// features (the order the epilogue pairs them in).
//
// Phase 2, gemm_ss_kernel: persistent CTA pairs (cluster of 2), 320 threads:
//   warp 0      producer: lane 0 loads the stage's A tile (128 weight rows x
//               64 bf16) and X tile (128 tokens x 64 bf16), 128-byte swizzle,
//               both completing on the leader CTA's barrier.
//   warp 1      MMA issuer (leader): tcgen05.mma.cta_group::2.kind::f16 with
//               A and B from shared-memory descriptors, M = 256 weight rows,
//               N = 256 tokens, K = 16; two 256-column accumulators in TMEM,
//               so that a tile's epilogue overlaps the next tile's MMAs.
//   warps 2-9   epilogue: tcgen05.ld of the finished accumulator, fp32 Y
//               stores (or the GeGLU pairing and bf16 h stores), then a
//               cluster arrive that frees the accumulator.
// Every wait is bounded; a timeout sets the CTA's abort flag, records the
// error, drains the CTA's own copies and MMAs and frees TMEM.
#include "qmm_internal.h"
#include "qmm_tc.cuh"

#include <algorithm>
#include <mutex>

namespace qmm {
namespace {

constexpr int SW = 128;                // weight rows per CTA (MMA M = 256 per pair)
constexpr int ST = 256;                // tokens per pair tile (MMA N)
constexpr int ST_CTA = ST / 2;
constexpr int SK = 64;                 // K per stage (one 128-byte swizzle row)
constexpr int SUMMA_K = 16;
#ifndef QMM_SS_STAGES
#define QMM_SS_STAGES 7
#endif
#ifndef QMM_SS_SPLIT_TAIL
#define QMM_SS_SPLIT_TAIL 1  // 1: a sparse last round runs as 128-token half tiles
#endif
constexpr int SSTAGES = QMM_SS_STAGES;
constexpr int A_TILE_BYTES = SW * SK * 2;      // 16 KB
constexpr int B_TILE_BYTES = ST_CTA * SK * 2;  // 16 KB
constexpr int SSTAGE_BYTES = A_TILE_BYTES + B_TILE_BYTES;
constexpr uint32_t SS_D_COLS = ST;             // one fp32 accumulator
constexpr uint32_t SS_TMEM_COLS = 512;         // two accumulators
static_assert(2 * SS_D_COLS <= SS_TMEM_COLS, "tensor memory budget");

constexpr int S_WARP_PROD = 0;
constexpr int S_WARP_MMA = 1;
constexpr int S_WARP_EPI0 = 2;
#ifndef QMM_SS_EPI_WARPS
#define QMM_SS_EPI_WARPS 8
#endif
constexpr int S_EPI = QMM_SS_EPI_WARPS;  // 4 or 8: one or two per lane quarter
static_assert(S_EPI == 4 || S_EPI == 8, "epilogue warps");
constexpr int S_THREADS = (S_WARP_EPI0 + S_EPI) * 32;

struct SsLayout {
    static constexpr int bars = SSTAGES * SSTAGE_BYTES;
    // full [SSTAGES] (leader), empty [SSTAGES] (both), d_full [2] (both),
    // d_empty [2] (leader), final
    static constexpr int nbars = 2 * SSTAGES + 5;
    static constexpr int tmem_slot = bars + nbars * 8;
    static constexpr int abort_flag = tmem_slot + 4;
    static constexpr int total = abort_flag + 4;
    static constexpr size_t smem_bytes = total + 1024;  // + alignment slack
};
static_assert(SsLayout::smem_bytes <= 232448, "shared memory per CTA");

// kind::f16: D fp32, A and B bf16, both K-major, M = 256 (the pair), N = 256
// tokens (a full tile) or 128 (a half tile of the last round).
constexpr uint32_t ss_idesc(int n_tokens) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n_tokens >> 3) << 17) |
           (static_cast<uint32_t>((2 * SW) >> 4) << 24);
}
constexpr uint32_t kSsIdesc = ss_idesc(ST);
constexpr uint32_t kSsIdescHalf = ss_idesc(ST / 2);

struct SsParams {
    float *y;     // plain: fp32 [m][ldy]
    uint16_t *h;  // GeGLU: bf16 [m][n]
    int m, n, k;
    int ldy;      // row stride of y (n, or wider when a call covers a column range)
    int num_t_blocks;  // token blocks of ST
    int num_tiles;     // pair tiles
    int full_items;    // work items 0 .. full_items-1 are whole tiles ...
    int num_items;     // ... the rest are half tiles (128 tokens) of the last round
    LaunchCtx ctx;
};

// Work item w of the persistent schedule: a whole tile, or -- when the last
// round would leave most pairs idle -- one 128-token half of a tile.
struct SsItem {
    int tb, wb;   // token block, weight block
    int tok0;     // first token
    bool half;    // 128 tokens instead of 256
};
__device__ __forceinline__ SsItem ss_item(const SsParams &p, int w) {
    SsItem it;
    int t = w, hh = 0;
    it.half = w >= p.full_items;
    if (it.half) {
        t = p.full_items + ((w - p.full_items) >> 1);
        hh = (w - p.full_items) & 1;
    }
    it.tb = t % p.num_t_blocks;
    it.wb = t / p.num_t_blocks;
    it.tok0 = it.tb * ST + hh * (ST / 2);
    return it;
}

// D (TMEM) += A (shared-memory descriptor) x B (shared-memory descriptor),
// both CTAs' halves.
__device__ __forceinline__ void umma_bf16_pair_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                                  uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// ---- phase 1: block-format weights -> bf16 rows ------------------------------

// Workspace row `orow` of the GeGLU form: CTA tile fb = orow / 128 holds
// features fb*64 .. fb*64+63; in lane quarter q (32 rows) the first 16 rows
// are gate rows of features fb*64 + 16q .. +15, the next 16 the up rows of
// the same features.
__device__ __forceinline__ int64_t geglu_source_row(int64_t orow, bool *up) {
    const int64_t fb = orow >> 7;
    const int r = static_cast<int>(orow & 127);
    *up = (r & 16) != 0;
    return fb * 64 + (r >> 5) * 16 + (r & 15);
}

// One thread per 32-weight block.  The block's bytes (2-byte aligned) are
// read as 16-bit words into the word layout the exact decode helpers take
// (d in the low half of word 0, quants from byte 2); its 64 bytes of bf16 go
// through shared memory so that each warp store writes 512 contiguous bytes
// (a 256-thread CTA covers 256 consecutive blocks = 16 KB of output, because
// workspace rows are exactly K weights long).  Grid-stride over CTA groups.
constexpr int kDeqThreads = 256;
constexpr int kDeqStageRow = kDeqThreads + 2;  // 16-byte pieces per row: 258 keeps reads conflict-free

template <Fmt F, bool G>
__global__ void __launch_bounds__(kDeqThreads) dequant_bf16_kernel(const uint8_t *__restrict__ w,
                                                                   const uint8_t *__restrict__ w2,
                                                                   uint16_t *__restrict__ out,
                                                                   int64_t n, int64_t k,
                                                                   int64_t out_rows, uint32_t magic) {
    constexpr int kBB = F == Fmt::Q4_0 ? kQ4_0Bytes : kQ8_0Bytes;
    constexpr int NH = kBB / 2;            // 16-bit words of a block: 9 or 17
    constexpr int NW = (NH + 1) / 2;       // 32-bit words: 5 or 9
    __shared__ uint4 stage[4 * kDeqStageRow];  // piece q of thread t at [q][t]
    // the workspace may still be read by the preceding GEMM of this stream
    pdl_wait();
    const int64_t nb = k / kQK;
    const int64_t total = out_rows * nb;
    const int t = threadIdx.x;
    for (int64_t base = static_cast<int64_t>(blockIdx.x) * kDeqThreads; base < total;
         base += static_cast<int64_t>(gridDim.x) * kDeqThreads) {
        const int64_t idx = base + t;
        uint4 o[4] = {make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u),
                      make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u)};
        if (idx < total) {
            const int64_t orow = idx / nb, b = idx - orow * nb;
            int64_t srow = orow;
            const uint8_t *src = w;
            if constexpr (G) {
                bool up;
                srow = geglu_source_row(orow, &up);
                src = up ? w2 : w;
            }
            if (srow < n) {  // rows past N stay zero weights
                const uint16_t *h = reinterpret_cast<const uint16_t *>(src + (srow * nb + b) * kBB);
                uint32_t wd[NW];
#pragma unroll
                for (int i = 0; i < NW; ++i) {
                    const uint32_t lo = __ldg(h + 2 * i);
                    const uint32_t hi = 2 * i + 1 < NH ? static_cast<uint32_t>(__ldg(h + 2 * i + 1)) : 0u;
                    wd[i] = lo | (hi << 16);
                }
                if constexpr (F == Fmt::Q4_0) {
                    uint32_t w36[36];  // block 0 of a chunk window: only words 0..4 are read
#pragma unroll
                    for (int i = 0; i < 36; ++i) w36[i] = i < NW ? wd[i] : 0u;
                    dequant_words_bf16<0, 4>(w36, 0, magic, o);
                } else {
                    uint32_t v[16];
                    dequant_q8_block_bf16(wd, 0, magic | 0x80u, magic | 0x8000u, v);
#pragma unroll
                    for (int q = 0; q < 4; ++q) o[q] = make_uint4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                }
            }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) stage[q * kDeqStageRow + t] = o[q];
        __syncthreads();
        // output piece p (16 bytes) of this group: piece p % 4 of block p / 4
        uint4 *dst = reinterpret_cast<uint4 *>(out + base * kQK);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int pc = t + kDeqThreads * r;
            if (base + pc / 4 < total) dst[pc] = stage[(pc & 3) * kDeqStageRow + (pc >> 2)];
        }
        __syncthreads();
    }
    pdl_launch_dependents();
}

// ---- phase 2: shared-memory-operand GEMM ------------------------------------

template <bool G>
__global__ void __launch_bounds__(S_THREADS, 1)
    gemm_ss_kernel(const __grid_constant__ CUtensorMap tmap_a,
                   const __grid_constant__ CUtensorMap tmap_x,
                   const __grid_constant__ CUtensorMap tmap_x_half, SsParams p) {
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

    auto bar = [&](int i) -> uint32_t { return sbase + SsLayout::bars + 8u * i; };
    auto full = [&](int s) { return bar(s); };
    auto empty = [&](int s) { return bar(SSTAGES + s); };
    auto d_full = [&](int b) { return bar(2 * SSTAGES + b); };
    auto d_empty = [&](int b) { return bar(2 * SSTAGES + 2 + b); };
    const uint32_t final_bar = bar(2 * SSTAGES + 4);
    int *abort_flag = reinterpret_cast<int *>(sgen + SsLayout::abort_flag);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sgen + SsLayout::tmem_slot);

    if (threadIdx.x == 0) {
        for (int s = 0; s < SSTAGES; ++s) {
            mbar_init_addr(full(s), 2);  // one expect-tx arrive per CTA's producer
            mbar_init_addr(empty(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init_addr(d_full(b), 1);
            mbar_init_addr(d_empty(b), 2 * S_EPI);
        }
        mbar_init_addr(final_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == S_WARP_MMA) tmem_alloc_pair(sbase + SsLayout::tmem_slot, SS_TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    cluster_barrier();  // the peer's barriers exist before anyone signals them
    tc_fence_after();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t *>(tmem_slot);

    pdl_wait();  // the workspace and X are written by preceding kernels

    const int KB = p.k / SK;
    const uint32_t my_items =
        pair < p.num_items ? static_cast<uint32_t>((p.num_items - pair + num_pairs - 1) / num_pairs) : 0u;

    if (warp == S_WARP_PROD) {
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_a)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_x)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_x_half)) : "memory");
            uint32_t it = 0;
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int w = pair; ok && w < p.num_items; w += num_pairs) {
                const SsItem item = ss_item(p, w);
                const int arow = item.wb * 2 * SW + static_cast<int>(rank) * SW;
                // this CTA's share of the item's tokens: 128 (whole tile) or 64 (half)
                const int xrow = item.tok0 + static_cast<int>(rank) * (item.half ? ST_CTA / 2 : ST_CTA);
                const uint32_t bytes = item.half ? A_TILE_BYTES + B_TILE_BYTES / 2 : SSTAGE_BYTES;
                const CUtensorMap *xmap = item.half ? &tmap_x_half : &tmap_x;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!wait_or_abort(empty(s), ph ^ 1u, abort_flag, ctx)) {
                        ok = false;
                        break;
                    }
                    const uint32_t xf = map_to_rank(full(s), 0);
                    mbar_expect_tx_cluster(xf, bytes);
                    const uint32_t dst = sbase + s * SSTAGE_BYTES;
                    tma_load_2d_pair(dst, &tmap_a, kb * SK, arow, xf);
                    tma_load_2d_pair(dst + A_TILE_BYTES, xmap, kb * SK, xrow, xf);
                    ++it;
                    if (++s == SSTAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (leader) {  // both CTAs' copies complete on the leader's barriers
                for (int q = 0; q < SSTAGES; ++q) {
                    if (it > static_cast<uint32_t>(q)) {
                        const uint32_t last = it - 1 - ((it - 1 - q) % SSTAGES);
                        wait_drain(full(q), (last / SSTAGES) & 1u, ctx);
                    }
                }
            }
        }
    } else if (warp == S_WARP_MMA) {
        if (leader && lane == 0) {
            const uint32_t total = my_items * static_cast<uint32_t>(KB);
            int w = pair;  // the current work item
            uint32_t idesc = ss_item(p, w).half ? kSsIdescHalf : kSsIdesc;
            const uint64_t desc0 = sw128_desc(sbase);
            constexpr uint64_t kStageStep = SSTAGE_BYTES >> 4;  // descriptor address units
            constexpr uint64_t kBOffset = A_TILE_BYTES >> 4;
            uint32_t kb = 0, tile = 0, buf = 0;
            int s = 0;
            uint32_t ph = 0;
            uint64_t adesc = desc0;
            bool issued = false, ok = true;
            for (uint32_t g = 0; ok && g < total; ++g) {
                if (kb == 0 &&
                    !wait_or_abort_cluster(d_empty(static_cast<int>(buf)), ((tile >> 1) & 1u) ^ 1u,
                                           abort_flag, ctx))
                    break;
                if (!wait_or_abort(full(s), ph, abort_flag, ctx)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + buf * SS_D_COLS;
#pragma unroll
                for (int kk = 0; kk < SK / SUMMA_K; ++kk)  // 32 bytes along the swizzle row
                    umma_bf16_pair_ss(d_tmem, adesc + 2 * kk, adesc + kBOffset + 2 * kk, idesc,
                                      (kk != 0 || kb != 0) ? 1u : 0u);
                issued = true;
                umma_commit_pair(empty(s));
                if (++kb == static_cast<uint32_t>(KB)) {
                    umma_commit_pair(d_full(static_cast<int>(buf)));
                    kb = 0;
                    ++tile;
                    buf ^= 1u;
                    w += num_pairs;
                    if (w < p.num_items) idesc = ss_item(p, w).half ? kSsIdescHalf : kSsIdesc;
                }
                if (++s == SSTAGES) {
                    s = 0;
                    ph ^= 1u;
                    adesc = desc0;
                } else {
                    adesc += kStageStep;
                }
            }
            if (issued) {  // all MMAs of the pair complete before TMEM is freed
                umma_commit_pair(final_bar);
                wait_drain(final_bar, 0, ctx);
            }
        }
    } else {
        // epilogue: lane i of lane quarter q holds accumulator row 32q+i;
        // columns are tokens (the leader's 128, then the peer's)
        const int q = warp & 3;
        constexpr int CPW = (ST / 32) / (S_EPI / 4);  // 32-column chunks per warp (whole tile)
        const int part = (warp - S_WARP_EPI0) >> 2;   // which share of the columns
        uint32_t tile = 0;
        for (int w = pair; w < p.num_items; w += num_pairs, ++tile) {
            const SsItem item = ss_item(p, w);
            const int wb = item.wb;
            // accumulator column j is token tok0 + j (the leader's tokens, then the peer's)
            const int cpw = item.half ? CPW / 2 : CPW;
            const int c0 = part * cpw;
            const int buf = static_cast<int>(tile & 1u);
            if (!warp_wait_or_abort(d_full(buf), (tile >> 1) & 1u, abort_flag, ctx)) break;
            tc_fence_after();
            const uint32_t d_lane = tmem_base + buf * SS_D_COLS + (static_cast<uint32_t>(q * 32) << 16);
            if constexpr (G) {
                const bool upper = lane >= 16;  // holds the up row; takes columns 16..31
                const int f = wb * SW + static_cast<int>(rank) * (SW / 2) + q * 16 + (lane & 15);
                const bool f_ok = f < p.n;
#pragma unroll 1
                for (int c = c0; c < c0 + cpw; ++c) {
                    uint32_t v[32];
                    tmem_ld_32cols(d_lane + c * 32, v);
                    const int m0 = item.tok0 + c * 32 + (upper ? 16 : 0);
                    uint16_t hv[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
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
                const int n = wb * 2 * SW + static_cast<int>(rank) * SW + q * 32 + lane;
                const bool n_ok = n < p.n;
#pragma unroll 1
                for (int c = c0; c < c0 + cpw; ++c) {
                    uint32_t v[32];
                    tmem_ld_32cols(d_lane + c * 32, v);
                    const int m0 = item.tok0 + c * 32;
                    if (n_ok) {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (m0 + j < p.m)
                                p.y[static_cast<size_t>(m0 + j) * p.ldy + n] = __uint_as_float(v[j]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(map_to_rank(d_empty(buf), 0));
        }
    }

    pdl_launch_dependents();
    tc_fence_before();
    __syncthreads();
    cluster_barrier();  // the leader has drained; the peer's shared memory may go
    tc_fence_after();
    if (warp == S_WARP_MMA) tmem_dealloc_pair(tmem_base, SS_TMEM_COLS);
}

// Workspace rows: N (plain) or 128 rows per 64 features (GeGLU).
int64_t workspace_rows(int64_t n, bool geglu) { return geglu ? (n + 63) / 64 * 128 : n; }

// One two-phase product, split into the host work that can fail (tensor-map
// encoding, kernel attributes) and the two launches, so that a caller
// issuing several products can finish every check before launching any.
template <Fmt F, bool G>
struct TwoPhase {
    const uint8_t *w = nullptr, *w2 = nullptr;
    uint16_t *ws = nullptr;
    int64_t n = 0, k = 0, rows = 0;
    unsigned grid1 = 0;
    int pairs = 0;
    CUtensorMap ta, tx, tx_half;
    SsParams p;

    // ldy: row stride of y (0: n).  Launches nothing.
    cudaError_t prepare(const uint8_t *w_, const uint8_t *w2_, const uint16_t *x, float *y,
                        uint16_t *h, int64_t m, int64_t n_, int64_t k_, uint16_t *ws_,
                        const LaunchCtx &ctx, int64_t ldy = 0) {
        if (m > (1 << 30) || n_ > (1 << 30) || k_ > (1 << 24)) return cudaErrorInvalidValue;
        w = w_;
        w2 = w2_;
        ws = ws_;
        n = n_;
        k = k_;
        rows = workspace_rows(n, G);
        const int64_t groups = (rows * (k / kQK) + kDeqThreads - 1) / kDeqThreads;
        grid1 = static_cast<unsigned>(std::min<int64_t>(groups, 8LL * device_sm_count()));
        if (!encode_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ws, k, rows, k * 2, SK, SW,
                            CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_tmap_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, k, m, k * 2, SK, ST_CTA,
                            CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_tmap_2d(&tx_half, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, k, m, k * 2, SK,
                            ST_CTA / 2, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
        p.y = y;
        p.h = h;
        p.m = static_cast<int>(m);
        p.n = static_cast<int>(n);
        p.k = static_cast<int>(k);
        p.ldy = static_cast<int>(ldy > 0 ? ldy : n);
        p.num_t_blocks = static_cast<int>((m + ST - 1) / ST);
        // a pair tile covers 256 workspace rows: 256 outputs, or 128 GeGLU features
        const int64_t per_tile = G ? SW : 2 * SW;
        p.num_tiles = p.num_t_blocks * static_cast<int>((n + per_tile - 1) / per_tile);
        p.ctx = ctx;
        const int pair_count = std::max(1, device_sm_count() / 2);
        // a last round that would leave more than half the pairs idle runs as
        // 128-token halves of its tiles
        const int rem = p.num_tiles % pair_count;
        const bool split =
            QMM_SS_SPLIT_TAIL && p.num_tiles > pair_count && rem > 0 && 2 * rem <= pair_count;
        p.full_items = split ? p.num_tiles - rem : p.num_tiles;
        p.num_items = split ? p.num_tiles + rem : p.num_tiles;
        pairs = std::min(p.num_items, pair_count);
        static int smem_limits[kMaxDevices] = {0};
        return ensure_smem(gemm_ss_kernel<G>, SsLayout::smem_bytes, true, smem_limits);
    }

    cudaError_t launch(cudaStream_t stream) const {
        cudaError_t e = launch_kernel(dequant_bf16_kernel<F, G>, dim3(grid1), dim3(kDeqThreads), 0,
                                      stream, 1, w, w2, ws, n, k, rows, 0x4B000000u);
        if (e != cudaSuccess) return e;
        return launch_kernel(gemm_ss_kernel<G>, dim3(2 * pairs), dim3(S_THREADS),
                             SsLayout::smem_bytes, stream, 2, ta, tx, tx_half, p);
    }
};

template <Fmt F, bool G>
cudaError_t launch_two_phase(const uint8_t *w, const uint8_t *w2, const uint16_t *x, float *y,
                             uint16_t *h, int64_t m, int64_t n, int64_t k, uint16_t *ws,
                             cudaStream_t stream, const LaunchCtx &ctx) {
    TwoPhase<F, G> tp;
    const cudaError_t e = tp.prepare(w, w2, x, y, h, m, n, k, ws, ctx);
    return e != cudaSuccess ? e : tp.launch(stream);
}

// The library's own scratch for qmm_gemm_q4_0_prefill: bf16 weight rows of
// one column chunk at a time (64 MiB: 16384 rows at K = 2048, 256 rows at
// the largest K the entry point accepts).  Every GPU that loads the library
// holds it until the process exits.
constexpr size_t kScratchBytes = size_t(64) << 20;
static __device__ __align__(256) uint16_t g_prefill_scratch[kScratchBytes / sizeof(uint16_t)];
static_assert(kScratchBytes == static_cast<size_t>(kPrefillMaxK) * 2 * (2 * SW),
              "one 256-row chunk at the largest accepted K fills the scratch");

// Device address of the scratch, resolved once per device (with that device
// current) on the first call of the entry point there.  In host code the
// array's name is only a stand-in for the symbol, never a device address.
std::mutex g_scratch_mu;
void *g_scratch_ptr[kMaxDevices] = {};

cudaError_t prefill_scratch(void **out) {
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_prefill_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_gemm_q4_0_prefill(const uint8_t *w, const uint16_t *x, float *y, int64_t m,
                                     int64_t n, int64_t k, cudaStream_t stream,
                                     const LaunchCtx &ctx) {
    if (k > kPrefillMaxK) return cudaErrorInvalidValue;  // the API rejects it first
    if (!use_two_phase_gemm(m, n, k)) {  // one phase; the scratch takes K-split partial products
        void *scratch = nullptr;
        const cudaError_t e = prefill_scratch(&scratch);
        if (e != cudaSuccess) return e;
        // the K-split budget qmm_gemm_q4_0_ws takes too: the same bits
        return launch_gemm_q4_0(w, x, y, m, n, k, stream, ctx, static_cast<float *>(scratch),
                                fused_part_budget(n, k));
    }
    // weight rows per chunk: whole pair tiles that fit the scratch
    const int64_t chunk =
        static_cast<int64_t>(kScratchBytes / (static_cast<size_t>(k) * 2)) / (2 * SW) * (2 * SW);
    void *scratch = nullptr;
    cudaError_t e = prefill_scratch(&scratch);
    if (e != cudaSuccess) return e;
    uint16_t *ws = static_cast<uint16_t *>(scratch);
    const int64_t row_bytes = (k / kQK) * kQ4_0Bytes;
    // every host step that can fail runs before the first launch: here for
    // the last chunk, and in the loop for the first one (every other chunk
    // has the first chunk's shape)
    const int64_t last0 = (n - 1) / chunk * chunk;
    TwoPhase<Fmt::Q4_0, false> tp;
    e = tp.prepare(w + last0 * row_bytes, nullptr, x, y + last0, nullptr, m, n - last0, k, ws,
                   ctx, n);
    if (e != cudaSuccess) return e;
    for (int64_t n0 = 0; n0 < n; n0 += chunk) {
        const int64_t nc = std::min(chunk, n - n0);
        // columns n0 .. n0+nc of y: the chunk's outputs, row stride n
        e = tp.prepare(w + n0 * row_bytes, nullptr, x, y + n0, nullptr, m, nc, k, ws, ctx, n);
        if (e == cudaSuccess) e = tp.launch(stream);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

size_t gemm_workspace_bytes(int64_t n, int64_t k, bool geglu) {
    return static_cast<size_t>(workspace_rows(n, geglu)) * static_cast<size_t>(k) * 2;
}

size_t fused_part_budget(int64_t n, int64_t k) {
    return std::min(kScratchBytes, gemm_workspace_bytes(n, k, false));
}

cudaError_t launch_gemm_two_phase(Fmt fmt, const uint8_t *w, const uint16_t *x, float *y,
                                  int64_t m, int64_t n, int64_t k, uint16_t *ws,
                                  cudaStream_t stream, const LaunchCtx &ctx) {
    return fmt == Fmt::Q4_0
               ? launch_two_phase<Fmt::Q4_0, false>(w, nullptr, x, y, nullptr, m, n, k, ws, stream, ctx)
               : launch_two_phase<Fmt::Q8_0, false>(w, nullptr, x, y, nullptr, m, n, k, ws, stream, ctx);
}

cudaError_t launch_gemm_geglu_two_phase(const uint8_t *wg, const uint8_t *wu, const uint16_t *x,
                                        uint16_t *h, int64_t m, int64_t n, int64_t k, uint16_t *ws,
                                        cudaStream_t stream, const LaunchCtx &ctx) {
    return launch_two_phase<Fmt::Q4_0, true>(wg, wu, x, nullptr, h, m, n, k, ws, stream, ctx);
}

}  // namespace qmm
