// gemm.cu -- block-scaled grouped GEMMs on the 5th-generation tensor cores
// (tcgen05, sm_103a) for the MoE expert layer:
//   pmn_grouped_gemm_nvfp4   forward expert GEMM, NVFP4 x NVFP4      [Layers]
//                            (bf16, fp32 or SwiGLU epilogue)
//   pmn_w1_gemm_swiglu_nvfp4 the w1 GEMM with SwiGLU in its epilogue,
//                            then NVFP4 (4/6) of h            [NVLink], [Cost]
//   pmn_w2_gemm_rht_s2f6     the same with RHT-32 + S2F6 epilogue    [NVLink]
//   pmn_gemm_mxfp8           backward MXFP8 GEMMs, M- or K-grouped   [SR]
// (sections of the page "Thinking Machines ... Inkling 2 Small ... native
// 4-bit forward", arex-research.com), plus the library's status strings,
// device error word and bounded-wait limit.
//
// One persistent kernel per call, one CTA per SM:
//   warp 0      TMA producer: code tiles (128 rows x 128 bytes, 128-byte
//               swizzle) and raw scale tiles into a 3- to 5-stage ring
//   scale-factor warps: put each stage's scale factors into its TMEM slot,
//               then sf_ready.  256-wide NVFP4 tiles: warps 2, 3, 8, 9, one
//               per TMEM sub-partition, tcgen05.st from the raw rows.
//               Otherwise warps 2, 3 (even / odd stage slots) re-lay them
//               into the 32x128-bit form tcgen05.cp expects and copy them.
//   warp 1      one lane issues the MMAs of a stage once its scale factors
//               are in TMEM, committing to the stage's empty barrier
//   warps 4..   epilogue (4, or 8 on the K-grouped fp32 tiles): TMEM ->
//               registers (one row per thread), outer scales, bf16/fp32,
//               SwiGLU or RHT + S2F6, staged in shared memory and written by
//               TMA tensor stores in full 128-byte lines (the 32-row tiles of
//               short segments store their rows directly)
// 128-wide tiles hold two TMEM accumulators, so the epilogue of one tile
// overlaps the main loop of the next; 256-wide tiles hold one and release it
// as soon as it has been read.  Every wait is bounded: on timeout a device
// error bit is latched and the CTA winds down (no trap).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "../../include/pmn.h"
#include "numerics.cuh"
#include "sm100.cuh"

using namespace pmn;
using namespace pmn::sm100;

__device__ int g_pmn_device_error = 0;

// Wall-time limit of the library's bounded device waits, read at each launch.
static std::atomic<uint64_t> g_wait_limit_ns{4000000000ull};
uint64_t pmn_wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }

extern "C" uint64_t pmn_set_wait_limit_ns(uint64_t ns) { return g_wait_limit_ns.exchange(ns); }

// Pipeline trace points for profiling builds (-DPMN_TRACE): CTA 0 records
// clock64() at each hand-off; compiled out otherwise.
#ifdef PMN_TRACE
__device__ long long g_pmn_trace[8][256];
extern "C" __attribute__((visibility("default"))) int pmn_trace_copy(long long *host)
{
    return cudaMemcpyFromSymbol(host, g_pmn_trace, sizeof(g_pmn_trace)) == cudaSuccess ? 0 : 1;
}
#define PMN_TRACE_POINT(slot, idx)                                            \
    do {                                                                      \
        if (blockIdx.x == 0 && (idx) < 256) g_pmn_trace[slot][idx] = clock64(); \
    } while (0)
#else
#define PMN_TRACE_POINT(slot, idx) \
    do {                           \
    } while (0)
#endif

namespace {

constexpr int KIND_NVFP4 = 0, KIND_MXFP8 = 1;
constexpr int BM = 128;
constexpr int BN_MIN = 128;  // N-tiles are 128 or 256 columns
#ifndef PMN_GEMM_STAGES  // 128-wide NVFP4 tiles (the w2 GEMM with the RHT + S2F6 epilogue)
#define PMN_GEMM_STAGES 5
#endif
#ifndef PMN_GEMM_STAGES_MXFP8  // 128-wide MXFP8 tiles (problems whose N is not a multiple of 256)
#define PMN_GEMM_STAGES_MXFP8 5
#endif
#ifndef PMN_EPI_BUFS  // 128-wide tiles; one buffer leaves room for a fifth NVFP4 stage (measured: w2 GEMM
#define PMN_EPI_BUFS 1  // 0.99 -> 0.90 ms; dW1 3.89 -> 3.83 ms)
#endif
#ifndef PMN_MAX_GROUPS
#define PMN_MAX_GROUPS 1024
#endif
constexpr int EPI_BUFS = PMN_EPI_BUFS;      // epilogue staging buffers per warp
constexpr int STAGE_OUT_BYTES = 32 * 128;  // one epilogue staging buffer: 32 rows x 128 bytes
constexpr int MAX_GROUPS = PMN_MAX_GROUPS;
constexpr uint32_t TMEM_COLS = 512;

// Per (format, N-tile width) layout.  TBN = 256 tiles hold a single TMEM
// accumulator (two of 256 columns would leave no room for scale factors) and
// three stages; TBN = 128 tiles double-buffer the accumulator.  A stage holds
// the A and B tiles (TMA) and, where TMA brings them (SF_TMA), the raw scale
// rows; otherwise the scale-factor warps read the rows from global memory.
// Global loads win only where a warp-wide load covers few cache lines: MXFP8
// scale rows of the M-grouped 256-wide problems are 48..128 bytes long;
// K-grouped rows are whole token ranges apart, NVFP4 rows are 16 bytes per
// stage.
//
// The MMA reads a stage's scale factors from TMEM in a layout replicated
// into the four 32-lane sub-partitions (column j of a 128-row block holds
// rows 32j .. 32j+31).  Two ways to put them there:
//  - two warps re-lay the rows into 32 x 128-bit chunks in shared memory and
//    tcgen05.cp copies each chunk into all four sub-partitions.  The copies
//    queue in order with the MMAs on the tensor pipe;
//  - SF_ST (256-wide NVFP4 tiles): four warps, one per sub-partition, write
//    the words with tcgen05.st from registers, so the tensor pipe carries
//    only MMAs.  There a stage needs 12 copies against 4 MMAs (measured: w1
//    GEMM 1.29 -> 1.15 ms).  Elsewhere the copies are fewer or the issue
//    slots of two more warps cost more than they save (measured: the
//    128-wide w2 + RHT GEMM 0.89 -> 0.92 ms, MXFP8 dX 1.61 -> 2.18 ms with
//    global scale rows).
//
// EW = 8 (the K-grouped fp32 weight gradients on 256-wide tiles): eight
// epilogue warps, two per TMEM lane quadrant, each owning 128 of the tile's
// 256 columns, so a thread holds its whole half-row of fp32 accumulators in
// registers and the single accumulator is released after four chunk reads.
// Their scale rows come by TMA (K-grouped rows are token ranges apart).
template <int KIND, int TBN, int EW = 4, bool SHORT = false>
struct Cfg {
    static constexpr int RB = TBN / 128;  // 128-row blocks of B
    static constexpr bool SF_TMA = !(KIND == KIND_MXFP8 && TBN == 256 && EW == 4);
#ifndef PMN_SF_ST  // scale factors into TMEM by tcgen05.st (four warps) instead of tcgen05.cp
#define PMN_SF_ST 1
#endif
    static constexpr bool SF_ST = PMN_SF_ST && EW == 4 && KIND == KIND_NVFP4 && TBN == 256;
    // SHORT (M-grouped problems whose segments are a few rows, e.g. a decode
    // batch): a tile covers 32 rows of one segment and only those 32 rows of A
    // (and their scales) are loaded.  The MMA still reads 128 rows of A from
    // the stage; rows 32..127 come from whatever follows in the stage and give
    // accumulator rows that are never stored.  The epilogue stores its rows
    // directly (no staging buffers), so a stage of mostly weight bytes fits
    // five times (256-wide) or eight times (128-wide).
    static constexpr int AM = SHORT ? 32 : BM;  // rows of A per tile (and per stage load)
    static constexpr int A_BYTES = AM * 128;
    // raw scale bytes per row and stage: NVFP4 needs 16; MXFP8 needs 4, which
    // never straddle a 16-byte box because every K start (M-grouped: 0,
    // K-grouped: expert segments aligned to 128) is a multiple of 128
    static constexpr int RAW_W = !SF_TMA ? 0 : 16;
    static constexpr int B_TILE_BYTES = TBN * 128;
    static constexpr int RAW_A = AM * RAW_W, RAW_B = TBN * RAW_W;
    static constexpr int SFT_CHUNKS = KIND == KIND_NVFP4 ? 4 : 1;  // K-step chunks per stage
    static constexpr int SFT_A = SF_ST ? 0 : 512 * SFT_CHUNKS, SFT_B = SF_ST ? 0 : 512 * SFT_CHUNKS * RB;
    static constexpr int SFT_OFF = A_BYTES + B_TILE_BYTES + RAW_A + RAW_B;  // re-laid chunks in a stage
    static constexpr int STAGE_RAW = SFT_OFF + SFT_A + SFT_B;
    static constexpr int STAGE_BYTES = (STAGE_RAW + 1023) / 1024 * 1024;
#ifndef PMN_W256_MX_STAGES  // 256-wide MXFP8 tiles: 4 stages with one epilogue staging buffer per warp
#define PMN_W256_MX_STAGES 4
#endif
#ifndef PMN_KG256_STAGES  // 256-wide K-grouped tiles (EW = 8)
#define PMN_KG256_STAGES 3
#endif
    static constexpr bool DIRECT = SHORT;  // epilogue rows stored straight to global memory
    static constexpr int STAGES = SHORT ? (TBN == 256 ? 5 : 8)
                                  : EW == 8 ? PMN_KG256_STAGES
                                  : TBN == 256 ? (KIND == KIND_MXFP8 ? PMN_W256_MX_STAGES : 3)
                                               : (KIND == KIND_MXFP8 ? PMN_GEMM_STAGES_MXFP8 : PMN_GEMM_STAGES);
    static constexpr int EPI = DIRECT ? 0 : EW == 8 ? 1 : TBN == 256 ? (STAGES == 4 ? 1 : 2) : EPI_BUFS;  // staging buffers per warp
    static_assert(!SHORT || (KIND == KIND_NVFP4 && EW == 4 && SF_TMA && B_TILE_BYTES >= 96 * 128), "short tiles: NVFP4");
    // warps 0..3: producer, MMA, scale factors; then EW epilogue warps; then
    // (SF_ST) the scale-factor warps of sub-partitions 0 and 1
    static constexpr int THREADS = 128 + 32 * EW + (SF_ST ? 64 : 0);
    static constexpr int ACC = TBN == 256 ? 1 : 2;
    static constexpr uint32_t SF_COL0 = ACC * TBN;  // scale factors live after the accumulators
    static constexpr uint32_t SFA_COLS = 4 * SFT_CHUNKS, SFB_COLS = 4 * SFT_CHUNKS * RB;
    static constexpr uint32_t SF_COLS_STAGE = SFA_COLS + SFB_COLS;
    static constexpr int SMEM_BYTES =
        1024 + STAGES * STAGE_BYTES + EW * EPI * STAGE_OUT_BYTES + 1024 + (MAX_GROUPS + 1) * 4;
    static_assert(SF_COL0 + STAGES * SF_COLS_STAGE <= TMEM_COLS, "TMEM budget");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

struct GemmArgs {
    const int32_t *offsets;  // device [groups + 1]
    int groups;
    int group_k;             // 0: M-grouped, 1: K-grouped
    int out_kind;            // PMN_OUT_*
    int64_t m;               // rows of A (M-grouped: total rows)
    int64_t n;
    int64_t k;               // contraction length (K-grouped: total)
    const uint8_t *sa, *sb;  // scale factors of A and B (row-major, one row per operand row)
    int64_t sa_pitch, sb_pitch;
    const float *a_outer;    // NVFP4 only
    const float *b_outer;
    void *out;
    uint8_t *out_sc;
    uint64_t seed;
    float *debug_acc;        // RHT + S2F6 only, optional: the scaled fp32 accumulator [m, n]
    uint64_t wait_ns;        // limit of every bounded wait (pmn_set_wait_limit_ns)
};

struct Tile {
    int g;
    int64_t m0, n0, row_end;
    int64_t kb, ke;
    int nks;  // k-stages (128 bytes of K per stage)
};

// Instruction descriptor of the block-scaled MMA (M = 128, N = TBN, both
// operands K-major): operand formats in bits 7..9 / 10..12, N >> 3 in
// 17..22, scale format in 23 (0 = E4M3, 1 = E8M0), M >> 4 in 24..28, scale
// factor byte ids for B in 4..5 and A in 29..30.
template <int KIND, int TBN>
__device__ __forceinline__ uint32_t make_idesc(uint32_t sf_id)
{
    const uint32_t fmt = KIND == KIND_NVFP4 ? 1u : 0u;  // E2M1 (mxf4nvf4) / E4M3 (mxf8f6f4)
    const uint32_t sfmt = KIND == KIND_NVFP4 ? 0u : 1u;
    return (sf_id << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)(TBN >> 3) << 17) | (sfmt << 23) |
           ((uint32_t)(BM >> 4) << 24) | (sf_id << 29);
}

// Tile t of the grouped problem.  `gc` is the caller's group cursor: every
// role walks its tiles in increasing order, so the group of t is found by
// stepping forward from the group of the previous lookup (a few shared-memory
// reads, against a binary search on the critical path between tiles).
template <int KIND, int TBN, int AM = BM>
__device__ __forceinline__ Tile get_tile(int t, const GemmArgs &p, const int *s_cum, int &gc)
{
    int lo = gc;
    if (s_cum[lo] > t) lo = 0;  // not monotone: restart from the first group
    while (lo + 1 < p.groups && s_cum[lo + 1] <= t) ++lo;
    gc = lo;
    Tile ti;
    ti.g = lo;
    const int local = t - s_cum[lo];
    if (!p.group_k) {
        const int nt = (int)(p.n / TBN);
        const int mi = local / nt, ni = local - mi * nt;  // consecutive tiles: adjacent N-tiles
        ti.m0 = __ldg(p.offsets + lo) + (int64_t)mi * AM;
        ti.n0 = (int64_t)ni * TBN;
        ti.row_end = __ldg(p.offsets + lo + 1);
        if (AM < BM) ti.row_end = min(ti.row_end, ti.m0 + AM);  // rows past the loaded ones are not stored
        ti.kb = 0;
        ti.ke = p.k;
    } else {
        const int nt = (int)(p.n / TBN);
        const int mi = local / nt, ni = local - mi * nt;
        ti.m0 = (int64_t)mi * BM;
        ti.n0 = (int64_t)ni * TBN;
        ti.row_end = p.m;
        ti.kb = __ldg(p.offsets + lo);
        ti.ke = __ldg(p.offsets + lo + 1);
    }
    const int64_t kbytes = KIND == KIND_NVFP4 ? (ti.ke - ti.kb) / 2 : (ti.ke - ti.kb);
    ti.nks = (int)((kbytes + 127) / 128);
    return ti;
}

__device__ __forceinline__ void latch_error(int bit) { atomicOr(&g_pmn_device_error, bit); }


// Copies a stage's re-laid scale-factor chunks from shared memory into the
// stage's TMEM columns (A: one 32x128b.warpx4 copy per K-step; B: one per
// K-step and 128-row block).  Issued by one thread, which then commits.
template <class C>
__device__ __forceinline__ void sf_to_tmem(uint8_t *stages, uint32_t stg, uint32_t tmem)
{
    const uint8_t *sftA = stages + stg * C::STAGE_BYTES + C::SFT_OFF;
    const uint8_t *sftB = sftA + C::SFT_A;
    const uint32_t sfa = tmem + C::SF_COL0 + stg * C::SF_COLS_STAGE;
    const uint32_t sfb = sfa + C::SFA_COLS;
#pragma unroll
    for (int c = 0; c < C::SFT_CHUNKS; ++c) {
        tc_cp_32x128b_warpx4(sfa + 4 * c, smem_desc(smem_u32(sftA + 512 * c), 0, 128, 0));
#pragma unroll
        for (int h = 0; h < C::RB; ++h)
            tc_cp_32x128b_warpx4(sfb + 4 * (c * C::RB + h),
                                 smem_desc(smem_u32(sftB + 512 * (c * C::RB + h)), 0, 128, 0));
    }
}

// Every lane of the warp waits; the outcome is made warp-uniform so that a
// timeout can never split the warp before a .sync.aligned instruction.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns)
{
    const bool ok = mbar_wait(bar, parity, limit_ns);
    return __all_sync(0xFFFFFFFFu, ok) != 0;
}

template <int KIND, int OUT, int TBN, int EW, bool SHORT>
__global__ void __launch_bounds__(Cfg<KIND, TBN, EW, SHORT>::THREADS, 1)
    block_scaled_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                             const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
                             const __grid_constant__ CUtensorMap tmO, const GemmArgs p)
{
    using C = Cfg<KIND, TBN, EW, SHORT>;
    constexpr int STAGES = C::STAGES;
    constexpr bool SWI = OUT == PMN_OUT_SWIGLU_BF16;
    static_assert(EW == 4 || (EW == 8 && OUT == PMN_OUT_F32 && TBN == 256), "eight epilogue warps: fp32, 256-wide");
    static_assert(!SWI || (KIND == KIND_NVFP4 && TBN == 256), "SwiGLU tiles are 256-wide NVFP4 tiles");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *stages = smem;
    uint8_t *staging = smem + STAGES * C::STAGE_BYTES;  // epilogue: 4 warps x EPI x 4 KB
    uint64_t *bars = reinterpret_cast<uint64_t *>(staging + EW * C::EPI * STAGE_OUT_BYTES);
    // barrier slots: full[S], empty[S], sf_ready[S], acc_full[2], acc_empty[2], drain
    const uint32_t bar_full = smem_u32(bars), bar_empty = bar_full + 8 * STAGES;
    const uint32_t bar_sfr = bar_empty + 8 * STAGES;  // scale factors re-laid for the stage
    const uint32_t bar_acc_full = bar_sfr + 8 * STAGES, bar_acc_empty = bar_acc_full + 16;
    const uint32_t bar_drain = bar_acc_empty + 16;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 3 * STAGES + 5);
    int *s_abort = reinterpret_cast<int *>(tmem_slot + 1);
    int *s_total = s_abort + 1;
    int *s_cum = reinterpret_cast<int *>(staging + EW * C::EPI * STAGE_OUT_BYTES + 1024);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
            mbar_init(bar_sfr + 8 * s, C::SF_ST ? 4 : 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_acc_full + 8 * b, 1);
            mbar_init(bar_acc_empty + 8 * b, EW);
        }
        mbar_init(bar_drain, 1);
        *s_abort = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        if (C::SF_TMA) {
            tma_prefetch_desc(&tmSA);
            tma_prefetch_desc(&tmSB);
        }
        tma_prefetch_desc(&tmO);
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    if (threadIdx.x == 32) {
        // per-group tile counts and their prefix (tile -> group lookup); the
        // offsets are checked first (monotone, in range, K segments 128-aligned
        // so every stage's scale bytes sit in one 16-byte box) -- bad offsets
        // run no tile and latch PMN_DEVERR_BAD_OFFSETS.  Tiles read the
        // offsets themselves from global memory (cached).
        int cum = 0;
        bool good = true;
        const int64_t limit = p.group_k ? p.k : p.m;
        int prev = 0;
        for (int gi = 0; gi <= p.groups; ++gi) {
            const int o = p.offsets[gi];
            if (o < 0 || o > limit || (gi > 0 && o < prev)) good = false;
            if (p.group_k && (o & 127)) good = false;
            prev = o;
        }
        for (int gi = 0; gi < p.groups && good; ++gi) {
            s_cum[gi] = cum;
            if (!p.group_k) {
                int rows = p.offsets[gi + 1] - p.offsets[gi];
                cum += ((rows + C::AM - 1) / C::AM) * (int)(p.n / TBN);
            } else {
                cum += (int)(p.m / BM) * (int)(p.n / TBN);
            }
        }
        if (good) s_cum[p.groups] = cum;
        *s_total = good ? cum : 0;
        if (!good && blockIdx.x == 0) latch_error(PMN_DEVERR_BAD_OFFSETS);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int total = *s_total;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            uint32_t stage = 0, phase = 0;
            uint32_t issued = 0, last_parity = 0;
            int n_issued = 0, gc = 0;
            for (int t = blockIdx.x; t < total && !*(volatile int *)s_abort; t += gridDim.x) {
                const Tile ti = get_tile<KIND, TBN, C::AM>(t, p, s_cum, gc);
                // SwiGLU tiles: h columns n0/2 .. n0/2 + 127 need the expert's gate
                // rows n0/2 + (0..127) and up rows n/2 + n0/2 + (0..127) of B, loaded
                // as two 128-row boxes into the B tile's two halves
                const int64_t brow = p.group_k ? ti.n0 : (int64_t)ti.g * p.n + (SWI ? ti.n0 / 2 : ti.n0);
                const int64_t brow_up = brow + p.n / 2;
                for (int ks = 0; ks < ti.nks; ++ks) {
                    if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1, p.wait_ns)) {
                        *(volatile int *)s_abort = 1;
                        latch_error(PMN_DEVERR_WAIT_TIMEOUT);
                        break;
                    }
                    PMN_TRACE_POINT(0, n_issued);
                    ++n_issued;
                    uint8_t *st = stages + stage * C::STAGE_BYTES;
                    const uint32_t fb = bar_full + 8 * stage;
                    mbar_arrive_expect_tx(fb, C::A_BYTES + C::B_TILE_BYTES + (C::SF_TMA ? (uint32_t)(C::AM + TBN) * 16u : 0u));
                    // 128 bytes of K per stage: 256 fp4 or 128 fp8 values
                    const int32_t xk = (int32_t)(KIND == KIND_NVFP4 ? (int64_t)ks * 128 : ti.kb + (int64_t)ks * 128);
                    tma_load_2d(smem_u32(st), &tmA, fb, xk, (int32_t)ti.m0);
                    tma_load_2d(smem_u32(st + C::A_BYTES), &tmB, fb, xk, (int32_t)brow);
                    if (SWI) tma_load_2d(smem_u32(st + C::A_BYTES + 128 * 128), &tmB, fb, xk, (int32_t)brow_up);
                    if (C::SF_TMA) {
                        // raw scale rows: 16-byte boxes (the MXFP8 stage's 4 bytes at (xk / 32) % 16)
                        const int32_t xs = KIND == KIND_NVFP4 ? ks * 16 : (int32_t)((xk / 32) & ~int32_t(15));
                        const uint32_t rb = smem_u32(st + C::A_BYTES + C::B_TILE_BYTES + C::RAW_A);
                        tma_load_2d(smem_u32(st + C::A_BYTES + C::B_TILE_BYTES), &tmSA, fb, xs, (int32_t)ti.m0);
                        tma_load_2d(rb, &tmSB, fb, xs, (int32_t)brow);
                        if (SWI) tma_load_2d(rb + 128 * 16, &tmSB, fb, xs, (int32_t)brow_up);
                    }
                    issued |= 1u << stage;
                    last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            // make sure no copy is still landing in shared memory
            for (int s = 0; s < STAGES; ++s)
                if (issued & (1u << s)) (void)mbar_wait(bar_full + 8 * s, (last_parity >> s) & 1u, 1000000000ull);
        }
    } else if (warp == 2 || warp == 3 || (C::SF_ST && warp >= 4 + EW)) {
        // ---------------------------------------------------- scale factors
        // A stage's scale words, 4-column block by block: block (operand
        // block blk = A or 128-row block h of B, K-step chunk c), lane r0,
        // column r1 = the scale word of row r0 + 32 r1.  SF_ST: each of the
        // four warps writes them into its own TMEM sub-partition and arrives
        // on sf_ready after its stores complete.  Otherwise they are written
        // as 32 x 128-bit chunks to shared memory, copied by tcgen05.cp, and
        // the copies' commit is sf_ready.
        const uint32_t tq = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
        auto sf_put = [&](uint32_t stage, int blk, int c, uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3) {
            const int chunk = blk == 0 ? c : c * C::RB + (blk - 1);  // block index within its operand
            if constexpr (C::SF_ST) {
                const uint32_t col = C::SF_COL0 + stage * C::SF_COLS_STAGE + (blk == 0 ? 0u : C::SFA_COLS) + 4 * chunk;
                tmem_st_32x32b_x4(tq + col, w0, w1, w2, w3);
            } else {
                uint8_t *sft = stages + stage * C::STAGE_BYTES + C::SFT_OFF + (blk == 0 ? 0 : C::SFT_A);
                *reinterpret_cast<uint4 *>(sft + chunk * 512 + lane * 16) = make_uint4(w0, w1, w2, w3);
            }
        };
        auto sf_done = [&](uint32_t stage, int seq) {
            if constexpr (C::SF_ST) {
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (warp == 2) PMN_TRACE_POINT(2, seq);  // one sub-partition's arrival
                    mbar_arrive(bar_sfr + 8 * stage);
                }
            } else {
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    PMN_TRACE_POINT(2, seq);
                    tc_fence_after();
                    sf_to_tmem<C>(stages, stage, tmem);  // the kernel's own layout
                    tc_commit(bar_sfr + 8 * stage);  // sf_ready once the copies land
                }
            }
        };
        // without SF_ST, warp 2 takes the even stages of the sequence, warp 3
        // the odd ones; with it, every warp takes every stage
        constexpr uint32_t NSPLIT = C::SF_ST ? 1u : 2u;
        const uint32_t mine = C::SF_ST ? 0u : (uint32_t)(warp - 2);
        if constexpr (C::SF_TMA) {
            // Raw rows arrive with the stage's TMA data: wait for it, re-lay.
            constexpr int raw_w = 16;
            uint32_t stage = 0, phase = 0;
            bool ok = true;
            int n_seq = 0, gc = 0;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const Tile ti = get_tile<KIND, TBN, C::AM>(t, p, s_cum, gc);
                for (int ks = 0; ks < ti.nks; ++ks) {
                    const int seq = n_seq++;
                    if (NSPLIT == 2u && (stage & 1u) != mine) {
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1;
                        }
                        continue;
                    }
                    ok = warp_wait(bar_full + 8 * stage, phase, p.wait_ns);
                    if (!ok || __any_sync(0xFFFFFFFFu, *(volatile int *)s_abort != 0)) {
                        if (!ok && lane == 0) {
                            *(volatile int *)s_abort = 1;
                            latch_error(PMN_DEVERR_WAIT_TIMEOUT);
                        }
                        ok = false;
                        break;
                    }
                    if (lane == 0 && (!C::SF_ST || warp == 2)) PMN_TRACE_POINT(1, seq);
                    uint8_t *st = stages + stage * C::STAGE_BYTES;
                    const uint8_t *rawA = st + C::A_BYTES + C::B_TILE_BYTES, *rawB = rawA + C::RAW_A;
#pragma unroll
                    for (int blk = 0; blk < 1 + C::RB; ++blk) {
                        const int op = blk == 0 ? 0 : 1, h = blk == 0 ? 0 : blk - 1;
                        const uint8_t *raw = (op ? rawB : rawA) + h * 128 * raw_w;
                        if (KIND == KIND_NVFP4) {
                            uint4 w[4];
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                w[j] = *reinterpret_cast<const uint4 *>(raw + (lane + 32 * j) * 16);
#pragma unroll
                            for (int c = 0; c < 4; ++c)
                                sf_put(stage, blk, c, u4_word(w[0], c), u4_word(w[1], c), u4_word(w[2], c),
                                       u4_word(w[3], c));
                        } else {
                            // the stage's 4 scale bytes: word ((k0 / 32) % 16) / 4 of the raw row
                            const int64_t k0 = ti.kb + (int64_t)ks * 128;
                            const int wsel = (int)((k0 / 32) & 15) >> 2;  // warp-uniform
                            uint32_t v[4];
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                v[j] = u4_word(*reinterpret_cast<const uint4 *>(raw + (lane + 32 * j) * raw_w), wsel);
                            sf_put(stage, blk, 0, v[0], v[1], v[2], v[3]);
                        }
                    }
                    sf_done(stage, seq);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
        } else {
            // Rows are read straight from global memory (four per lane and
            // operand block); a warp's loads run two of its stages ahead of
            // the stage it writes, so their latency overlaps the waits.
            constexpr int W = KIND == KIND_NVFP4 ? 4 : 1;  // scale words per row and stage
            constexpr int NR = 4 * (1 + C::RB);  // scale rows one lane fetches
            struct It {
                int t, ks, gc;
                Tile ti;
            };
            auto settle = [&](It &it) {  // first stage at or after (t, ks)
                while (it.t < total && it.ks >= it.ti.nks) {
                    it.t += gridDim.x;
                    it.ks = 0;
                    if (it.t < total) it.ti = get_tile<KIND, TBN, C::AM>(it.t, p, s_cum, it.gc);
                }
            };
            auto fetch = [&](const It &it, uint32_t (&v)[NR][W]) {
                const int64_t brow = p.group_k ? it.ti.n0 : (int64_t)it.ti.g * p.n + it.ti.n0;
#pragma unroll
                for (int j = 0; j < NR; ++j) {
                    const bool opa = j < 4;
                    const int64_t row = opa ? it.ti.m0 + lane + 32 * j : brow + lane + 32 * (j - 4);
                    const bool ok_row = !opa || p.group_k || row < p.m;  // M-grouped A: last tile may pass the end
                    const uint8_t *base = opa ? p.sa : p.sb;
                    const int64_t pitch = opa ? p.sa_pitch : p.sb_pitch;
                    const uint8_t *rp = base + row * pitch;
                    if constexpr (W == 4) {
                        uint4 w = make_uint4(0u, 0u, 0u, 0u);
                        if (ok_row) w = __ldg(reinterpret_cast<const uint4 *>(rp + 16 * it.ks));
                        v[j][0] = w.x;
                        v[j][1] = w.y;
                        v[j][2] = w.z;
                        v[j][3] = w.w;
                    } else if (!p.group_k) {
                        v[j][0] = ok_row ? __ldg(reinterpret_cast<const uint32_t *>(rp + 4 * it.ks)) : 0u;
                    } else {
                        // K segments start at any multiple of 32: the four bytes
                        // may straddle two aligned words; bytes past the row end
                        // are never used (the stage's last K-steps are skipped)
                        const int64_t c0 = (it.ti.kb + (int64_t)it.ks * 128) / 32;
                        const int64_t ca = c0 & ~int64_t(3);
                        const uint32_t w0 = __ldg(reinterpret_cast<const uint32_t *>(rp + ca));
                        const uint32_t w1 =
                            ca + 4 < pitch ? __ldg(reinterpret_cast<const uint32_t *>(rp + ca + 4)) : 0u;
                        v[j][0] = __funnelshift_r(w0, w1, (uint32_t)(c0 & 3) * 8u);
                    }
                }
            };
            // stages of this warp, in order: f is the next one to fetch
            It f{(int)blockIdx.x, 0, 0, Tile{}};
            if (f.t < total) f.ti = get_tile<KIND, TBN, C::AM>(f.t, p, s_cum, f.gc);
            settle(f);
            uint32_t fseq = 0;
            if (mine) {
                ++f.ks;
                settle(f);
                fseq = 1;
            }
            auto prefetch = [&](uint32_t (&v)[NR][W], bool &valid, uint32_t &seq) {
                valid = f.t < total;
                seq = fseq;
                if (valid) fetch(f, v);
#pragma unroll
                for (uint32_t u = 0; u < NSPLIT; ++u) {
                    ++f.ks;
                    settle(f);
                }
                fseq += NSPLIT;
            };
            bool ok = true;
            // write the stage held in `use` (fetched DEPTH - 1 turns earlier),
            // after fetching a later stage into `pre`; register sets rotate by
            // name, so no load result is consumed before its turn comes
            auto turn = [&](uint32_t (&use)[NR][W], bool vuse, uint32_t quse, uint32_t (&pre)[NR][W], bool &vpre,
                            uint32_t &qpre) {
                if (!vuse) return false;
                prefetch(pre, vpre, qpre);
                const uint32_t stage = quse % STAGES, phase = (quse / STAGES) & 1u;
                ok = warp_wait(bar_empty + 8 * stage, phase ^ 1u, p.wait_ns);
                if (!ok || __any_sync(0xFFFFFFFFu, *(volatile int *)s_abort != 0)) {
                    if (!ok && lane == 0) {
                        *(volatile int *)s_abort = 1;
                        latch_error(PMN_DEVERR_WAIT_TIMEOUT);
                    }
                    ok = false;
                    return false;
                }
                if (lane == 0 && (!C::SF_ST || warp == 2)) PMN_TRACE_POINT(1, quse);
#pragma unroll
                for (int blk = 0; blk < 1 + C::RB; ++blk) {
                    // operand block: A, or 128-row block h of B
                    const int j0 = 4 * blk;
#pragma unroll
                    for (int c = 0; c < C::SFT_CHUNKS; ++c)
                        sf_put(stage, blk, c, use[j0][c], use[j0 + 1][c], use[j0 + 2][c], use[j0 + 3][c]);
                }
                sf_done(stage, (int)quse);
                return true;
            };
            uint32_t s0[NR][W], s1[NR][W];
            bool v0, v1;
            uint32_t q0, q1;
            prefetch(s0, v0, q0);
            uint32_t s2[NR][W];
            bool v2;
            uint32_t q2;
            prefetch(s1, v1, q1);
            while (ok) {
                if (!turn(s0, v0, q0, s2, v2, q2)) break;
                if (!turn(s1, v1, q1, s0, v0, q0)) break;
                if (!turn(s2, v2, q2, s1, v1, q1)) break;
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------- MMA issuer
        // One lane issues the MMAs.  The scale-factor warps have already
        // copied the stage's scale factors into its TMEM slot (sf_ready is
        // their commit); a slot is only rewritten after the stage's earlier
        // MMAs completed (their commit freed the stage).
        if (lane == 0) {
            uint32_t stage = 0, phase = 0, abuf = 0, aphase = 0;
            bool ok = true;
            int n_mma = 0;
            // next tile with a non-empty contraction at or after t0 (the
            // epilogue writes the zero product of an empty one by itself)
            int gc = 0;
            auto next_tile = [&](int t0, Tile &out) {
                for (int tt = t0; tt < total; tt += gridDim.x) {
                    out = get_tile<KIND, TBN, C::AM>(tt, p, s_cum, gc);
                    if (out.nks > 0) return tt;
                }
                return total;
            };
            auto fail = [&]() {
                *(volatile int *)s_abort = 1;
                latch_error(PMN_DEVERR_WAIT_TIMEOUT);
                ok = false;
            };
            Tile ti;
            int t = next_tile(blockIdx.x, ti);
            while (ok && t < total) {
                if (!mbar_wait(bar_acc_empty + 8 * abuf, aphase ^ 1, p.wait_ns) || *(volatile int *)s_abort) {
                    if (!*(volatile int *)s_abort) fail();
                    ok = false;
                    break;
                }
                tc_fence_after();
                int tn = total;
                Tile tin;
                const uint32_t d_tmem = tmem + abuf * TBN;
                for (int ks = 0; ks < ti.nks; ++ks) {
                    // the stage's A and B tiles (implied by sf_ready where the
                    // scale-factor warps waited for the stage's TMA data) and
                    // its scale factors in TMEM
                    if ((!C::SF_TMA && !mbar_wait(bar_full + 8 * stage, phase, p.wait_ns)) ||
                        !mbar_wait(bar_sfr + 8 * stage, phase, p.wait_ns)) {
                        fail();
                        break;
                    }
                    tc_fence_after();
                    PMN_TRACE_POINT(3, n_mma);
                    uint8_t *st = stages + stage * C::STAGE_BYTES;
                    const uint32_t sfa = tmem + C::SF_COL0 + stage * C::SF_COLS_STAGE;
                    const uint32_t sfb = sfa + C::SFA_COLS;
                    const uint32_t a_addr = smem_u32(st), b_addr = smem_u32(st + C::A_BYTES);
                    int nk = 4;
                    if (KIND == KIND_MXFP8) {
                        const int64_t left = ti.ke - (ti.kb + (int64_t)ks * 128);
                        nk = left >= 128 ? 4 : (int)(left / 32);
                    }
                    for (int s = 0; s < nk; ++s) {
                        // 32 bytes of K per MMA inside the 128-byte swizzled row
                        const uint64_t ad = smem_desc(a_addr + 32 * s, 16, 1024, 2);
                        const uint64_t bd = smem_desc(b_addr + 32 * s, 16, 1024, 2);
                        const uint32_t acc = (ks > 0 || s > 0) ? 1u : 0u;
                        if (KIND == KIND_NVFP4)
                            mma_nvfp4(d_tmem, ad, bd, make_idesc<KIND, TBN>(0), sfa + 4 * s, sfb + 4 * C::RB * s, acc);
                        else
                            mma_mxfp8(d_tmem, ad, bd, make_idesc<KIND, TBN>((uint32_t)s), sfa, sfb, acc);
                    }
                    tc_commit(bar_empty + 8 * stage);
                    if (ks == ti.nks - 1) tc_commit(bar_acc_full + 8 * abuf);
                    // the next tile is looked up while this stage's MMAs run
                    if (ks == 0) tn = next_tile(t + gridDim.x, tin);
                    PMN_TRACE_POINT(4, n_mma);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                    PMN_TRACE_POINT(5, n_mma);
                    ++n_mma;
                }
                if (++abuf == C::ACC) {
                    abuf = 0;
                    aphase ^= 1;
                }
                t = tn;
                ti = tin;
            }
            // drain: every tcgen05 operation of this thread has completed
            tc_commit(bar_drain);
            (void)mbar_wait(bar_drain, 0, 1000000000ull);
        }
        __syncwarp();
    } else if (warp >= 4 && warp < 4 + EW) {
        // ---------------------------------------------------- epilogue
        // Warp q owns accumulator lanes (rows) 32q .. 32q+31.  A slice whose
        // 32 rows are all valid is staged in shared memory (32 rows x 128 B,
        // 128-byte swizzle, EPI buffers) and written by a TMA tensor store in
        // full 128-byte lines; a slice cut by an expert boundary is written
        // row by row with predicated stores.
        const int q = warp & 3;
        constexpr int CW = TBN / (EW / 4);  // columns per epilogue warp
        const int cb = ((warp - 4) >> 2) * CW;  // the warp's first column in the tile
        uint8_t *stg = staging + (warp - 4) * C::EPI * STAGE_OUT_BYTES;
        // fp32 outputs (the weight gradients, written once) are stored with an
        // L2 evict_last policy: measured 1-2 % faster than the default or
        // evict_first for dW1 / dW2
        uint64_t st_policy = 0;
        if (OUT == PMN_OUT_F32) asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(st_policy));
        constexpr int CH_PER_STORE = OUT == PMN_OUT_F32 ? 1 : ((OUT == PMN_OUT_BF16 || SWI) ? 2 : 4);
        uint32_t nstore = 0;
        uint32_t abuf = 0, aphase = 0;
        int n_epi = 0, gc = 0;
        // RHT: the block signs sigma (the same for every block) are folded into
        // the expert scale, gbs[j] = (-1)^sigma_j * g_e: (acc * g_t) * gbs[j] is
        // exactly the sign-flipped (acc * g_t) * g_e
        const uint32_t sigma = OUT == PMN_OUT_RHT_S2F6 ? rht_sigma(p.seed) : 0u;
        float gbs[OUT == PMN_OUT_RHT_S2F6 ? 32 : 1];
        for (int t = blockIdx.x; t < total; t += gridDim.x) {
            const Tile ti = get_tile<KIND, TBN, C::AM>(t, p, s_cum, gc);
            const int64_t row = ti.m0 + 32 * q + lane;
            const bool valid = row < ti.row_end;
            if (ti.nks == 0) {
                // empty contraction: the product is zero
                if (valid && OUT == PMN_OUT_F32) {
                    float *o = reinterpret_cast<float *>(p.out) + ((int64_t)ti.g * p.m + row) * p.n + ti.n0 + cb;
                    for (int c = 0; c < CW; c += 4) *reinterpret_cast<float4 *>(o + c) = make_float4(0.f, 0.f, 0.f, 0.f);
                } else if (valid && OUT == PMN_OUT_BF16) {
                    uint16_t *o = reinterpret_cast<uint16_t *>(p.out) + ((int64_t)ti.g * p.m + row) * p.n + ti.n0;
                    for (int c = 0; c < TBN; c += 8) *reinterpret_cast<uint4 *>(o + c) = make_uint4(0u, 0u, 0u, 0u);
                } else if (valid && SWI) {  // silu(0) * 0
                    uint16_t *o = reinterpret_cast<uint16_t *>(p.out) + row * (p.n / 2) + ti.n0 / 2;
                    for (int c = 0; c < TBN / 2; c += 8) *reinterpret_cast<uint4 *>(o + c) = make_uint4(0u, 0u, 0u, 0u);
                }
                continue;
            }
            if (!warp_wait(bar_acc_full + 8 * abuf, aphase, p.wait_ns)) {
                if (lane == 0) {
                    *(volatile int *)s_abort = 1;
                    latch_error(PMN_DEVERR_WAIT_TIMEOUT);
                }
                break;
            }
            tc_fence_after();
            if (q == 0 && lane == 0) PMN_TRACE_POINT(6, n_epi);
            const bool slice_any = ti.m0 + 32 * q < ti.row_end;
            const bool slice_full = ti.m0 + 32 * q + 32 <= ti.row_end;
            float scale = 1.0f;
            if (KIND == KIND_NVFP4 && valid) scale = p.a_outer[row];
            const float gb = KIND == KIND_NVFP4 ? p.b_outer[ti.g] : 1.0f;
            if constexpr (OUT == PMN_OUT_RHT_S2F6) {
#pragma unroll
                for (int j = 0; j < 32; ++j) gbs[j] = __uint_as_float(__float_as_uint(gb) ^ (((sigma >> j) & 1u) << 31));
            }
            const int64_t obase = p.group_k ? (int64_t)ti.g * p.m : 0;
            const int64_t orow = obase + row;
            uint64_t sc_word = 0u;
            // The accumulator slice is read 32 columns at a time and converted
            // to the output's bytes.  Where the converted slice fits in
            // registers (at most 128 words a thread: bf16 tiles and 128-wide
            // fp32 tiles) every chunk is read first and the accumulator released
            // to the next tile's MMAs before any store; otherwise (and for the
            // register-hungry RHT + S2F6 conversion) chunks are read, converted
            // and stored in turn and the release follows the last read.
            constexpr int NCH = OUT == PMN_OUT_F32 ? 8 : ((OUT == PMN_OUT_BF16 || SWI) ? 4 : 2);  // 16-byte pieces per chunk
            constexpr int NC = CW / 32;  // 32-column chunks of the warp
            constexpr bool TWO_PHASE = NC * NCH <= 32 && OUT != PMN_OUT_RHT_S2F6 && !SWI;
            const uint32_t tbase = tmem + ((uint32_t)(32 * q) << 16) + abuf * TBN + cb;
            auto convert = [&](uint32_t (&r)[32], int c, uint4 (&o)[NCH]) {
                float v[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
                if constexpr (KIND == KIND_NVFP4 && OUT == PMN_OUT_RHT_S2F6) {
                    // scalar: these products feed the butterfly sums
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __fmul_rn(__fmul_rn(v[j], scale), gbs[j]);
                } else if constexpr (KIND == KIND_NVFP4) {
                    // packed: these products are stored or converted, never summed
#pragma unroll
                    for (int j = 0; j < 32; j += 2) {
                        mul2(v[j], v[j + 1], scale, scale, v[j], v[j + 1]);
                        mul2(v[j], v[j + 1], gb, gb, v[j], v[j + 1]);
                    }
                }
                if constexpr (OUT == PMN_OUT_F32) {
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        o[j] = make_uint4(__float_as_uint(v[4 * j]), __float_as_uint(v[4 * j + 1]),
                                          __float_as_uint(v[4 * j + 2]), __float_as_uint(v[4 * j + 3]));
                } else if constexpr (OUT == PMN_OUT_BF16) {
                    uint32_t w[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        __nv_bfloat162 b2 = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
                        w[j] = *reinterpret_cast<uint32_t *>(&b2);
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j) o[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
                } else {
                    if (p.debug_acc != nullptr && valid) {  // the epilogue's input (signs undone), before the transform
                        float4 *d4 = reinterpret_cast<float4 *>(p.debug_acc + orow * p.n + ti.n0 + 32 * c);
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            float u[4];
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                u[k] = __uint_as_float(__float_as_uint(v[4 * j + k]) ^ (((sigma >> (4 * j + k)) & 1u) << 31));
                            d4[j] = make_float4(u[0], u[1], u[2], u[3]);
                        }
                    }
                    uint32_t qv[8];
                    const uint32_t sb = rht32_s2f6_signed(v, qv);
                    o[0] = make_uint4(qv[0], qv[1], qv[2], qv[3]);
                    o[1] = make_uint4(qv[4], qv[5], qv[6], qv[7]);
                    sc_word |= (uint64_t)sb << (8 * c);
                }
            };
            auto release = [&]() {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(bar_acc_empty + 8 * abuf);
                    if (q == 0) PMN_TRACE_POINT(7, n_epi);
                }
            };
            auto store = [&](int c, const uint4 (&o)[NCH]) {
                const int part = c % CH_PER_STORE;
                if constexpr (!C::DIRECT) {
                    if (slice_full) {
                        uint8_t *buf = stg + (nstore % C::EPI) * STAGE_OUT_BYTES;
                        if (part == 0) {
                            if (lane == 0) bulk_wait_group_read<C::EPI - 1>();  // this buffer's last store has read it
                            __syncwarp();
                        }
#pragma unroll
                        for (int j = 0; j < NCH; ++j) {
                            const int ci = part * NCH + j;
                            *reinterpret_cast<uint4 *>(buf + lane * 128 + ((ci ^ (lane & 7)) << 4)) = o[j];
                        }
                        if (part == CH_PER_STORE - 1) {
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                const int32_t x = (int32_t)((SWI ? ti.n0 / 2 : ti.n0) + cb + 32 * (c - part));
                                const int32_t y = (int32_t)(obase + ti.m0 + 32 * q);
                                if (OUT == PMN_OUT_F32) tma_store_2d_hint(&tmO, smem_u32(buf), x, y, st_policy);
                                else tma_store_2d(&tmO, smem_u32(buf), x, y);
                                bulk_commit_group();
                            }
                            ++nstore;
                        }
                        return;
                    }
                }
                // a slice cut by an expert boundary (and every slice of a
                // 32-row tile) is written row by row
                if (valid) {
                    const int64_t col = (SWI ? ti.n0 / 2 : ti.n0) + cb + 32 * c;
                    uint8_t *o8;
                    if (SWI) o8 = reinterpret_cast<uint8_t *>(reinterpret_cast<uint16_t *>(p.out) + orow * (p.n / 2) + col);
                    else if (OUT == PMN_OUT_F32) o8 = reinterpret_cast<uint8_t *>(reinterpret_cast<float *>(p.out) + orow * p.n + col);
                    else if (OUT == PMN_OUT_BF16) o8 = reinterpret_cast<uint8_t *>(reinterpret_cast<uint16_t *>(p.out) + orow * p.n + col);
                    else o8 = reinterpret_cast<uint8_t *>(p.out) + orow * p.n + col;
#pragma unroll
                    for (int j = 0; j < NCH; ++j) reinterpret_cast<uint4 *>(o8)[j] = o[j];
                }
            };
            // The warp's accumulator slice rounded to bf16 (y = acc * scale * gb
            // for NVFP4), read 16 columns at a time and software-pipelined: the
            // next 16 columns load while the current ones convert, so the
            // read-out before the accumulator's release costs about one load
            // latency per read instead of a load and its wait per chunk.
            auto read_bf16 = [&](uint32_t (&yb)[NC][16]) {
                uint32_t ra[16], rb[16];
                tmem_ld_32x32b_x16(tbase, ra);
                tmem_ld_wait();
#pragma unroll
                for (int h = 0; h < 2 * NC; ++h) {
                    uint32_t(&cur)[16] = (h & 1) ? rb : ra;
                    uint32_t(&nxt)[16] = (h & 1) ? ra : rb;
                    if (h + 1 < 2 * NC) tmem_ld_32x32b_x16(tbase + 16 * (h + 1), nxt);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        float v0 = __uint_as_float(cur[2 * j]), v1 = __uint_as_float(cur[2 * j + 1]);
                        if constexpr (KIND == KIND_NVFP4) {  // packed products feed only the conversion
                            mul2(v0, v1, scale, scale, v0, v1);
                            mul2(v0, v1, gb, gb, v0, v1);
                        }
                        __nv_bfloat162 b2 = __floats2bfloat162_rn(v0, v1);
                        yb[h >> 1][8 * (h & 1) + j] = *reinterpret_cast<uint32_t *>(&b2);
                    }
                    if (h + 1 < 2 * NC) tmem_ld_wait();
                }
            };
            if constexpr (SWI) {
                // accumulator columns 0..127 hold the gate values, 128..255 the up
                // values of the same 128 h columns.  y = acc * g_t * g_e is rounded
                // to bf16 as the bf16 output does (every chunk is read, then the
                // accumulator is released to the next tile's MMAs); h = silu(gate)
                // * up is then formed in binary32 from those bf16 values while the
                // MMAs run -- the same arithmetic as the SwiGLU input mode of the
                // row quantiser, so h equals the unfused path's bit for bit.
                uint32_t yb[NC][16];
                read_bf16(yb);
                release();
                if (slice_any) {
#pragma unroll
                    for (int c = 0; c < NC / 2; ++c) {
                        uint32_t w[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const uint32_t gw = yb[c][j], uw = yb[c + NC / 2][j];
                            float hv[2];
#pragma unroll
                            for (int u = 0; u < 2; ++u) {
                                const float a = __uint_as_float(u ? (gw & 0xFFFF0000u) : (gw << 16));
                                const float b = __uint_as_float(u ? (uw & 0xFFFF0000u) : (uw << 16));
                                hv[u] = silu_mul(a, b);
                            }
                            __nv_bfloat162 b2 = __floats2bfloat162_rn(hv[0], hv[1]);
                            w[j] = *reinterpret_cast<uint32_t *>(&b2);
                        }
                        uint4 o[NCH];
#pragma unroll
                        for (int j = 0; j < 4; ++j) o[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
                        store(c, o);
                    }
                }
            } else if constexpr (TWO_PHASE) {
                uint4 ch[NC][NCH];
                if constexpr (OUT == PMN_OUT_F32) {
                    // fp32: the chunks' words are the output; one wait for all reads
#pragma unroll
                    for (int c = 0; c < NC; ++c) tmem_ld_32x32b_x32(tbase + 32 * c, reinterpret_cast<uint32_t (&)[32]>(ch[c]));
                    tmem_ld_wait();
                    release();
                    if (KIND == KIND_NVFP4) {
#pragma unroll
                        for (int c = 0; c < NC; ++c) convert(reinterpret_cast<uint32_t (&)[32]>(ch[c]), c, ch[c]);
                    }
                } else {
                    uint32_t yb[NC][16];  // bf16: the packed tile
                    read_bf16(yb);
                    release();
#pragma unroll
                    for (int c = 0; c < NC; ++c)
#pragma unroll
                        for (int k = 0; k < NCH; ++k)
                            ch[c][k] = make_uint4(yb[c][4 * k], yb[c][4 * k + 1], yb[c][4 * k + 2], yb[c][4 * k + 3]);
                }
                if (slice_any) {
#pragma unroll
                    for (int c = 0; c < NC; ++c) store(c, ch[c]);
                }
            } else {
#pragma unroll 1
                for (int c = 0; c < NC; ++c) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(tbase + 32 * c, r);
                    tmem_ld_wait();
                    if (c == NC - 1) release();
                    if (!slice_any) continue;
                    uint4 o[NCH];
                    convert(r, c, o);
                    store(c, o);
                }
            }
            if (OUT == PMN_OUT_RHT_S2F6 && valid) {
                if (TBN == 256) *reinterpret_cast<uint64_t *>(p.out_sc + orow * (p.n / 32) + ti.n0 / 32) = sc_word;
                else *reinterpret_cast<uint32_t *>(p.out_sc + orow * (p.n / 32) + ti.n0 / 32) = (uint32_t)sc_word;
            }
            ++n_epi;
            if (++abuf == C::ACC) {
                abuf = 0;
                aphase ^= 1;
            }
        }
        if (lane == 0) bulk_wait_group_all();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
}

// ====================================================================== host
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// 2-D uint8 tensor [rows, width_bytes] with row pitch `pitch` bytes; box
// box_w x 128 rows.
bool make_map(CUtensorMap *m, const void *base, uint64_t width_bytes, uint64_t rows, uint64_t pitch, uint32_t box_w,
              bool swizzle128, uint32_t box_rows = 128)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {width_bytes, rows};
    cuuint64_t strides[1] = {pitch};
    cuuint32_t box[2] = {box_w, box_rows};
    cuuint32_t es[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Output tensor [rows, n] of element size esize for the epilogue's TMA
// stores: box = 128 bytes x 32 rows, 128-byte swizzle.
bool make_out_map(CUtensorMap *m, void *base, int out_kind, uint64_t n, uint64_t rows)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const bool b16 = out_kind == PMN_OUT_BF16 || out_kind == PMN_OUT_SWIGLU_BF16;
    const CUtensorMapDataType dt = out_kind == PMN_OUT_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : b16                   ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                           : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    const uint64_t es = out_kind == PMN_OUT_F32 ? 4 : (b16 ? 2 : 1);
    cuuint64_t dims[2] = {n, rows};
    cuuint64_t strides[1] = {n * es};
    cuuint32_t box[2] = {(cuuint32_t)(128 / es), 32};
    cuuint32_t elem[2] = {1, 1};
    CUresult r = fn(m, dt, 2, base, dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int num_sms()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

// A 2-D uint8 tensor to be loaded by TMA: base, row width and row pitch in
// bytes, rows.
struct MapSpec {
    const void *base;
    uint64_t width_bytes, rows, pitch;
};

struct GemmMaps {
    MapSpec a, b, sa, sb;
};

#ifndef PMN_GEMM_WIDE_KG  // 256-wide tiles with eight epilogue warps for the K-grouped fp32 gradients
#define PMN_GEMM_WIDE_KG 1
#endif
#ifndef PMN_GEMM_WIDE_M  // 256-wide tiles for M-grouped problems
#define PMN_GEMM_WIDE_M 1
#endif
#ifndef PMN_GEMM_SHORT  // 32-row tiles for NVFP4 problems of a few rows per group
#define PMN_GEMM_SHORT 1
#endif

template <int KIND, int OUT, int TBN, int EW = 4, bool SHORT = false>
pmn_status launch_gemm_tbn(const GemmMaps &ms, const CUtensorMap &o, const GemmArgs &args, cudaStream_t s)
{
    using C = Cfg<KIND, TBN, EW, SHORT>;
    CUtensorMap a, b, sa, sb;
    const uint32_t raw_w = 16;  // raw scale rows: one 16-byte box per row and stage
    const uint32_t b_box = OUT == PMN_OUT_SWIGLU_BF16 ? 128 : TBN;  // SwiGLU: gate and up halves load separately
    if (!make_map(&a, ms.a.base, ms.a.width_bytes, ms.a.rows, ms.a.pitch, 128, true, C::AM) ||
        !make_map(&b, ms.b.base, ms.b.width_bytes, ms.b.rows, ms.b.pitch, 128, true, b_box) ||
        !make_map(&sa, ms.sa.base, ms.sa.width_bytes, ms.sa.rows, ms.sa.pitch, raw_w, false, C::AM) ||
        !make_map(&sb, ms.sb.base, ms.sb.width_bytes, ms.sb.rows, ms.sb.pitch, raw_w, false, b_box))
        return PMN_ERR_CUDA;
    GemmArgs ka = args;  // for scale-factor warps that read global memory
    ka.wait_ns = pmn_wait_limit_ns();
    ka.sa = static_cast<const uint8_t *>(ms.sa.base);
    ka.sb = static_cast<const uint8_t *>(ms.sb.base);
    ka.sa_pitch = (int64_t)ms.sa.pitch;
    ka.sb_pitch = (int64_t)ms.sb.pitch;
    auto kern = block_scaled_gemm_kernel<KIND, OUT, TBN, EW, SHORT>;
    const int smem = C::SMEM_BYTES;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return PMN_ERR_CUDA;
    const int sms = num_sms();
    if (sms <= 0) return PMN_ERR_CUDA;
    kern<<<dim3((unsigned)sms), dim3(C::THREADS), smem, s>>>(a, b, sa, sb, o, ka);
    return cudaGetLastError() == cudaSuccess ? PMN_OK : PMN_ERR_CUDA;
}

// Tile width: 256 columns (N = 256 MMAs, half the operand traffic per
// output) for M-grouped problems whose N is a multiple of 256 and whose
// epilogue is a plain conversion; 128 otherwise (K-grouped gradients: short
// per-expert K; the RHT + S2F6 epilogue), with double-buffered accumulators.
template <int KIND, int OUT>
pmn_status launch_gemm(const GemmMaps &ms, const CUtensorMap &o, const GemmArgs &args, cudaStream_t s)
{
    // 256-wide M-grouped tiles except under the RHT + S2F6 epilogue on long
    // segments, whose conversion is long enough that overlapping it with the
    // next tile's MMAs (two 128-wide accumulators) beats the halved A traffic
    // NVFP4 M-grouped problems of a few rows per group (16 or fewer on
    // average, e.g. a decode batch): 32-row tiles (Cfg SHORT)
    const bool tiny_segments = KIND == KIND_NVFP4 && !args.group_k && args.m <= 16 * (int64_t)args.groups;
    if constexpr (OUT == PMN_OUT_SWIGLU_BF16) {
        if (PMN_GEMM_SHORT && tiny_segments) return launch_gemm_tbn<KIND, OUT, 256, 4, true>(ms, o, args, s);
        return launch_gemm_tbn<KIND, OUT, 256>(ms, o, args, s);
    } else if constexpr (KIND == KIND_MXFP8 && OUT == PMN_OUT_F32) {
        // K-grouped weight gradients: 256-wide tiles with eight epilogue warps
        if (PMN_GEMM_WIDE_KG && args.group_k && args.n % 256 == 0)
            return launch_gemm_tbn<KIND, OUT, 256, 8>(ms, o, args, s);
        if (PMN_GEMM_WIDE_M && !args.group_k && args.n % 256 == 0)
            return launch_gemm_tbn<KIND, OUT, 256>(ms, o, args, s);
        return launch_gemm_tbn<KIND, OUT, 128>(ms, o, args, s);
    } else {
        // RHT + S2F6 on short segments (fewer than 64 rows per group on
        // average, e.g. a decode batch): the epilogue has few rows to transform
        // and the wide tile streams twice the weight bytes per stage (decode
        // w2 GEMM 0.298 -> 0.265 ms); the bytes are the same at either width
        const bool short_segments = args.m < 64 * (int64_t)args.groups;
        if constexpr (KIND == KIND_NVFP4 && OUT == PMN_OUT_RHT_S2F6) {
            // 32-row tiles keep two 128-wide accumulators here: only one warp
            // holds the tile's rows, and its RHT overlaps the next tile's MMAs
            if (PMN_GEMM_SHORT && tiny_segments) return launch_gemm_tbn<KIND, OUT, 128, 4, true>(ms, o, args, s);
        }
        if (PMN_GEMM_WIDE_M && (OUT != PMN_OUT_RHT_S2F6 || short_segments) && !args.group_k && args.n % 256 == 0) {
            if constexpr (KIND == KIND_NVFP4 && OUT != PMN_OUT_RHT_S2F6)
                if (PMN_GEMM_SHORT && tiny_segments) return launch_gemm_tbn<KIND, OUT, 256, 4, true>(ms, o, args, s);
            return launch_gemm_tbn<KIND, OUT, 256>(ms, o, args, s);
        }
        return launch_gemm_tbn<KIND, OUT, 128>(ms, o, args, s);
    }
}

pmn_status nvfp4_common(const uint8_t *a_codes, const uint8_t *a_scales, const float *a_outer,
                        const uint8_t *b_codes, const uint8_t *b_scales, const float *b_outer,
                        const int32_t *offsets, int num_experts, int64_t total_rows, int64_t n, int64_t k,
                        int out_kind, void *out, uint8_t *out_sc, uint64_t seed, void *stream,
                        float *debug_acc = nullptr)
{
    if (num_experts <= 0 || num_experts > MAX_GROUPS || total_rows < 0 || n <= 0 || k <= 0) return PMN_ERR_INVALID_ARG;
    if (debug_acc && (out_kind != PMN_OUT_RHT_S2F6 || !aligned16(debug_acc))) return PMN_ERR_INVALID_ARG;
    if (n % BN_MIN != 0 || k % 256 != 0 || total_rows >= (int64_t(1) << 31)) return PMN_ERR_INVALID_ARG;
    if (!a_codes || !a_scales || !a_outer || !b_codes || !b_scales || !b_outer || !offsets || !out)
        return PMN_ERR_INVALID_ARG;
    if (!aligned16(a_codes) || !aligned16(a_scales) || !aligned16(b_codes) || !aligned16(b_scales) ||
        !aligned16(out) || ((uintptr_t)offsets & 3u) || ((uintptr_t)a_outer & 3u) || ((uintptr_t)b_outer & 3u))
        return PMN_ERR_INVALID_ARG;
    if (out_kind == PMN_OUT_RHT_S2F6 && !out_sc) return PMN_ERR_INVALID_ARG;
    if (out_kind == PMN_OUT_SWIGLU_BF16 && n % 256 != 0) return PMN_ERR_INVALID_ARG;
    if (total_rows == 0) return PMN_OK;
    CUtensorMap mo;
    const uint64_t brows = (uint64_t)num_experts * (uint64_t)n;
    if (!make_out_map(&mo, out, out_kind, out_kind == PMN_OUT_SWIGLU_BF16 ? n / 2 : n, total_rows))
        return PMN_ERR_CUDA;
    const uint64_t kb = (uint64_t)k / 2, ks = (uint64_t)k / 16;
    const GemmMaps ms{{a_codes, kb, (uint64_t)total_rows, kb}, {b_codes, kb, brows, kb},
                      {a_scales, ks, (uint64_t)total_rows, ks}, {b_scales, ks, brows, ks}};
    GemmArgs args{};
    args.offsets = offsets;
    args.groups = num_experts;
    args.group_k = 0;
    args.out_kind = out_kind;
    args.m = total_rows;
    args.n = n;
    args.k = k;
    args.a_outer = a_outer;
    args.b_outer = b_outer;
    args.out = out;
    args.out_sc = out_sc;
    args.seed = seed;
    args.debug_acc = debug_acc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    switch (out_kind) {
        case PMN_OUT_BF16: return launch_gemm<KIND_NVFP4, PMN_OUT_BF16>(ms, mo, args, s);
        case PMN_OUT_F32: return launch_gemm<KIND_NVFP4, PMN_OUT_F32>(ms, mo, args, s);
        case PMN_OUT_RHT_S2F6: return launch_gemm<KIND_NVFP4, PMN_OUT_RHT_S2F6>(ms, mo, args, s);
        case PMN_OUT_SWIGLU_BF16: return launch_gemm<KIND_NVFP4, PMN_OUT_SWIGLU_BF16>(ms, mo, args, s);
        default: return PMN_ERR_INVALID_ARG;
    }
}

}  // namespace

// ====================================================================== C ABI
extern "C" int pmn_version(void) { return 100; }

extern "C" const char *pmn_status_string(pmn_status st)
{
    switch (st) {
        case PMN_OK: return "ok";
        case PMN_ERR_INVALID_ARG: return "invalid argument";
        case PMN_ERR_UNSUPPORTED: return "unsupported";
        case PMN_ERR_CUDA: return "CUDA error";
        case PMN_ERR_TIMEOUT: return "device wait timed out";
        default: return "unknown status";
    }
}

pmn_status pmn_take_quant_device_error(cudaStream_t s, int *bits);  // quantize.cu
pmn_status pmn_quantize_h_rows(const uint16_t *h, int64_t rows, int cols, int fos, uint8_t *codes,
                               uint8_t *scales, float *outer, const int32_t *row_end, cudaStream_t s);  // quantize.cu

extern "C" pmn_status pmn_get_device_error(void *stream, int32_t *err)
{
    if (!err) return PMN_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int qbits = 0;
    if (pmn_take_quant_device_error(s, &qbits) != PMN_OK) return PMN_ERR_CUDA;
    int host = 0;
    if (cudaMemcpyFromSymbolAsync(&host, g_pmn_device_error, sizeof(int), 0, cudaMemcpyDeviceToHost, s) !=
        cudaSuccess)
        return PMN_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return PMN_ERR_CUDA;
    const int zero = 0;
    if (host != 0) {
        if (cudaMemcpyToSymbolAsync(g_pmn_device_error, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s) !=
                cudaSuccess ||
            cudaStreamSynchronize(s) != cudaSuccess)
            return PMN_ERR_CUDA;
    }
    *err = host | qbits;
    return PMN_OK;
}

extern "C" pmn_status pmn_grouped_gemm_nvfp4(const uint8_t *a_codes, const uint8_t *a_scales, const float *a_outer,
                                             const uint8_t *b_codes, const uint8_t *b_scales, const float *b_outer,
                                             const int32_t *offsets, int num_experts, int64_t total_rows, int64_t n,
                                             int64_t k, int out_kind, void *out, void *stream)
{
    if (out_kind != PMN_OUT_BF16 && out_kind != PMN_OUT_F32 && out_kind != PMN_OUT_SWIGLU_BF16)
        return PMN_ERR_INVALID_ARG;
    return nvfp4_common(a_codes, a_scales, a_outer, b_codes, b_scales, b_outer, offsets, num_experts, total_rows, n,
                        k, out_kind, out, nullptr, 0, stream);
}

extern "C" pmn_status pmn_w1_gemm_swiglu_nvfp4(const uint8_t *a_codes, const uint8_t *a_scales,
                                               const float *a_outer, const uint8_t *b_codes,
                                               const uint8_t *b_scales, const float *b_outer,
                                               const int32_t *offsets, int num_experts, int64_t total_rows,
                                               int64_t f, int64_t k, int four_over_six, void *h,
                                               uint8_t *codes, uint8_t *scales, float *outer, void *stream)
{
    if (four_over_six != 0 && four_over_six != 1) return PMN_ERR_INVALID_ARG;
    if (f <= 0 || f % 128 != 0 || f > 8192) return PMN_ERR_INVALID_ARG;
    if (!h || !codes || !scales || !outer || !aligned16(h) || !aligned16(codes) || !aligned16(scales) ||
        !aligned16(outer))
        return PMN_ERR_INVALID_ARG;
    const pmn_status st = nvfp4_common(a_codes, a_scales, a_outer, b_codes, b_scales, b_outer, offsets, num_experts,
                                       total_rows, 2 * f, k, PMN_OUT_SWIGLU_BF16, h, nullptr, 0, stream);
    if (st != PMN_OK || total_rows == 0) return st;
    return pmn_quantize_h_rows(static_cast<const uint16_t *>(h), total_rows, (int)f, four_over_six, codes, scales,
                               outer, offsets + num_experts, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" pmn_status pmn_w2_gemm_rht_s2f6(const uint8_t *a_codes, const uint8_t *a_scales, const float *a_outer,
                                           const uint8_t *b_codes, const uint8_t *b_scales, const float *b_outer,
                                           const int32_t *offsets, int num_experts, int64_t total_rows, int64_t n,
                                           int64_t k, uint64_t seed, int8_t *out, uint8_t *out_scales,
                                           float *debug_acc, void *stream)
{
    return nvfp4_common(a_codes, a_scales, a_outer, b_codes, b_scales, b_outer, offsets, num_experts, total_rows, n,
                        k, PMN_OUT_RHT_S2F6, out, out_scales, seed, stream, debug_acc);
}

extern "C" pmn_status pmn_gemm_mxfp8(const uint8_t *a, const uint8_t *a_scales, const uint8_t *b,
                                     const uint8_t *b_scales, const int32_t *offsets, int num_groups, int group_mode,
                                     int64_t m, int64_t n, int64_t k, int out_kind, void *out, void *stream)
{
    if (num_groups <= 0 || num_groups > MAX_GROUPS || m < 0 || n <= 0 || k < 0) return PMN_ERR_INVALID_ARG;
    if (group_mode != PMN_GROUP_M && group_mode != PMN_GROUP_K) return PMN_ERR_INVALID_ARG;
    if (out_kind != PMN_OUT_BF16 && out_kind != PMN_OUT_F32) return PMN_ERR_INVALID_ARG;
    if (n % BN_MIN != 0 || m >= (int64_t(1) << 31) || k >= (int64_t(1) << 31)) return PMN_ERR_INVALID_ARG;
    if (group_mode == PMN_GROUP_M && (k % 128 != 0 || (k / 32) % 16 != 0)) return PMN_ERR_INVALID_ARG;
    if (group_mode == PMN_GROUP_K && (m % BM != 0 || k % 32 != 0 || (k / 32) % 16 != 0)) return PMN_ERR_INVALID_ARG;
    if (!a || !a_scales || !b || !b_scales || !offsets || !out) return PMN_ERR_INVALID_ARG;
    if (!aligned16(a) || !aligned16(a_scales) || !aligned16(b) || !aligned16(b_scales) || !aligned16(out) ||
        ((uintptr_t)offsets & 3u))
        return PMN_ERR_INVALID_ARG;
    if (m == 0) return PMN_OK;
    if (group_mode == PMN_GROUP_M && k == 0) return PMN_ERR_INVALID_ARG;
    const uint64_t brows = group_mode == PMN_GROUP_M ? (uint64_t)num_groups * (uint64_t)n : (uint64_t)n;
    CUtensorMap mo;
    if (k == 0) return PMN_ERR_INVALID_ARG;
    const uint64_t orows = group_mode == PMN_GROUP_M ? (uint64_t)m : (uint64_t)num_groups * (uint64_t)m;
    if (!make_out_map(&mo, out, out_kind, n, orows)) return PMN_ERR_CUDA;
    const uint64_t uk = (uint64_t)k, ks = (uint64_t)k / 32;
    const GemmMaps ms{{a, uk, (uint64_t)m, uk}, {b, uk, brows, uk}, {a_scales, ks, (uint64_t)m, ks},
                      {b_scales, ks, brows, ks}};
    GemmArgs args{};
    args.offsets = offsets;
    args.groups = num_groups;
    args.group_k = group_mode == PMN_GROUP_K;
    args.out_kind = out_kind;
    args.m = m;
    args.n = n;
    args.k = k;
    args.out = out;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (out_kind == PMN_OUT_BF16) return launch_gemm<KIND_MXFP8, PMN_OUT_BF16>(ms, mo, args, s);
    return launch_gemm<KIND_MXFP8, PMN_OUT_F32>(ms, mo, args, s);
}
