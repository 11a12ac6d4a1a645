// gemm.cu -- block-scaled grouped GEMMs on the 5th-generation tensor cores
// (tcgen05, sm_103a) for the MoE expert layer:
//   pmn_grouped_gemm_nvfp4   forward expert GEMM, NVFP4 x NVFP4      [Layers]
//   pmn_w2_gemm_rht_s2f6     the same with RHT-32 + S2F6 epilogue    [NVLink]
//   pmn_gemm_mxfp8           backward MXFP8 GEMMs, M- or K-grouped   [SR]
// (sections of the page "Thinking Machines ... Inkling 2 Small ... native
// 4-bit forward", arex-research.com).
//
// One persistent kernel per call, one CTA per SM, 8 warps:
//   warp 0      TMA producer: code tiles (128 rows x 128 bytes, 128-byte
//               swizzle) and raw scale tiles into a 4-stage ring
//   warp 2      re-lays each stage's scale factors into the 32x128-bit form
//               tcgen05.cp expects (runs ahead of the MMA issuer)
//   warp 1      copies the scale factors to TMEM and issues the MMAs (one
//               elected lane), committing to the stage's empty barrier
//   warps 4..7  epilogue: TMEM -> registers (one row per thread), outer
//               scales, bf16/fp32 or RHT + S2F6, staged in shared memory and
//               written by TMA tensor stores in full 128-byte lines
// Tiles are 128 x 128 with two TMEM accumulators, so the epilogue of one
// tile overlaps the main loop of the next.  Every wait is bounded: on timeout
// a device error bit is latched and the CTA winds down (no trap).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/pmn.h"
#include "numerics.cuh"
#include "sm100.cuh"

using namespace pmn;
using namespace pmn::sm100;

__device__ int g_pmn_device_error = 0;

namespace {

constexpr int KIND_NVFP4 = 0, KIND_MXFP8 = 1;
constexpr int BM = 128, BN = 128;
constexpr int STAGES = 4;
constexpr int STAGE_OUT_BYTES = 32 * 128;  // one epilogue staging buffer: 32 rows x 128 bytes
constexpr int TILE_BYTES = 128 * 128;  // one operand tile: 128 rows x 128 bytes
constexpr int MAX_GROUPS = 1024;
constexpr int NUM_THREADS = 256;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t SF_COL0 = 2 * BN;  // scale factors live after the two accumulators

template <int KIND>
struct Cfg {
    // raw scale tile per operand: 128 rows x RAW_W bytes (TMA, no swizzle)
    static constexpr int RAW_W = KIND == KIND_NVFP4 ? 16 : 32;
    static constexpr int RAW_BYTES = 128 * RAW_W;
    // re-laid scale chunks per operand: one 512-byte chunk per tcgen05.cp
    static constexpr int SFT_CHUNKS = KIND == KIND_NVFP4 ? 4 : 1;
    static constexpr int SFT_BYTES = 512 * SFT_CHUNKS;
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES + 2 * RAW_BYTES + 2 * SFT_BYTES;
    static constexpr uint32_t TX_BYTES = 2 * TILE_BYTES + 2 * RAW_BYTES;
    static constexpr uint32_t SF_COLS_STAGE = 2 * 4 * SFT_CHUNKS;  // A and B, 4 columns per chunk
    static constexpr int SMEM_BYTES =
        1024 + STAGES * STAGE_BYTES + 4 * 2 * STAGE_OUT_BYTES + 1024 + 2 * (MAX_GROUPS + 1) * 4;
};
static_assert(Cfg<KIND_NVFP4>::STAGE_BYTES % 1024 == 0, "stage alignment");
static_assert(Cfg<KIND_MXFP8>::STAGE_BYTES % 1024 == 0, "stage alignment");
static_assert(SF_COL0 + STAGES * Cfg<KIND_NVFP4>::SF_COLS_STAGE <= TMEM_COLS, "TMEM budget");

struct GemmArgs {
    const int32_t *offsets;  // device [groups + 1]
    int groups;
    int group_k;             // 0: M-grouped, 1: K-grouped
    int out_kind;            // PMN_OUT_*
    int64_t m;               // rows of A (M-grouped: total rows)
    int64_t n;
    int64_t k;               // contraction length (K-grouped: total)
    const float *a_outer;    // NVFP4 only
    const float *b_outer;
    void *out;
    uint8_t *out_sc;
    uint64_t seed;
};

struct Tile {
    int g;
    int64_t m0, n0, row_end;
    int64_t kb, ke;
    int nks;  // k-stages (128 bytes of K per stage)
};

// Instruction descriptor of the block-scaled MMA (M = 128, N = 128, both
// operands K-major): operand formats in bits 7..9 / 10..12, N >> 3 in
// 17..22, scale format in 23 (0 = E4M3, 1 = E8M0), M >> 4 in 24..28, scale
// factor byte ids for B in 4..5 and A in 29..30.
template <int KIND>
__device__ __forceinline__ uint32_t make_idesc(uint32_t sf_id)
{
    const uint32_t fmt = KIND == KIND_NVFP4 ? 1u : 0u;  // E2M1 (mxf4nvf4) / E4M3 (mxf8f6f4)
    const uint32_t sfmt = KIND == KIND_NVFP4 ? 0u : 1u;
    return (sf_id << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)(BN >> 3) << 17) | (sfmt << 23) |
           ((uint32_t)(BM >> 4) << 24) | (sf_id << 29);
}

template <int KIND>
__device__ __forceinline__ Tile get_tile(int t, const GemmArgs &p, const int *s_off, const int *s_cum)
{
    int lo = 0, hi = p.groups;
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (s_cum[mid] <= t) lo = mid;
        else hi = mid;
    }
    Tile ti;
    ti.g = lo;
    const int local = t - s_cum[lo];
    if (!p.group_k) {
        const int rows = s_off[lo + 1] - s_off[lo];
        const int mt = (rows + BM - 1) / BM;
        const int ni = local / mt, mi = local - ni * mt;
        ti.m0 = s_off[lo] + (int64_t)mi * BM;
        ti.n0 = (int64_t)ni * BN;
        ti.row_end = s_off[lo + 1];
        ti.kb = 0;
        ti.ke = p.k;
    } else {
        const int nt = (int)(p.n / BN);
        const int mi = local / nt, ni = local - mi * nt;
        ti.m0 = (int64_t)mi * BM;
        ti.n0 = (int64_t)ni * BN;
        ti.row_end = p.m;
        ti.kb = s_off[lo];
        ti.ke = s_off[lo + 1];
    }
    const int64_t kbytes = KIND == KIND_NVFP4 ? (ti.ke - ti.kb) / 2 : (ti.ke - ti.kb);
    ti.nks = (int)((kbytes + 127) / 128);
    return ti;
}

__device__ __forceinline__ void latch_error(int bit) { atomicOr(&g_pmn_device_error, bit); }

// Every lane of the warp waits; the outcome is made warp-uniform so that a
// timeout can never split the warp before a .sync.aligned instruction.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity)
{
    const bool ok = mbar_wait(bar, parity);
    return __all_sync(0xFFFFFFFFu, ok) != 0;
}

template <int KIND, int OUT>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    block_scaled_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                             const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
                             const __grid_constant__ CUtensorMap tmO, const GemmArgs p)
{
    using C = Cfg<KIND>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *stages = smem;
    uint8_t *staging = smem + STAGES * C::STAGE_BYTES;  // epilogue: 4 warps x 2 x 4 KB
    uint64_t *bars = reinterpret_cast<uint64_t *>(staging + 4 * 2 * STAGE_OUT_BYTES);
    // barrier slots: full[S], empty[S], sf_ready[S], acc_full[2], acc_empty[2], drain
    const uint32_t bar_full = smem_u32(bars), bar_empty = bar_full + 8 * STAGES;
    const uint32_t bar_sfr = bar_empty + 8 * STAGES;  // scale factors re-laid for the stage
    const uint32_t bar_acc_full = bar_sfr + 8 * STAGES, bar_acc_empty = bar_acc_full + 16;
    const uint32_t bar_drain = bar_acc_empty + 16;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 3 * STAGES + 5);
    int *s_abort = reinterpret_cast<int *>(tmem_slot + 1);
    int *s_total = s_abort + 1;
    int *s_off = reinterpret_cast<int *>(staging + 4 * 2 * STAGE_OUT_BYTES + 1024);
    int *s_cum = s_off + (MAX_GROUPS + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
            mbar_init(bar_sfr + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_acc_full + 8 * b, 1);
            mbar_init(bar_acc_empty + 8 * b, 4);
        }
        mbar_init(bar_drain, 1);
        *s_abort = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmSA);
        tma_prefetch_desc(&tmSB);
        tma_prefetch_desc(&tmO);
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    if (threadIdx.x == 32) {
        // per-group tile counts and their prefix (tile -> group lookup); the
        // offsets are checked first (monotone, in range, K segments 32-aligned
        // so every TMA coordinate stays 16-byte aligned) -- bad offsets run
        // no tile and latch PMN_DEVERR_BAD_OFFSETS.
        int cum = 0;
        bool good = true;
        const int64_t limit = p.group_k ? p.k : p.m;
        for (int gi = 0; gi <= p.groups; ++gi) {
            s_off[gi] = p.offsets[gi];
            if (s_off[gi] < 0 || s_off[gi] > limit || (gi > 0 && s_off[gi] < s_off[gi - 1])) good = false;
            if (p.group_k && (s_off[gi] & 31)) good = false;
        }
        for (int gi = 0; gi < p.groups; ++gi) {
            s_cum[gi] = cum;
            if (!p.group_k) {
                int rows = s_off[gi + 1] - s_off[gi];
                cum += ((rows + BM - 1) / BM) * (int)(p.n / BN);
            } else {
                cum += (int)(p.m / BM) * (int)(p.n / BN);
            }
        }
        s_cum[p.groups] = cum;
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
            for (int t = blockIdx.x; t < total && !*(volatile int *)s_abort; t += gridDim.x) {
                const Tile ti = get_tile<KIND>(t, p, s_off, s_cum);
                const int64_t brow = p.group_k ? ti.n0 : (int64_t)ti.g * p.n + ti.n0;
                for (int ks = 0; ks < ti.nks; ++ks) {
                    if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1)) {
                        *(volatile int *)s_abort = 1;
                        latch_error(PMN_DEVERR_WAIT_TIMEOUT);
                        break;
                    }
                    uint8_t *st = stages + stage * C::STAGE_BYTES;
                    const uint32_t fb = bar_full + 8 * stage;
                    mbar_arrive_expect_tx(fb, C::TX_BYTES);
                    int32_t xk, xs;
                    if (KIND == KIND_NVFP4) {
                        xk = ks * 128;  // 256 fp4 values per stage
                        xs = ks * 16;   // 16 scale bytes per stage
                    } else {
                        const int64_t k0 = ti.kb + (int64_t)ks * 128;
                        xk = (int32_t)k0;
                        xs = (int32_t)((k0 / 32) & ~int64_t(15));  // 16-byte aligned start
                    }
                    tma_load_2d(smem_u32(st), &tmA, fb, xk, (int32_t)ti.m0);
                    tma_load_2d(smem_u32(st + TILE_BYTES), &tmB, fb, xk, (int32_t)brow);
                    tma_load_2d(smem_u32(st + 2 * TILE_BYTES), &tmSA, fb, xs, (int32_t)ti.m0);
                    tma_load_2d(smem_u32(st + 2 * TILE_BYTES + C::RAW_BYTES), &tmSB, fb, xs, (int32_t)brow);
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
    } else if (warp == 2) {
        // ---------------------------------------------------- scale-factor re-lay
        // Waits for a stage's TMA data, re-lays its scale factors into the
        // 32 x 128-bit chunks tcgen05.cp expects (chunk s, 16-byte line r0 =
        // the scale words of rows r0, r0+32, r0+64, r0+96) and signals
        // sf_ready; it runs up to STAGES stages ahead of the MMA issuer.
        uint32_t stage = 0, phase = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
            const Tile ti = get_tile<KIND>(t, p, s_off, s_cum);
            for (int ks = 0; ks < ti.nks; ++ks) {
                ok = warp_wait(bar_full + 8 * stage, phase);
                if (!ok || __any_sync(0xFFFFFFFFu, *(volatile int *)s_abort != 0)) {
                    if (!ok && lane == 0) {
                        *(volatile int *)s_abort = 1;
                        latch_error(PMN_DEVERR_WAIT_TIMEOUT);
                    }
                    ok = false;
                    break;
                }
                uint8_t *st = stages + stage * C::STAGE_BYTES;
                const uint8_t *rawA = st + 2 * TILE_BYTES, *rawB = rawA + C::RAW_BYTES;
                uint8_t *sftA = st + 2 * TILE_BYTES + 2 * C::RAW_BYTES, *sftB = sftA + C::SFT_BYTES;
                if (KIND == KIND_NVFP4) {
#pragma unroll
                    for (int op = 0; op < 2; ++op) {
                        const uint8_t *raw = op ? rawB : rawA;
                        uint8_t *sft = op ? sftB : sftA;
                        uint4 w[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j) w[j] = *reinterpret_cast<const uint4 *>(raw + (lane + 32 * j) * 16);
                        *reinterpret_cast<uint4 *>(sft + 0 * 512 + lane * 16) = make_uint4(w[0].x, w[1].x, w[2].x, w[3].x);
                        *reinterpret_cast<uint4 *>(sft + 1 * 512 + lane * 16) = make_uint4(w[0].y, w[1].y, w[2].y, w[3].y);
                        *reinterpret_cast<uint4 *>(sft + 2 * 512 + lane * 16) = make_uint4(w[0].z, w[1].z, w[2].z, w[3].z);
                        *reinterpret_cast<uint4 *>(sft + 3 * 512 + lane * 16) = make_uint4(w[0].w, w[1].w, w[2].w, w[3].w);
                    }
                } else {
                    const int64_t k0 = ti.kb + (int64_t)ks * 128;
                    const int rem = (int)((k0 / 32) & 15);  // byte offset of this stage's 4 scales in the raw row
                    const int wsel = rem >> 2, sh = (rem & 3) * 8;  // warp-uniform
#pragma unroll
                    for (int op = 0; op < 2; ++op) {
                        const uint8_t *raw = op ? rawB : rawA;
                        uint8_t *sft = op ? sftB : sftA;
                        uint32_t v[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const uint4 *rw = reinterpret_cast<const uint4 *>(raw + (lane + 32 * j) * 32);
                            const uint4 a0 = rw[0], a1 = rw[1];
                            uint32_t lo, hi;
                            switch (wsel) {
                                case 0: lo = a0.x; hi = a0.y; break;
                                case 1: lo = a0.y; hi = a0.z; break;
                                case 2: lo = a0.z; hi = a0.w; break;
                                default: lo = a0.w; hi = a1.x; break;
                            }
                            v[j] = sh ? __funnelshift_r(lo, hi, sh) : lo;
                        }
                        *reinterpret_cast<uint4 *>(sft + lane * 16) = make_uint4(v[0], v[1], v[2], v[3]);
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_sfr + 8 * stage);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------- MMA issuer
        uint32_t stage = 0, phase = 0, abuf = 0, aphase = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x) {
            const Tile ti = get_tile<KIND>(t, p, s_off, s_cum);
            if (ti.nks == 0) continue;
            bool ok = warp_wait(bar_acc_empty + 8 * abuf, aphase ^ 1);
            const bool aborted = __any_sync(0xFFFFFFFFu, *(volatile int *)s_abort != 0);
            if (!ok || aborted) {
                if (!ok && lane == 0) {
                    *(volatile int *)s_abort = 1;
                    latch_error(PMN_DEVERR_WAIT_TIMEOUT);
                }
                break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem + abuf * BN;
            for (int ks = 0; ks < ti.nks; ++ks) {
                ok = warp_wait(bar_sfr + 8 * stage, phase);
                if (!ok) {
                    if (lane == 0) {
                        *(volatile int *)s_abort = 1;
                        latch_error(PMN_DEVERR_WAIT_TIMEOUT);
                    }
                    break;
                }
                uint8_t *st = stages + stage * C::STAGE_BYTES;
                uint8_t *sftA = st + 2 * TILE_BYTES + 2 * C::RAW_BYTES, *sftB = sftA + C::SFT_BYTES;
                if (lane == 0) {
                    tc_fence_after();
                    const uint32_t sfa = tmem + SF_COL0 + stage * C::SF_COLS_STAGE;
                    const uint32_t sfb = sfa + 4 * C::SFT_CHUNKS;
                    const uint32_t a_addr = smem_u32(st), b_addr = smem_u32(st + TILE_BYTES);
#pragma unroll
                    for (int c = 0; c < C::SFT_CHUNKS; ++c) {
                        tc_cp_32x128b_warpx4(sfa + 4 * c, smem_desc(smem_u32(sftA + 512 * c), 0, 128, 0));
                        tc_cp_32x128b_warpx4(sfb + 4 * c, smem_desc(smem_u32(sftB + 512 * c), 0, 128, 0));
                    }
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
                            mma_nvfp4(d_tmem, ad, bd, make_idesc<KIND>(0), sfa + 4 * s, sfb + 4 * s, acc);
                        else
                            mma_mxfp8(d_tmem, ad, bd, make_idesc<KIND>((uint32_t)s), sfa, sfb, acc);
                    }
                    tc_commit(bar_empty + 8 * stage);
                }
                __syncwarp();
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            if (!ok) break;
            if (lane == 0) tc_commit(bar_acc_full + 8 * abuf);
            __syncwarp();
            if (++abuf == 2) {
                abuf = 0;
                aphase ^= 1;
            }
        }
        // drain: every tcgen05 operation of this thread has completed
        if (lane == 0) {
            tc_commit(bar_drain);
            (void)mbar_wait(bar_drain, 0, 1000000000ull);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ---------------------------------------------------- epilogue
        // Warp q owns accumulator lanes (rows) 32q .. 32q+31.  A slice whose
        // 32 rows are all valid is staged in shared memory (32 rows x 128 B,
        // 128-byte swizzle, two buffers) and written by a TMA tensor store in
        // full 128-byte lines; a slice cut by an expert boundary is written
        // row by row with predicated stores.
        const int q = warp & 3;
        uint8_t *stg = staging + q * 2 * STAGE_OUT_BYTES;
        constexpr int CH_PER_STORE = OUT == PMN_OUT_F32 ? 1 : (OUT == PMN_OUT_BF16 ? 2 : 4);
        uint32_t nstore = 0;
        uint32_t abuf = 0, aphase = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x) {
            const Tile ti = get_tile<KIND>(t, p, s_off, s_cum);
            const int64_t row = ti.m0 + 32 * q + lane;
            const bool valid = row < ti.row_end;
            if (ti.nks == 0) {
                // empty contraction: the product is zero
                if (valid && OUT == PMN_OUT_F32) {
                    float *o = reinterpret_cast<float *>(p.out) + ((int64_t)ti.g * p.m + row) * p.n + ti.n0;
                    for (int c = 0; c < BN; c += 4) *reinterpret_cast<float4 *>(o + c) = make_float4(0.f, 0.f, 0.f, 0.f);
                } else if (valid && OUT == PMN_OUT_BF16) {
                    uint16_t *o = reinterpret_cast<uint16_t *>(p.out) + ((int64_t)ti.g * p.m + row) * p.n + ti.n0;
                    for (int c = 0; c < BN; c += 8) *reinterpret_cast<uint4 *>(o + c) = make_uint4(0u, 0u, 0u, 0u);
                }
                continue;
            }
            if (!warp_wait(bar_acc_full + 8 * abuf, aphase)) {
                if (lane == 0) {
                    *(volatile int *)s_abort = 1;
                    latch_error(PMN_DEVERR_WAIT_TIMEOUT);
                }
                break;
            }
            tc_fence_after();
            const bool slice_any = ti.m0 + 32 * q < ti.row_end;
            const bool slice_full = ti.m0 + 32 * q + 32 <= ti.row_end;
            float scale = 1.0f;
            if (KIND == KIND_NVFP4 && valid) scale = p.a_outer[row];
            const float gb = KIND == KIND_NVFP4 ? p.b_outer[ti.g] : 1.0f;
            const uint32_t sigma = OUT == PMN_OUT_RHT_S2F6 ? rht_sigma(p.seed) : 0u;
            const int64_t obase = p.group_k ? (int64_t)ti.g * p.m : 0;
            const int64_t orow = obase + row;
            uint32_t sc_word = 0u;
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(tmem + ((uint32_t)(32 * q) << 16) + abuf * BN + 32 * c, r);
                tmem_ld_wait();
                if (c == BN / 32 - 1) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar_acc_empty + 8 * abuf);
                }
                if (!slice_any) continue;
                float v[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    v[j] = __uint_as_float(r[j]);
                    if (KIND == KIND_NVFP4) v[j] = __fmul_rn(__fmul_rn(v[j], scale), gb);
                }
                // the 16-byte chunks this 32-column piece contributes to a 128-byte row
                uint4 chunk[8];
                int nch;
                if (OUT == PMN_OUT_F32) {
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        chunk[j] = make_uint4(__float_as_uint(v[4 * j]), __float_as_uint(v[4 * j + 1]),
                                              __float_as_uint(v[4 * j + 2]), __float_as_uint(v[4 * j + 3]));
                    nch = 8;
                } else if (OUT == PMN_OUT_BF16) {
                    uint32_t w[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        __nv_bfloat162 b2 = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
                        w[j] = *reinterpret_cast<uint32_t *>(&b2);
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j) chunk[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
                    nch = 4;
                } else {
                    uint32_t qv[8];
                    const uint32_t sb = rht32_s2f6(v, sigma, qv);
                    chunk[0] = make_uint4(qv[0], qv[1], qv[2], qv[3]);
                    chunk[1] = make_uint4(qv[4], qv[5], qv[6], qv[7]);
                    nch = 2;
                    sc_word |= sb << (8 * c);
                }
                const int part = c % CH_PER_STORE;
                if (slice_full) {
                    uint8_t *buf = stg + (nstore & 1u) * STAGE_OUT_BYTES;
                    if (part == 0) {
                        if (lane == 0) bulk_wait_group_read<1>();  // the older store has left this buffer
                        __syncwarp();
                    }
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        if (j < nch) {
                            const int ci = part * nch + j;
                            *reinterpret_cast<uint4 *>(buf + lane * 128 + ((ci ^ (lane & 7)) << 4)) = chunk[j];
                        }
                    if (part == CH_PER_STORE - 1) {
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            const int32_t x = (int32_t)(ti.n0 + 32 * (c - part));
                            tma_store_2d(&tmO, smem_u32(buf), x, (int32_t)(obase + ti.m0 + 32 * q));
                            bulk_commit_group();
                        }
                        ++nstore;
                    }
                } else if (valid) {
                    const int64_t col = ti.n0 + 32 * c;
                    uint8_t *o;
                    if (OUT == PMN_OUT_F32) o = reinterpret_cast<uint8_t *>(reinterpret_cast<float *>(p.out) + orow * p.n + col);
                    else if (OUT == PMN_OUT_BF16) o = reinterpret_cast<uint8_t *>(reinterpret_cast<uint16_t *>(p.out) + orow * p.n + col);
                    else o = reinterpret_cast<uint8_t *>(p.out) + orow * p.n + col;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        if (j < nch) reinterpret_cast<uint4 *>(o)[j] = chunk[j];
                }
            }
            if (OUT == PMN_OUT_RHT_S2F6 && valid)
                *reinterpret_cast<uint32_t *>(p.out_sc + orow * (p.n / 32) + ti.n0 / 32) = sc_word;
            if (++abuf == 2) {
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
              bool swizzle128)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {width_bytes, rows};
    cuuint64_t strides[1] = {pitch};
    cuuint32_t box[2] = {box_w, 128};
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
    const CUtensorMapDataType dt = out_kind == PMN_OUT_F32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : out_kind == PMN_OUT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                              : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    const uint64_t es = out_kind == PMN_OUT_F32 ? 4 : (out_kind == PMN_OUT_BF16 ? 2 : 1);
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

template <int KIND, int OUT>
pmn_status launch_gemm(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &sa, const CUtensorMap &sb,
                       const CUtensorMap &o, const GemmArgs &args, cudaStream_t s)
{
    auto kern = block_scaled_gemm_kernel<KIND, OUT>;
    const int smem = Cfg<KIND>::SMEM_BYTES;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return PMN_ERR_CUDA;
    const int sms = num_sms();
    if (sms <= 0) return PMN_ERR_CUDA;
    kern<<<sms, NUM_THREADS, smem, s>>>(a, b, sa, sb, o, args);
    return cudaGetLastError() == cudaSuccess ? PMN_OK : PMN_ERR_CUDA;
}

pmn_status nvfp4_common(const uint8_t *a_codes, const uint8_t *a_scales, const float *a_outer,
                        const uint8_t *b_codes, const uint8_t *b_scales, const float *b_outer,
                        const int32_t *offsets, int num_experts, int64_t total_rows, int64_t n, int64_t k,
                        int out_kind, void *out, uint8_t *out_sc, uint64_t seed, void *stream)
{
    if (num_experts <= 0 || num_experts > MAX_GROUPS || total_rows < 0 || n <= 0 || k <= 0) return PMN_ERR_INVALID_ARG;
    if (n % BN != 0 || k % 256 != 0 || total_rows >= (int64_t(1) << 31)) return PMN_ERR_INVALID_ARG;
    if (!a_codes || !a_scales || !a_outer || !b_codes || !b_scales || !b_outer || !offsets || !out)
        return PMN_ERR_INVALID_ARG;
    if (!aligned16(a_codes) || !aligned16(a_scales) || !aligned16(b_codes) || !aligned16(b_scales) ||
        !aligned16(out) || ((uintptr_t)offsets & 3u) || ((uintptr_t)a_outer & 3u) || ((uintptr_t)b_outer & 3u))
        return PMN_ERR_INVALID_ARG;
    if (out_kind == PMN_OUT_RHT_S2F6 && !out_sc) return PMN_ERR_INVALID_ARG;
    if (total_rows == 0) return PMN_OK;
    CUtensorMap ma, mb, msa, msb, mo;
    const uint64_t brows = (uint64_t)num_experts * (uint64_t)n;
    if (!make_out_map(&mo, out, out_kind, n, total_rows)) return PMN_ERR_CUDA;
    if (!make_map(&ma, a_codes, k / 2, total_rows, k / 2, 128, true) ||
        !make_map(&mb, b_codes, k / 2, brows, k / 2, 128, true) ||
        !make_map(&msa, a_scales, k / 16, total_rows, k / 16, 16, false) ||
        !make_map(&msb, b_scales, k / 16, brows, k / 16, 16, false))
        return PMN_ERR_CUDA;
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
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    switch (out_kind) {
        case PMN_OUT_BF16: return launch_gemm<KIND_NVFP4, PMN_OUT_BF16>(ma, mb, msa, msb, mo, args, s);
        case PMN_OUT_F32: return launch_gemm<KIND_NVFP4, PMN_OUT_F32>(ma, mb, msa, msb, mo, args, s);
        case PMN_OUT_RHT_S2F6: return launch_gemm<KIND_NVFP4, PMN_OUT_RHT_S2F6>(ma, mb, msa, msb, mo, args, s);
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

extern "C" pmn_status pmn_get_device_error(void *stream, int32_t *err)
{
    if (!err) return PMN_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
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
    *err = host;
    return PMN_OK;
}

extern "C" pmn_status pmn_grouped_gemm_nvfp4(const uint8_t *a_codes, const uint8_t *a_scales, const float *a_outer,
                                             const uint8_t *b_codes, const uint8_t *b_scales, const float *b_outer,
                                             const int32_t *offsets, int num_experts, int64_t total_rows, int64_t n,
                                             int64_t k, int out_kind, void *out, void *stream)
{
    if (out_kind != PMN_OUT_BF16 && out_kind != PMN_OUT_F32) return PMN_ERR_INVALID_ARG;
    return nvfp4_common(a_codes, a_scales, a_outer, b_codes, b_scales, b_outer, offsets, num_experts, total_rows, n,
                        k, out_kind, out, nullptr, 0, stream);
}

extern "C" pmn_status pmn_w2_gemm_rht_s2f6(const uint8_t *a_codes, const uint8_t *a_scales, const float *a_outer,
                                           const uint8_t *b_codes, const uint8_t *b_scales, const float *b_outer,
                                           const int32_t *offsets, int num_experts, int64_t total_rows, int64_t n,
                                           int64_t k, uint64_t seed, int8_t *out, uint8_t *out_scales, void *stream)
{
    return nvfp4_common(a_codes, a_scales, a_outer, b_codes, b_scales, b_outer, offsets, num_experts, total_rows, n,
                        k, PMN_OUT_RHT_S2F6, out, out_scales, seed, stream);
}

extern "C" pmn_status pmn_gemm_mxfp8(const uint8_t *a, const uint8_t *a_scales, const uint8_t *b,
                                     const uint8_t *b_scales, const int32_t *offsets, int num_groups, int group_mode,
                                     int64_t m, int64_t n, int64_t k, int out_kind, void *out, void *stream)
{
    if (num_groups <= 0 || num_groups > MAX_GROUPS || m < 0 || n <= 0 || k < 0) return PMN_ERR_INVALID_ARG;
    if (group_mode != PMN_GROUP_M && group_mode != PMN_GROUP_K) return PMN_ERR_INVALID_ARG;
    if (out_kind != PMN_OUT_BF16 && out_kind != PMN_OUT_F32) return PMN_ERR_INVALID_ARG;
    if (n % BN != 0 || m >= (int64_t(1) << 31) || k >= (int64_t(1) << 31)) return PMN_ERR_INVALID_ARG;
    if (group_mode == PMN_GROUP_M && (k % 128 != 0 || (k / 32) % 16 != 0)) return PMN_ERR_INVALID_ARG;
    if (group_mode == PMN_GROUP_K && (m % BM != 0 || k % 32 != 0 || (k / 32) % 16 != 0)) return PMN_ERR_INVALID_ARG;
    if (!a || !a_scales || !b || !b_scales || !offsets || !out) return PMN_ERR_INVALID_ARG;
    if (!aligned16(a) || !aligned16(a_scales) || !aligned16(b) || !aligned16(b_scales) || !aligned16(out) ||
        ((uintptr_t)offsets & 3u))
        return PMN_ERR_INVALID_ARG;
    if (m == 0) return PMN_OK;
    if (group_mode == PMN_GROUP_M && k == 0) return PMN_ERR_INVALID_ARG;
    const uint64_t brows = group_mode == PMN_GROUP_M ? (uint64_t)num_groups * (uint64_t)n : (uint64_t)n;
    CUtensorMap ma, mb, msa, msb, mo;
    if (k == 0) return PMN_ERR_INVALID_ARG;
    const uint64_t orows = group_mode == PMN_GROUP_M ? (uint64_t)m : (uint64_t)num_groups * (uint64_t)m;
    if (!make_out_map(&mo, out, out_kind, n, orows)) return PMN_ERR_CUDA;
    if (!make_map(&ma, a, k, m, k, 128, true) || !make_map(&mb, b, k, brows, k, 128, true) ||
        !make_map(&msa, a_scales, k / 32, m, k / 32, 32, false) ||
        !make_map(&msb, b_scales, k / 32, brows, k / 32, 32, false))
        return PMN_ERR_CUDA;
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
    if (out_kind == PMN_OUT_BF16) return launch_gemm<KIND_MXFP8, PMN_OUT_BF16>(ma, mb, msa, msb, mo, args, s);
    return launch_gemm<KIND_MXFP8, PMN_OUT_F32>(ma, mb, msa, msb, mo, args, s);
}
