// quantize.cu -- HBM-bound quantisation kernels of the MoE expert-layer path:
//   pmn_nvfp4_quantize              NVFP4 with outer scales and 4/6   [SR], [Cost]
//   pmn_mxfp8_quantize              bf16 -> MXFP8 (RN), both orientations
//   pmn_mxfp8_quantize_swiglu       SwiGLU -> MXFP8 (RN) of h, the MXFP8 forward [Cost]
//   pmn_requant_transpose_sr_mxfp8  dequant -> transpose -> SR MXFP8  [SR]
//   pmn_requant_transpose_sr_nvfp4  dequant -> transpose -> SR NVFP4 (FP4 backward) [SR]
//   pmn_rht_s2f6_quantize           RHT-32 + S2F6 combine quantisation [NVLink]
//   pmn_combine_receive_s2f6        S2F6 decode + inverse RHT-32 + top-k sum [NVLink]
//   pmn_nvfp4_quantize_per_group_noalloc, pmn_nvfp4_quantize_workspace_bytes,
//   pmn_wait_selftest               (the boundary's scratch and failure handling)
// and the h coding step of pmn_w1_gemm_swiglu_nvfp4 (gemm.cu).
// Sections cited are those of the page "Thinking Machines ... Inkling 2
// Small ... native 4-bit forward" (arex-research.com).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>
#include <type_traits>

#include "../../include/pmn.h"
#include "numerics.cuh"
#include "sm100.cuh"

using namespace pmn;

uint64_t pmn_wait_limit_ns();  // gemm.cu: the limit of every bounded device wait

namespace {

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline pmn_status launch_status()
{
    return cudaGetLastError() == cudaSuccess ? PMN_OK : PMN_ERR_CUDA;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

// ------------------------------------------------------------------ NVFP4 block
// One candidate block scale m (6, or 4 for the 4/6 choice) with outer scale g:
//   s = amax / (m g); S = RN_E4M3(s); sd = dec(S) g; r = 1/sd (0 if sd == 0)
//   c_i = RN_E2M1(x_i r)   (packed: element 2i low nibble)
// With the 4/6 choice each candidate also yields its summed squared
// dequantisation error (tree order i+8, +4, +2, +1).
struct BlockQ {
    uint32_t w0, w1;  // 8 code bytes
    uint32_t sbyte;
};

// Constants of one row's or one group's blocks: d = RN(m g), rd = RN(1/d).
struct QCtx {
    float g, d6, rd6, d4, rd4;
    bool fast6, fast4;  // rd finite and normal: the quotient shortcut below applies
};

__device__ __forceinline__ bool normal_finite(float v) { return fabsf(v) >= 1.17549435e-38f && fabsf(v) <= 3.4e38f; }

__device__ __forceinline__ QCtx make_qctx(float g, bool four_over_six)
{
    QCtx c;
    c.g = g;
    c.d6 = __fmul_rn(6.0f, g);
    c.rd6 = __frcp_rn(c.d6);
    c.fast6 = normal_finite(c.d6) && normal_finite(c.rd6);
    c.d4 = c.d6;
    c.rd4 = c.rd6;
    c.fast4 = false;
    if (four_over_six) {
        c.d4 = __fmul_rn(4.0f, g);
        c.rd4 = __frcp_rn(c.d4);
        c.fast4 = normal_finite(c.d4) && normal_finite(c.rd4);
    }
    return c;
}

// S = RN_E4M3(RN(amax / d)) for amax >= 0.  q = RN(amax * rd) is within
// about one ulp of amax / d (two roundings of relative size 2^-24 each), so
// the true quotient and its binary32 rounding both lie in [q - 2 ulp, q + 2
// ulp]; E4M3 rounding is monotone, so when both ends of that interval round
// to the same byte, so does RN(amax / d).  Otherwise (q within two ulps of an
// E4M3 rounding boundary) the correctly rounded quotient is formed.
__device__ __forceinline__ uint32_t block_scale_byte(float amax, float d, float rd, bool fast)
{
    if (amax == 0.0f) return 0u;
    if (fast) {
        const uint32_t qb = __float_as_uint(__fmul_rn(amax, rd));
        const uint32_t lo = cvt_e4m3(__uint_as_float(qb - 2u)), hi = cvt_e4m3(__uint_as_float(qb + 2u));
        if (lo == hi) return lo;
    }
    return cvt_e4m3(__fdiv_rn(amax, d));
}

__device__ __forceinline__ float quant_block_candidate(const float (&x)[16], float amax, float g, float d, float rd,
                                                       bool fast, bool want_err, BlockQ &out)
{
    const uint32_t S = block_scale_byte(amax, d, rd, fast);
    const uint32_t dS2 = e4m3_to_h2(S);  // dec(S) in both f16 halves (exact)
    const float sd = __fmul_rn(h2_lo_to_f32(dS2), g);
    const float r = (sd == 0.0f) ? 0.0f : __frcp_rn(sd);
    uint32_t c[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float p0, p1;
        mul2(x[2 * i], x[2 * i + 1], r, r, p0, p1);
        c[i] = cvt_e2m1x2(p0, p1);
    }
    out.w0 = __byte_perm(__byte_perm(c[0], c[1], 0x0040), __byte_perm(c[2], c[3], 0x0040), 0x5410);
    out.w1 = __byte_perm(__byte_perm(c[4], c[5], 0x0040), __byte_perm(c[6], c[7], 0x0040), 0x5410);
    out.sbyte = S;
    if (!want_err) return 0.0f;
    // dequantised value RN(RN(code * dec(S)) * g); code * dec(S) is exact in f16
    float e[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t cs2 = e2m1x2_mul_h2(c[i], dS2);
        const float d0 = __fsub_rn(x[2 * i], __fmul_rn(h2_lo_to_f32(cs2), g));
        const float d1 = __fsub_rn(x[2 * i + 1], __fmul_rn(h2_hi_to_f32(cs2), g));
        e[2 * i] = __fmul_rn(d0, d0);
        e[2 * i + 1] = __fmul_rn(d1, d1);
    }
#pragma unroll
    for (int h = 8; h >= 1; h >>= 1)
#pragma unroll
        for (int i = 0; i < h; ++i) e[i] = __fadd_rn(e[i], e[i + h]);
    return e[0];
}

__device__ __forceinline__ BlockQ quant_block(const float (&x)[16], const QCtx &c, bool four_over_six)
{
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
    BlockQ q6, q4;
    const float err6 = quant_block_candidate(x, amax, c.g, c.d6, c.rd6, c.fast6, four_over_six, q6);
    if (four_over_six) {
        const float err4 = quant_block_candidate(x, amax, c.g, c.d4, c.rd4, c.fast4, true, q4);
        if (err4 < err6) return q4;
    }
    return q6;
}

// outer scale g = amax / M (M = 6*448, or 4*448 with 4/6), 1 for a zero group
__device__ __forceinline__ float outer_from_amax(float amax, bool four_over_six)
{
    return amax == 0.0f ? 1.0f : __fdiv_rn(amax, four_over_six ? 1792.0f : 2688.0f);
}

// One warp per row; lane handles 16-blocks lane, lane+32, ...  NB = blocks per
// lane (ceil(cols/16/32)).  The whole row stays in registers, so x is read
// once.  SWIGLU: h = silu(gate) * up in binary32, rounded to bf16 first.
// Register targets, measured on rows of d_ff (SwiGLU) and d_model: 4 and 5
// resident CTAs per SM (7 % and 1.5 % faster than uncapped); wider rows keep
// their registers.
#ifndef PMN_QR_MIN_BLOCKS
#define PMN_QR_MIN_BLOCKS 4
#endif
#ifndef PMN_QR2_MIN_BLOCKS
#define PMN_QR2_MIN_BLOCKS 5
#endif
template <int NB, bool SWIGLU>
__global__ void __launch_bounds__(256, NB <= 4 ? PMN_QR_MIN_BLOCKS : 1) nvfp4_quant_rows_kernel(
    const uint16_t *__restrict__ x, int64_t rows, int cols, int64_t ldx, int four_over_six,
    uint8_t *__restrict__ codes, uint8_t *__restrict__ scales, float *__restrict__ outer,
    uint16_t *__restrict__ h_out)
{
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (row >= rows) return;
    const int nblk = cols >> 4;
    const uint16_t *xr = x + row * ldx;
    uint4 v[NB][2];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < NB; ++i) {
        int b = lane + 32 * i;
        if (b < nblk) {
            if (!SWIGLU) {
                const uint4 *p = reinterpret_cast<const uint4 *>(xr + b * 16);
                v[i][0] = __ldg(p);
                v[i][1] = __ldg(p + 1);
            } else {
                const uint4 *pg = reinterpret_cast<const uint4 *>(xr + b * 16);
                const uint4 *pu = reinterpret_cast<const uint4 *>(xr + cols + b * 16);
                uint4 gv[2] = {__ldg(pg), __ldg(pg + 1)};
                uint4 uv[2] = {__ldg(pu), __ldg(pu + 1)};
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const uint32_t *gw = reinterpret_cast<const uint32_t *>(&gv[half]);
                    const uint32_t *uw = reinterpret_cast<const uint32_t *>(&uv[half]);
                    uint32_t hw[4];
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        float a0 = bf16_lo(gw[t]), a1 = bf16_hi(gw[t]);
                        float u0 = bf16_lo(uw[t]), u1 = bf16_hi(uw[t]);
                        float h0 = silu_mul(a0, u0);
                        float h1 = silu_mul(a1, u1);
                        __nv_bfloat16 b0 = __float2bfloat16_rn(h0), b1 = __float2bfloat16_rn(h1);
                        hw[t] = (uint32_t)__bfloat16_as_ushort(b0) | ((uint32_t)__bfloat16_as_ushort(b1) << 16);
                    }
                    v[i][half] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                }
                if (h_out) {
                    uint4 *ph = reinterpret_cast<uint4 *>(h_out + row * cols + b * 16);
                    ph[0] = v[i][0];
                    ph[1] = v[i][1];
                }
            }
            const uint32_t *w = reinterpret_cast<const uint32_t *>(&v[i][0]);
#pragma unroll
            for (int t = 0; t < 8; ++t) amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[t])), fabsf(bf16_hi(w[t]))));
        }
    }
    const bool fos = four_over_six != 0;
    amax = warp_max(amax);
    const float g = outer_from_amax(amax, fos);
    const QCtx qc = make_qctx(g, fos);
    if (lane == 0) outer[row] = g;
#pragma unroll
    for (int i = 0; i < NB; ++i) {
        int b = lane + 32 * i;
        if (b < nblk) {
            float xf[16];
            const uint32_t *w = reinterpret_cast<const uint32_t *>(&v[i][0]);
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                xf[2 * t] = bf16_lo(w[t]);
                xf[2 * t + 1] = bf16_hi(w[t]);
            }
            BlockQ q = quant_block(xf, qc, fos);
            *reinterpret_cast<uint2 *>(codes + row * (cols >> 1) + b * 8) = make_uint2(q.w0, q.w1);
            scales[row * nblk + b] = (uint8_t)q.sbyte;
        }
    }
}

// ---------------------------------------------------------- per-group NVFP4
// Weights (one outer scale per expert) need the expert's amax before any of
// its blocks can be coded.  One persistent kernel does both passes over two
// streams of work items handed out by a ticket counter: A_i = amax of chunk i
// (chunk c of group g is i = g * nch + c), B_i = NVFP4 coding of chunk i.
// Tickets run A_0 .. A_{D-1}, then A_{D+k}, B_k alternately, then the last
// B items: the A stream leads by D >= nch items, so B_i's group has all its A
// items ticketed first; with D = nch + (CTAs in flight) they have mostly
// finished, and a chunk is coded about one group after its amax pass read
// it, while its rows are still in L2: HBM sees each weight byte read once.
// B waits (bounded) for its group's A count; no A item ever waits, so the
// streams progress whatever the number of resident CTAs.
constexpr int QG_THREADS = 256;
#ifndef PMN_QG_CHUNK
#define PMN_QG_CHUNK 2048
#endif
constexpr int QG_CHUNK = PMN_QG_CHUNK;  // 16-blocks per work item (32 Ki values)
constexpr int QG_PAD = 64;      // the ticket sits alone in its 256-byte line

// scratch words: [0] ticket, [QG_PAD + g] done count of A(g, *),
// [QG_PAD + groups + g] amax bits of group g; all zero at launch
inline size_t quant_groups_scratch_bytes(int64_t groups) { return (size_t)(QG_PAD + 2 * groups) * 4u; }

__device__ int g_pmn_quant_error = 0;

// Fixed scratch of the no-allocation entry point (groups <= QG_NOALLOC_GROUPS).
constexpr int QG_NOALLOC_GROUPS = 1024;
static __device__ __align__(256) uint32_t g_qg_scratch[QG_PAD + 2 * QG_NOALLOC_GROUPS];

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits until *count >= target (acquire).  Gives up after limit_ns of wall
// time: latches PMN_DEVERR_WAIT_TIMEOUT and returns false.  Never traps.
__device__ __forceinline__ bool wait_count(const uint32_t *count, uint32_t target, uint64_t limit_ns)
{
    if (ld_acquire_u32(count) >= target) return true;
    const uint64_t t0 = global_ns();
    while (ld_acquire_u32(count) < target) {
        __nanosleep(128);
        if (global_ns() - t0 > limit_ns) {
            atomicOr(&g_pmn_quant_error, PMN_DEVERR_WAIT_TIMEOUT);
            return false;
        }
    }
    return true;
}

// L2 cache policies (createpolicy) and 16-byte loads that carry one.
__device__ __forceinline__ uint64_t l2_policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint4 ld_l2_policy(const uint4 *ptr, uint64_t policy)
{
    uint4 v;
    asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(ptr), "l"(policy));
    return v;
}

#ifndef PMN_QG_MIN_BLOCKS  // resident CTAs per SM the register allocation aims for (measured: 4 beats 3
#define PMN_QG_MIN_BLOCKS 4  // by 4-8 %; 5 spills heavily)
#endif
__global__ void __launch_bounds__(QG_THREADS, PMN_QG_MIN_BLOCKS) nvfp4_quant_groups_kernel(
    const uint16_t *__restrict__ x, int64_t groups, int64_t blocks_per_group, int64_t nch, int64_t lead,
    int four_over_six, uint8_t *__restrict__ codes, uint8_t *__restrict__ scales, float *__restrict__ outer,
    uint32_t *scratch, uint64_t wait_ns)
{
    __shared__ uint32_t s_red[QG_THREADS / 32];
    __shared__ uint32_t s_ticket;
    __shared__ float s_g;
    __shared__ int s_stop;
    uint32_t *ticket = scratch, *done = scratch + QG_PAD, *amax = scratch + QG_PAD + groups;
    const int tid = threadIdx.x;
    const int64_t na = groups * nch, total = 2 * na, paired = na - lead;
    // L2 priorities: amax reads stay (the coding pass re-reads them about a
    // group later), coding reads leave
    const uint64_t keep = l2_policy_evict_last(), drop = l2_policy_evict_first();
    const bool fos = four_over_six != 0;
    if (tid == 0) s_ticket = atomicAdd(ticket, 1u);
    __syncthreads();
    for (;;) {
        const int64_t t = s_ticket;
        if (t >= total) break;
        // the next item's ticket is taken now and published at the end of
        // this item, so the atomic's round trip overlaps this item's work
        uint32_t next = 0u;
        if (tid == 0) next = atomicAdd(ticket, 1u);
        bool is_a;
        int64_t i;  // chunk index in its stream
        if (t < lead) {
            is_a = true;
            i = t;
        } else if (t - lead < 2 * paired) {
            is_a = ((t - lead) & 1) == 0;
            i = is_a ? lead + ((t - lead) >> 1) : ((t - lead) >> 1);
        } else {
            is_a = false;
            i = paired + (t - lead - 2 * paired);
        }
        const int64_t g = i / nch, c = i - g * nch;
        const int64_t b0 = c * QG_CHUNK, b1 = min(b0 + QG_CHUNK, blocks_per_group);
        const uint16_t *xg = x + g * blocks_per_group * 16;
        bool stop = false;
        if (is_a) {
            {
                // ---- A(g, c): max |x| over the chunk on bf16 bit patterns (the
                // 8 blocks of a thread fully unrolled: measured 1 % faster than 4)
                uint32_t m = 0u;
#pragma unroll 8
                for (int64_t b = b0 + tid; b < b1; b += QG_THREADS) {
                    const uint4 *q = reinterpret_cast<const uint4 *>(xg + b * 16);
                    const uint4 v0 = ld_l2_policy(q, keep), v1 = ld_l2_policy(q + 1, keep);
                    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
                    for (int k = 0; k < 8; ++k) m = __vmaxu2(m, w[k] & 0x7FFF7FFFu);  // per 16-bit half
                }
                m = max(m & 0xFFFFu, m >> 16);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
                if ((tid & 31) == 0) s_red[tid >> 5] = m;
                __syncthreads();
                if (tid == 0) {
                    uint32_t r = s_red[0];
                    for (int i = 1; i < QG_THREADS / 32; ++i) r = max(r, s_red[i]);
                    atomicMax(amax + g, r << 16);  // binary32 bits of the bf16 amax
                    __threadfence();
                    atomicAdd(done + g, 1u);
                }
            }
        } else {
            // ---- B(g, c): code the chunk once the group's amax is final.  The
            // first two blocks' loads are in flight while thread 0 waits.
            uint4 v[2][2];
            auto load2 = [&](int64_t bb) {
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int64_t bi = bb + u * QG_THREADS;
                    if (bi < b1) {
                        const uint4 *q = reinterpret_cast<const uint4 *>(xg + bi * 16);
                        v[u][0] = ld_l2_policy(q, drop);
                        v[u][1] = ld_l2_policy(q + 1, drop);
                    }
                }
            };
            load2(b0 + tid);
            if (tid == 0) {
                const int st = wait_count(done + g, (uint32_t)nch, wait_ns) ? 0 : 1;
                const float gv = outer_from_amax(__uint_as_float(ld_acquire_u32(amax + g)), fos);
                if (c == 0 && !st) outer[g] = gv;
                s_g = gv;
                s_stop = st;
            }
            __syncthreads();
            stop = s_stop != 0;
            const float gv = s_g;
            const QCtx qc = make_qctx(gv, fos);
            for (int64_t bb = b0 + tid; bb < b1 && !stop; bb += 2 * QG_THREADS) {
                uint4 cur[2][2];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    cur[u][0] = v[u][0];
                    cur[u][1] = v[u][1];
                }
                if (bb + 2 * QG_THREADS < b1) load2(bb + 2 * QG_THREADS);
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int64_t bi = bb + u * QG_THREADS;
                    if (bi >= b1) continue;
                    const uint32_t w[8] = {cur[u][0].x, cur[u][0].y, cur[u][0].z, cur[u][0].w,
                                           cur[u][1].x, cur[u][1].y, cur[u][1].z, cur[u][1].w};
                    float xf[16];
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        xf[2 * k] = bf16_lo(w[k]);
                        xf[2 * k + 1] = bf16_hi(w[k]);
                    }
                    const BlockQ qb = quant_block(xf, qc, fos);
                    const int64_t gb = g * blocks_per_group + bi;
                    *reinterpret_cast<uint2 *>(codes + gb * 8) = make_uint2(qb.w0, qb.w1);
                    scales[gb] = (uint8_t)qb.sbyte;
                }
            }
        }
        __syncthreads();  // every thread is done with s_red, s_g and s_ticket
        if (stop) break;
        if (tid == 0) s_ticket = next;
        __syncthreads();
    }
}

// A counter that nothing increments (the self-test's second wait).
static __device__ uint32_t g_never_counted = 0;

// Self-test of the bounded waits: thread 0 waits on an mbarrier that nothing
// arrives on, then on a counter that nothing increments, with the same wait
// primitives the GEMMs and the weight quantiser use.  Each wait gives up after
// limit_ns and latches PMN_DEVERR_WAIT_TIMEOUT; the kernel then returns.
__global__ void wait_selftest_kernel(uint64_t limit_ns)
{
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    const uint32_t b = sm100::smem_u32(&bar);
    sm100::mbar_init(b, 1);
    sm100::fence_barrier_init();
    if (!sm100::mbar_wait(b, 0, limit_ns)) atomicOr(&g_pmn_quant_error, PMN_DEVERR_WAIT_TIMEOUT);
    (void)wait_count(&g_never_counted, 1u, limit_ns);
}

// bf16 rows (no SwiGLU): the row is read twice instead of being held in
// registers -- once for its amax, then block by block for the codes (the
// second read hits L1/L2) -- so more warps fit per SM to hide the 4/6 scoring.
// row_end (optional, device): rows at or past *row_end are not read and are
// written as the quantisation of a zero row (codes 0, scales 0, outer 1).
template <int NB>
__global__ void __launch_bounds__(256, NB <= 8 ? PMN_QR2_MIN_BLOCKS : 1) nvfp4_quant_rows2_kernel(const uint16_t *__restrict__ x, int64_t rows,
                                                                int cols, int64_t ldx, int four_over_six,
                                                                uint8_t *__restrict__ codes,
                                                                uint8_t *__restrict__ scales, float *__restrict__ outer,
                                                                const int32_t *__restrict__ row_end)
{
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (row >= rows) return;
    const int nblk = cols >> 4;
    if (row_end != nullptr && row >= (int64_t)__ldg(row_end)) {
        for (int b = lane; b < nblk; b += 32) {
            *reinterpret_cast<uint2 *>(codes + row * (cols >> 1) + b * 8) = make_uint2(0u, 0u);
            scales[row * nblk + b] = 0;
        }
        if (lane == 0) outer[row] = 1.0f;
        return;
    }
    const uint16_t *xr = x + row * ldx;
    uint32_t m = 0u;
#pragma unroll
    for (int i = 0; i < NB; ++i) {
        const int b = lane + 32 * i;
        if (b < nblk) {
            const uint4 *p = reinterpret_cast<const uint4 *>(xr + b * 16);
            const uint4 v0 = __ldg(p), v1 = __ldg(p + 1);
            const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
            for (int t = 0; t < 8; ++t) m = __vmaxu2(m, w[t] & 0x7FFF7FFFu);  // |bf16| orders as integers
        }
    }
    m = max(m & 0xFFFFu, m >> 16);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    const bool fos = four_over_six != 0;
    const float g = outer_from_amax(__uint_as_float(m << 16), fos);
    const QCtx qc = make_qctx(g, fos);
    if (lane == 0) outer[row] = g;
#pragma unroll 2
    for (int i = 0; i < NB; ++i) {
        const int b = lane + 32 * i;
        if (b < nblk) {
            const uint4 *p = reinterpret_cast<const uint4 *>(xr + b * 16);
            const uint4 v0 = __ldg(p), v1 = __ldg(p + 1);
            const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
            float xf[16];
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                xf[2 * t] = bf16_lo(w[t]);
                xf[2 * t + 1] = bf16_hi(w[t]);
            }
            const BlockQ q = quant_block(xf, qc, fos);
            *reinterpret_cast<uint2 *>(codes + row * (cols >> 1) + b * 8) = make_uint2(q.w0, q.w1);
            scales[row * nblk + b] = (uint8_t)q.sbyte;
        }
    }
}

template <int NB>
void launch_rows(bool swiglu, dim3 grid, dim3 block, cudaStream_t s, const uint16_t *x, int64_t rows,
                 int cols, int64_t ldx, int fos, uint8_t *codes, uint8_t *scales, float *outer, uint16_t *h_out,
                 const int32_t *row_end = nullptr)
{
    if (swiglu)
        nvfp4_quant_rows_kernel<NB, true><<<grid, block, 0, s>>>(x, rows, cols, ldx, fos, codes, scales, outer, h_out);
    else
        nvfp4_quant_rows2_kernel<NB><<<grid, block, 0, s>>>(x, rows, cols, ldx, fos, codes, scales, outer, row_end);
}

// Per-row NVFP4 of bf16 rows [rows, cols] (dense), the rows at or past
// *row_end (device) written as zero rows.
pmn_status launch_rows_bf16(const uint16_t *x, int64_t rows, int cols, int fos, uint8_t *codes, uint8_t *scales,
                            float *outer, const int32_t *row_end, cudaStream_t s)
{
    const int nb = (cols / 16 + 31) / 32;
    dim3 block(256), grid((unsigned)((rows + 7) / 8));
    if (nb <= 1) launch_rows<1>(false, grid, block, s, x, rows, cols, cols, fos, codes, scales, outer, nullptr, row_end);
    else if (nb <= 2) launch_rows<2>(false, grid, block, s, x, rows, cols, cols, fos, codes, scales, outer, nullptr, row_end);
    else if (nb <= 4) launch_rows<4>(false, grid, block, s, x, rows, cols, cols, fos, codes, scales, outer, nullptr, row_end);
    else if (nb <= 8) launch_rows<8>(false, grid, block, s, x, rows, cols, cols, fos, codes, scales, outer, nullptr, row_end);
    else launch_rows<16>(false, grid, block, s, x, rows, cols, cols, fos, codes, scales, outer, nullptr, row_end);
    return launch_status();
}

// ------------------------------------------------------------------ MXFP8 RN (dY)
// rowwise: one thread per 32-block along the row.
__global__ void __launch_bounds__(256) mxfp8_quant_rowwise_kernel(const uint16_t *__restrict__ x,
                                                                  int64_t nblocks, int64_t bpr,
                                                                  uint8_t *__restrict__ out,
                                                                  uint8_t *__restrict__ out_sc)
{
    int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= nblocks) return;
    const uint4 *p = reinterpret_cast<const uint4 *>(x + t * 32);
    uint4 q[4] = {__ldg(p), __ldg(p + 1), __ldg(p + 2), __ldg(p + 3)};
    const uint32_t *w = reinterpret_cast<const uint32_t *>(q);
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[i])), fabsf(bf16_hi(w[i]))));
    const int e = mx_exponent_448(amax);
    const float sc = exp2_neg(e);  // y = x * 2^-e is exact
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t lo = cvt_e4m3x2_rn(__fmul_rn(bf16_lo(w[2 * i]), sc), __fmul_rn(bf16_hi(w[2 * i]), sc));
        const uint32_t hi = cvt_e4m3x2_rn(__fmul_rn(bf16_lo(w[2 * i + 1]), sc), __fmul_rn(bf16_hi(w[2 * i + 1]), sc));
        o[i] = lo | (hi << 16);
    }
    uint4 *po = reinterpret_cast<uint4 *>(out + t * 32);
    po[0] = make_uint4(o[0], o[1], o[2], o[3]);
    po[1] = make_uint4(o[4], o[5], o[6], o[7]);
    out_sc[t] = (uint8_t)(e + 127);
    (void)bpr;
}

// SwiGLU, then MXFP8 (round to nearest) of h, for the MXFP8 forward of the
// last layers [Cost]: y bf16 [rows, 2 f] holds gate | up; thread = one
// 32-block of h.  h = silu(gate) * up in binary32 (the same operations as the
// NVFP4 SwiGLU path), rounded to bf16, then quantised as the rowwise kernel
// above.  rows * f / 32 < 2^32 (checked by the caller).
__global__ void __launch_bounds__(256) mxfp8_swiglu_rowwise_kernel(const uint16_t *__restrict__ y, uint32_t nblocks,
                                                                   uint32_t bpr, uint8_t *__restrict__ out,
                                                                   uint8_t *__restrict__ out_sc,
                                                                   uint16_t *__restrict__ h_out)
{
    const uint32_t t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= nblocks) return;
    const uint32_t row = t / bpr, b = t - row * bpr;
    const int64_t f = (int64_t)bpr * 32;
    const uint4 *pg = reinterpret_cast<const uint4 *>(y + (int64_t)row * 2 * f + 32 * (int64_t)b);
    const uint4 *pu = reinterpret_cast<const uint4 *>(y + (int64_t)row * 2 * f + f + 32 * (int64_t)b);
    uint4 gv[4], uv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        gv[i] = __ldg(pg + i);
        uv[i] = __ldg(pu + i);
    }
    const uint32_t *gw = reinterpret_cast<const uint32_t *>(gv);
    const uint32_t *uw = reinterpret_cast<const uint32_t *>(uv);
    uint32_t hw[16];
    uint32_t m = 0u;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float a0 = bf16_lo(gw[i]), a1 = bf16_hi(gw[i]);
        const float h0 = silu_mul(a0, bf16_lo(uw[i]));
        const float h1 = silu_mul(a1, bf16_hi(uw[i]));
        hw[i] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(h0)) |
                ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(h1)) << 16);
        m = __vmaxu2(m, hw[i] & 0x7FFF7FFFu);  // |bf16| orders as integers
    }
    const float amax = __uint_as_float(max(m & 0xFFFFu, m >> 16) << 16);
    const int e = mx_exponent_448(amax);
    const float sc = exp2_neg(e);  // y * 2^-e is exact
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t lo = cvt_e4m3x2_rn(__fmul_rn(bf16_lo(hw[2 * i]), sc), __fmul_rn(bf16_hi(hw[2 * i]), sc));
        const uint32_t hi =
            cvt_e4m3x2_rn(__fmul_rn(bf16_lo(hw[2 * i + 1]), sc), __fmul_rn(bf16_hi(hw[2 * i + 1]), sc));
        o[i] = lo | (hi << 16);
    }
    uint4 *po = reinterpret_cast<uint4 *>(out + (int64_t)t * 32);
    po[0] = make_uint4(o[0], o[1], o[2], o[3]);
    po[1] = make_uint4(o[4], o[5], o[6], o[7]);
    out_sc[t] = (uint8_t)(e + 127);
    if (h_out) {
        uint4 *ph = reinterpret_cast<uint4 *>(h_out + (int64_t)t * 32);
#pragma unroll
        for (int i = 0; i < 4; ++i) ph[i] = make_uint4(hw[4 * i], hw[4 * i + 1], hw[4 * i + 2], hw[4 * i + 3]);
    }
}

// ------------------------------------------------------------------ requant [SR]
// One CTA per tile of 128 input rows x 128 input cols.
// Phase 1: each thread decodes an 8-row x 8-column block: code * S is exact
//   in f16 (E2M1 x E4M3, 2^-10 .. 2688), formed by the hardware E2M1 decode
//   and a packed f16 multiply, transposed in registers and written as 128-bit
//   rows of the transposed tile cS[c][r] (f16, chunk index swizzled so both
//   phases are bank-conflict free).
// Phase 2: task (c, rb) forms the 32-block of output row c.  The canonical
//   dequantised value is d = (code * S) * g (one rounding); with the block's
//   E8M0 exponent e, y = d * 2^-e equals RN(code * S * (g * 2^-e)) because a
//   power-of-two scaling commutes with rounding -- so y takes one multiply.
//   For a per-expert g the block maximum is fl(max|code * S| * g) (rounding
//   is monotone), found on the f16 bit patterns with packed integer max.
//   E4M3 bytes: hardware stochastic rounding fed with Philox words (one
//   Philox call per 16 elements), or round-to-nearest-even.
constexpr int RQ_T = 128;

// 16-byte chunk `logical` (rows 8*logical ..) of transposed row c.  A 128-bit
// shared access is served per quarter-warp, so 8 lanes must land in 8 distinct
// 16-byte bank groups (index mod 8).  Phase 1 quarters vary c over 8 columns
// 8 apart (XOR with c ^ c>>3 spreads them); phase 2 quarters take 2 adjacent
// c times logical chunks k, 4+k, 8+k, 12+k: bit 3 of `logical` is folded into
// bit 1 so those four differ mod 8, and adjacent c differ in bit 0.
__device__ __forceinline__ int rq_chunk(int c, int logical)
{
    return c * 16 + (logical ^ ((c ^ (c >> 3)) & 7) ^ ((logical >> 3) << 1));
}

// transposed MXFP8 (RN): 128 x 128 tile.  Phase 1 as in the requantisation:
// each thread loads an 8-row x 8-column block (16-byte row pieces), transposes
// it in registers and stores 16-byte chunks (8 rows of one column) into the
// swizzled tile.  Phase 2: task (c, rb) forms the 32-block of output row c;
// four consecutive lanes write one 128-byte line of the output row.
// ROWS: the same pass also writes the rowwise MXFP8 of the tile (the input is
// read once for both orientations): in phase 1 the four lanes that hold one
// row's 32-column block (column groups 4b .. 4b+3, adjacent lanes) take the
// block's amax with two shuffles and each converts its 8 values, with the
// arithmetic of mxfp8_quant_rowwise_kernel.
// Resident CTAs per SM the register allocation aims for.  Column blocks only:
// 5 (6 % faster than the uncapped 4; 6 spills).  Both orientations: 4 (at 5
// the added row pass spills, 21 % slower; 3 is 10 % slower).
#ifndef PMN_MXT_MIN_BLOCKS
#define PMN_MXT_MIN_BLOCKS 5
#endif
#ifndef PMN_MXB_MIN_BLOCKS
#define PMN_MXB_MIN_BLOCKS 4
#endif
template <bool ROWS>
__global__ void __launch_bounds__(256, ROWS ? PMN_MXB_MIN_BLOCKS : PMN_MXT_MIN_BLOCKS) mxfp8_quant_transposed_kernel(const uint16_t *__restrict__ x,
                                                                     int64_t rows, int64_t cols,
                                                                     uint8_t *__restrict__ out,
                                                                     uint8_t *__restrict__ out_sc,
                                                                     uint8_t *__restrict__ out_r,
                                                                     uint8_t *__restrict__ out_r_sc)
{
    __shared__ __align__(16) uint4 cS[RQ_T * 16];  // [c][16 chunks of 8 rows] bf16
    const int64_t r0 = (int64_t)blockIdx.y * RQ_T, c0 = (int64_t)blockIdx.x * RQ_T;
    {
        const int cg = threadIdx.x & 15, rg = threadIdx.x >> 4;
        const bool col_ok = c0 + 8 * cg < cols;
        const int rows_left = (int)min((int64_t)8, rows - (r0 + 8 * rg));
        const uint16_t *xp = x + (r0 + 8 * rg) * cols + c0 + 8 * cg;
        uint4 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            v[i] = make_uint4(0u, 0u, 0u, 0u);
            if (col_ok && i < rows_left) v[i] = __ldg(reinterpret_cast<const uint4 *>(xp + i * cols));
        }
        if constexpr (ROWS) {
            // rowwise blocks: lanes 4b .. 4b+3 of a 16-lane row group hold one
            // row's 32 columns (out-of-range lanes hold zeros and store nothing)
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
                float amax = 0.0f;
#pragma unroll
                for (int k = 0; k < 4; ++k) amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[k])), fabsf(bf16_hi(w[k]))));
                amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
                amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
                const int e = mx_exponent_448(amax);
                const float sc = exp2_neg(e);  // y = x * 2^-e is exact
                uint32_t o[2];
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    float p0, p1, p2, p3;
                    mul2(bf16_lo(w[2 * k]), bf16_hi(w[2 * k]), sc, sc, p0, p1);
                    mul2(bf16_lo(w[2 * k + 1]), bf16_hi(w[2 * k + 1]), sc, sc, p2, p3);
                    o[k] = cvt_e4m3x2_rn(p0, p1) | (cvt_e4m3x2_rn(p2, p3) << 16);
                }
                if (col_ok && i < rows_left) {
                    const int64_t row = r0 + 8 * rg + i, col = c0 + 8 * cg;
                    *reinterpret_cast<uint2 *>(out_r + row * cols + col) = make_uint2(o[0], o[1]);
                    if ((cg & 3) == 0) out_r_sc[row * (cols / 32) + col / 32] = (uint8_t)(e + 127);
                }
            }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {  // columns 2k, 2k+1
            uint32_t lo[4], hi[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t a = u4_word(v[2 * i], k), bb = u4_word(v[2 * i + 1], k);
                lo[i] = __byte_perm(a, bb, 0x5410);
                hi[i] = __byte_perm(a, bb, 0x7632);
            }
            const int cl = 8 * cg + 2 * k;
            cS[rq_chunk(cl, rg)] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            cS[rq_chunk(cl + 1, rg)] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        }
    }
    __syncthreads();
#pragma unroll 1
    for (int task = threadIdx.x; task < RQ_T * 4; task += blockDim.x) {
        const int c = task >> 2, rb = task & 3;
        const int64_t oc = c0 + c, orow0 = r0 + rb * 32;
        if (oc >= cols || orow0 >= rows) continue;
        uint32_t hw[16];  // 32 bf16 values: rows rb*32 .. rb*32+31
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint4 u = cS[rq_chunk(c, 4 * rb + k)];
            hw[4 * k] = u.x;
            hw[4 * k + 1] = u.y;
            hw[4 * k + 2] = u.z;
            hw[4 * k + 3] = u.w;
        }
        uint32_t m = 0u;
#pragma unroll
        for (int j = 0; j < 16; ++j) m = __vmaxu2(m, hw[j] & 0x7FFF7FFFu);  // |bf16| orders as integers
        const float amax = __uint_as_float(max(m & 0xFFFFu, m >> 16) << 16);
        const int e = mx_exponent_448(amax);
        const float sc = exp2_neg(e);
        uint32_t o[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float p0, p1, p2, p3;
            mul2(bf16_lo(hw[2 * i]), bf16_hi(hw[2 * i]), sc, sc, p0, p1);
            mul2(bf16_lo(hw[2 * i + 1]), bf16_hi(hw[2 * i + 1]), sc, sc, p2, p3);
            o[i] = cvt_e4m3x2_rn(p0, p1) | (cvt_e4m3x2_rn(p2, p3) << 16);
        }
        uint4 *po = reinterpret_cast<uint4 *>(out + oc * rows + orow0);
        po[0] = make_uint4(o[0], o[1], o[2], o[3]);
        po[1] = make_uint4(o[4], o[5], o[6], o[7]);
        out_sc[oc * (rows / 32) + orow0 / 32] = (uint8_t)(e + 127);
    }
}

// Two E2M1 codes (byte K of `word`) decoded by the hardware to f16x2 and
// multiplied by an E4M3 scale held as f16x2: exact, as in e2m1x8_mul_h2.
template <int K>
__device__ __forceinline__ uint32_t e2m1x2_byte_mul_h2(uint32_t word, uint32_t scale_h2)
{
    uint32_t h2, p;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b%2;\n\t}"
        : "=r"(h2) : "r"(word), "n"(K));
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(p) : "r"(h2), "r"(scale_h2));
    return p;
}

// Philox4x32-10 for counters whose high word is shared by a whole thread: the
// first round's product of the tag and the second round's product of the
// resulting first word depend only on (tag, high word, key), so they are
// formed once per thread.  Same arithmetic as philox4x32_10.
struct PhiloxPrefix {
    uint32_t k0, k1, y1, x2hi, x2lo;  // see philox_from_prefix
};

__device__ __forceinline__ PhiloxPrefix philox_prefix(uint64_t seed, uint32_t tag, uint32_t jhi)
{
    PhiloxPrefix p;
    p.k0 = (uint32_t)seed;
    p.k1 = (uint32_t)(seed >> 32);
    const uint32_t x1 = __umulhi(0xCD9E8D57u, tag) ^ jhi ^ p.k0;  // round 1 output word 0
    p.y1 = 0xCD9E8D57u * tag;                                   // round 1 output word 1
    p.x2hi = __umulhi(0xD2511F53u, x1);                         // round 2, first product
    p.x2lo = 0xD2511F53u * x1;
    return p;
}

__device__ __forceinline__ uint4 philox_from_prefix(const PhiloxPrefix &p, uint32_t jlo)
{
    // round 1: c = (jlo, jhi, tag, 0)
    const uint32_t z1 = __umulhi(0xD2511F53u, jlo) ^ p.k1, w1 = 0xD2511F53u * jlo;
    // round 2: c = (x1, y1, z1, w1) with keys bumped once
    const uint32_t k0 = p.k0 + 0x9E3779B9u, k1 = p.k1 + 0xBB67AE85u;
    uint4 c = make_uint4(__umulhi(0xCD9E8D57u, z1) ^ p.y1 ^ k0, 0xCD9E8D57u * z1, p.x2hi ^ w1 ^ k1, p.x2lo);
    uint32_t q0 = k0, q1 = k1;
#pragma unroll
    for (int r = 2; r < 10; ++r) {
        q0 += 0x9E3779B9u;
        q1 += 0xBB67AE85u;
        c = philox_round(c, q0, q1);
    }
    return c;
}

// Requantisation of one thread's 16 input rows (lanes l and l ^ 16 hold the
// two halves of a 32-row block) x 8 input columns.  word[i] / s2[i]: the code
// word (columns 2k, 2k + 1 in byte k) and the E4M3 block scale (as f16x2) of
// row i; g: the group's outer scale, or the 16 rows' (PER_ROW).  j0: the
// Philox counter of (first column, first row); jstep = rows / 16 steps to the
// next column.  Output row orow0 + c (c = 0 .. 7) gets its 16-byte chunk at
// oS[(orow0 + c) * 8 + chunk] and, from the low lane of the pair, its E8M0
// byte at scS[(orow0 + c) * 4 + rb].
template <bool PER_ROW>
__device__ __forceinline__ void rq_block16x8(const uint32_t (&word)[16], const uint32_t (&s2)[16],
                                             const float (&g)[PER_ROW ? 16 : 1], unsigned act, uint64_t j0,
                                             uint64_t jstep, uint64_t seed, uint32_t tag, int stochastic,
                                             bool low, int orow0, int chunk, int rb, uint4 *oS, uint8_t *scS)
{
    const uint32_t jhi0 = (uint32_t)(j0 >> 32);
    const bool one_hi = (uint32_t)((j0 + 7 * jstep) >> 32) == jhi0;
    const PhiloxPrefix pre = philox_prefix(seed, tag, jhi0);
    auto emit = [&](int c, const float (&y)[16], int e) {
        const uint64_t j = j0 + (uint64_t)c * jstep;
        uint32_t o[4];
        if (stochastic) {
            const uint4 wd = one_hi ? philox_from_prefix(pre, (uint32_t)j) : sr_words16(seed, tag, j);
            o[0] = cvt_e4m3x4_rs(y[0], y[1], y[2], y[3], wd.x);
            o[1] = cvt_e4m3x4_rs(y[4], y[5], y[6], y[7], wd.y);
            o[2] = cvt_e4m3x4_rs(y[8], y[9], y[10], y[11], wd.z);
            o[3] = cvt_e4m3x4_rs(y[12], y[13], y[14], y[15], wd.w);
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k)
                o[k] = cvt_e4m3x2_rn(y[4 * k], y[4 * k + 1]) | (cvt_e4m3x2_rn(y[4 * k + 2], y[4 * k + 3]) << 16);
        }
        oS[(orow0 + c) * 8 + chunk] = make_uint4(o[0], o[1], o[2], o[3]);
        if (low) scS[(orow0 + c) * 4 + rb] = (uint8_t)(e + 127);
    };
    auto column_pair = [&](auto kc) {
        constexpr int K = decltype(kc)::value;
        uint32_t cs[16];  // exact code * S of columns 2K (low halves) and 2K + 1 (high halves)
#pragma unroll
        for (int i = 0; i < 16; ++i) cs[i] = e2m1x2_byte_mul_h2<K>(word[i], s2[i]);
        if (!PER_ROW) {
            uint32_t m[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) m[i] = h2_absmax_xs(cs[2 * i], cs[2 * i + 1]);
#pragma unroll
            for (int h = 4; h >= 1; h >>= 1)
#pragma unroll
                for (int i = 0; i < h; ++i) m[i] = h2_absmax_xs(m[i], m[i + h]);
            const uint32_t mm = h2_absmax_xs(m[0], __shfl_xor_sync(act, m[0], 16)) & 0x7FFF7FFFu;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const float amax_cs = hf ? h2_hi_to_f32(mm) : h2_lo_to_f32(mm);
                const int e = mx_exponent_448(__fmul_rn(amax_cs, g[0]));
                // exact; an all-zero block keeps its signed zeros (g * 2^127 could overflow)
                const float gp = amax_cs == 0.0f ? 0.0f : __fmul_rn(g[0], exp2_neg(e));
                float y[16];
#pragma unroll
                for (int i = 0; i < 16; i += 2) {
                    const float a0 = hf ? h2_hi_to_f32(cs[i]) : h2_lo_to_f32(cs[i]);
                    const float a1 = hf ? h2_hi_to_f32(cs[i + 1]) : h2_lo_to_f32(cs[i + 1]);
                    mul2(a0, a1, gp, gp, y[i], y[i + 1]);
                }
                emit(2 * K + hf, y, e);
            }
        } else {
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                float y[16], amax = 0.0f;
#pragma unroll
                for (int i = 0; i < 16; i += 2) {
                    const float a0 = hf ? h2_hi_to_f32(cs[i]) : h2_lo_to_f32(cs[i]);
                    const float a1 = hf ? h2_hi_to_f32(cs[i + 1]) : h2_lo_to_f32(cs[i + 1]);
                    mul2(a0, a1, g[i], g[i + 1], y[i], y[i + 1]);
                    amax = fmaxf(amax, fmaxf(fabsf(y[i]), fabsf(y[i + 1])));
                }
                amax = fmaxf(amax, __shfl_xor_sync(act, amax, 16));
                const int e = mx_exponent_448(amax);
                const float sc = exp2_neg(e);
#pragma unroll
                for (int i = 0; i < 16; i += 2) mul2(y[i], y[i + 1], sc, sc, y[i], y[i + 1]);  // exact
                emit(2 * K + hf, y, e);
            }
        }
    };
    column_pair(std::integral_constant<int, 0>());
    column_pair(std::integral_constant<int, 1>());
    column_pair(std::integral_constant<int, 2>());
    column_pair(std::integral_constant<int, 3>());
}

// Requantisation of an NVFP4 tensor [batch, rows, cols] to MXFP8 of its
// transpose [batch, cols, rows].  CTA = 4 warps = a 128-row x 128-column
// tile.  Thread = 16 input rows x 8 input columns; lanes l and l ^ 16 hold the
// two halves of a 32-row block, so each input column's values are half of one
// output 32-block: its amax takes one shuffle, its 16 elements are one Philox
// counter (16j .. 16j+15) and its bytes one 16-byte chunk.  The chunks are
// staged in shared memory ([output row][8 chunks], chunk index XOR bits 3..5 of
// the output row: conflict-free both ways) and written as whole 128-byte lines
// after one barrier.  COLS > 0 fixes the row length at compile time so the 16
// row loads use immediate offsets.
// Register targets (measured): 5 resident CTAs per SM for the per-group form;
// the per-row form keeps 16 more outer scales and is left uncapped.
template <bool PER_ROW, int COLS>
__global__ void __launch_bounds__(128, PER_ROW ? 1 : 5) requant_transpose_kernel(
    const uint8_t *__restrict__ codes, const uint8_t *__restrict__ scales, const float *__restrict__ outer,
    int64_t rows, int64_t cols_rt, uint64_t seed, uint32_t tag, int stochastic,
    uint8_t *__restrict__ out, uint8_t *__restrict__ out_sc)
{
    __shared__ __align__(16) uint4 oS[128 * 8];  // [output row][16-row chunk ^ swizzle]
    __shared__ __align__(4) uint8_t scS[128 * 4];  // [output row][32-row block]: E8M0 bytes
    const int64_t cols = COLS > 0 ? (int64_t)COLS : cols_rt;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, q = lane & 15, hf = lane >> 4;
    const int64_t b = blockIdx.z;
    const int64_t r0 = (int64_t)blockIdx.y * 128, c0 = (int64_t)blockIdx.x * 128;
    const int64_t rb0 = r0 + 32 * w;  // the warp's 32-row block
    const int64_t col0 = c0 + 8 * q;
    const bool active = rb0 < rows && col0 < cols;  // lanes l, l ^ 16 agree
    const unsigned act = __ballot_sync(0xFFFFFFFFu, active);
    if (active) {
    const int64_t row0 = rb0 + 16 * hf;
    const int64_t cols2 = cols / 2, cols16 = cols / 16;
    const uint8_t *cp = codes + (b * rows + row0) * cols2 + col0 / 2;
    const uint8_t *sp = scales + (b * rows + row0) * cols16 + col0 / 16;
    uint32_t word[16], s2[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) word[i] = __ldg(reinterpret_cast<const uint32_t *>(cp + i * cols2));
#pragma unroll
    for (int i = 0; i < 16; ++i) s2[i] = e4m3_to_h2(__ldg(sp + i * cols16));
    float g[PER_ROW ? 16 : 1];
    if (PER_ROW) {
#pragma unroll
        for (int i = 0; i < 16; ++i) g[i] = __ldg(outer + b * rows + row0 + i);
    } else {
        g[0] = __ldg(outer + b);
    }
    // Philox counter of (column col0, rows row0 .. row0+15); column col0 + c adds c * rows / 16
    const uint64_t j0 = (uint64_t)((b * cols + col0) * rows + row0) >> 4;
    // output rows 8q .. 8q+7 share bits 3..5, so the chunk index XOR them spreads a quarter-warp
    rq_block16x8<PER_ROW>(word, s2, g, act, j0, (uint64_t)rows >> 4, seed, tag, stochastic, hf == 0, 8 * q,
                          (2 * w + hf) ^ (q & 7), w, oS, scS);
    }
    __syncthreads();
    // whole lines: 8 consecutive threads write the 128 bytes of one output row
    const int rows_here = (int)min((int64_t)128, rows - r0), cols_here = (int)min((int64_t)128, cols - c0);
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int idx = it * 128 + threadIdx.x, c = idx >> 3, ch = idx & 7;
        if (c < cols_here && 16 * ch < rows_here)
            *reinterpret_cast<uint4 *>(out + (b * cols + c0 + c) * rows + r0 + 16 * ch) = oS[c * 8 + (ch ^ ((c >> 3) & 7))];
    }
    if ((int)threadIdx.x < cols_here) {
        const int c = threadIdx.x;
        uint8_t *dst = out_sc + (b * cols + c0 + c) * (rows / 32) + r0 / 32;
        if (rows_here == 128 && ((reinterpret_cast<uintptr_t>(dst) & 3u) == 0)) {
            *reinterpret_cast<uint32_t *>(dst) = *reinterpret_cast<const uint32_t *>(scS + 4 * c);
        } else {
            for (int k = 0; 32 * k < rows_here; ++k) dst[k] = scS[4 * c + k];
        }
    }
}

// ------------------------------------------------------------------ requant to NVFP4 (FP4 backward)
// The FP4 backward the pages name as future work: the [SR] steps (dequantise,
// transpose, requantise with stochastic rounding) with the NVFP4 format.
// Outer scale of the transposed entry b: g' = (max over its input blocks of
// dec(S) * g) / 448, 1 if every scale is zero.  Block scale: the smallest
// E4M3 value >= amax / RN(6 g'), so no value clips; codes by stochastic
// rounding of y = d * RN(1 / RN(dec(S') g')) onto E2M1 with 16 random bits
// (the rule and bit layout of the MXFP8 requantisation), or nearest even.

// Largest dec(S) * g of each entry, as float bits (non-negative floats order
// as integers, so atomicMax is order-independent).  A CTA reduces 32 KB of one
// entry's scales with 16-byte loads and takes one atomic (grid
// (ceil(words / 8192), batch)): the atomics of an entry are few enough not to
// serialise on its one address.  Over the codes with the sign bit clear, dec
// is non-decreasing in the byte (0x7F decodes as 480); the others decode to
// <= 0 and never raise the maximum; and RN(x g) is non-decreasing in x for
// g >= 0.  So the largest product of a set of bytes that share g is
// RN(dec(their largest sign-clear byte) * g): bytes are compared as unsigned
// integers and decoded once per word (per-row outer: a word's four scales lie
// in one row) or once per thread (one outer per entry).
constexpr int SMX_PIECES = 8;  // 16-byte pieces per thread
__global__ void __launch_bounds__(256) nvfp4_scale_max_kernel(const uint8_t *__restrict__ scales,
                                                              const float *__restrict__ outer, int per_row,
                                                              uint32_t rows, uint32_t wpr,
                                                              uint32_t *__restrict__ gmax)
{
    __shared__ float red[8];
    const int64_t b = blockIdx.y;
    const uint32_t nw = rows * wpr;  // rows % 32 == 0: every entry starts 16-byte aligned, nw % 4 == 0
    const uint4 *sp = reinterpret_cast<const uint4 *>(scales + (uint64_t)b * nw * 4u);
    float m = 0.0f;
    uint32_t acc = 0u;  // per-byte maximum of the sign-clear bytes (one outer per entry)
#pragma unroll
    for (int it = 0; it < SMX_PIECES; ++it) {
        const uint32_t p = blockIdx.x * (256u * SMX_PIECES) + it * 256u + threadIdx.x;
        if (p < nw / 4u) {
            const uint4 v = __ldg(sp + p);
            const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
            if (per_row) {
                uint32_t r = (4u * p) / wpr, k = 4u * p - r * wpr;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint32_t x = w4[kk] & __vcmpltu4(w4[kk], 0x80808080u);
                    uint32_t t = __vmaxu4(x, x >> 16);
                    t = __vmaxu4(t, t >> 8);
                    m = fmaxf(m, __fmul_rn(e4m3_to_f32(t & 0xFFu), __ldg(outer + b * rows + r)));
                    if (++k == wpr) { k = 0u; ++r; }
                }
            } else {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) acc = __vmaxu4(acc, w4[kk] & __vcmpltu4(w4[kk], 0x80808080u));
            }
        }
    }
    if (!per_row) {
        uint32_t t = __vmaxu4(acc, acc >> 16);
        t = __vmaxu4(t, t >> 8);
        m = __fmul_rn(e4m3_to_f32(t & 0xFFu), __ldg(outer + b));
    }
    m = warp_max(m);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        float mm = red[0];
#pragma unroll
        for (int i = 1; i < 8; ++i) mm = fmaxf(mm, red[i]);
        if (mm > 0.0f) atomicMax(gmax + b, __float_as_uint(mm));
    }
}

__device__ __forceinline__ float nvfp4_outer_from_max(uint32_t bits)
{
    return bits == 0u ? 1.0f : __fdiv_rn(__uint_as_float(bits), 448.0f);
}

__global__ void nvfp4_outer_finalize_kernel(float *out_outer, int64_t batch)
{
    const int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (b < batch) out_outer[b] = nvfp4_outer_from_max(__float_as_uint(out_outer[b]));
}

// Stochastic rounding of y onto E2M1 (sign kept): with ulp the grid step at
// |y| (0.5 below 2, 1 below 4, 2 above) and t = |y| / ulp, the grid index is
// floor(t) plus the carry of rb16 + the 16 leading fraction bits, i.e.
// (floor(t 2^16) + rb16) >> 16; 6 saturates.  t 2^16 < 2^19 is exact, and
// adding 2^23 rounded toward zero leaves floor(t 2^16) in the low mantissa
// bits, so no float-to-integer conversion is needed.
__device__ __forceinline__ uint32_t e2m1_sr(float y, uint32_t rb16)
{
    const float a = fminf(fabsf(y), 7.0f);  // every value >= 6 gives code 7
    const float sc = a < 2.0f ? 131072.0f : (a < 4.0f ? 65536.0f : 32768.0f);  // 2^16 / ulp
    const uint32_t u = __float_as_uint(__fadd_rz(__fmul_rn(a, sc), 8388608.0f)) - 0x4B000000u;
    const uint32_t k = (u + rb16) >> 16;
    const uint32_t code = a < 2.0f ? k : (a < 4.0f ? k + 2u : min(k + 4u, 7u));
    return code | (signbit(y) ? 8u : 0u);
}

// Hardware stochastic rounding of four values to E2M1 (nibble i = element i,
// sign kept).  The convert applies the same add-and-carry rule as e2m1_sr but
// reads its random bits in another order than the E4M3 one: element 0 takes
// bytes 2 and 0 of rbits as one 16-bit value, element 2 bytes 3 and 1,
// elements 1 and 3 the same values bit-reversed (measured over 4 M inputs).
// Swapping bytes 1 and 2 of a Philox word therefore gives every element the
// 16 bits that sr_bits_of assigns it.  PMN_FP4_HW_SR=0 selects the integer
// rounding e2m1_sr instead (the same bytes).
#ifndef PMN_FP4_HW_SR
#define PMN_FP4_HW_SR 1
#endif
__device__ __forceinline__ uint32_t cvt_e2m1x4_rs(float e0, float e1, float e2, float e3, uint32_t word)
{
    uint16_t r;
    asm("cvt.rs.satfinite.e2m1x4.f32 %0, {%1, %2, %3, %4}, %5;"
        : "=h"(r)
        : "f"(e3), "f"(e2), "f"(e1), "f"(e0), "r"(__byte_perm(word, 0u, 0x3120u)));
    return r;
}

// 16 random bits of element e (0..15) of a Philox block: word e / 4; low or
// high half; odd elements bit-reversed.
__device__ __forceinline__ uint32_t sr_bits_of(const uint4 &wd, int e)
{
    const uint32_t w = (e >> 2) == 0 ? wd.x : (e >> 2) == 1 ? wd.y : (e >> 2) == 2 ? wd.z : wd.w;
    const uint32_t h = (e & 2) ? (w >> 16) : (w & 0xFFFFu);
    return (e & 1) ? (__brev(h) >> 16) : h;
}

// Thread = 16 input rows x 8 input columns, as requant_transpose_kernel: the
// 16 rows of one column are exactly one output 16-block and one Philox
// counter.  CTA = 4 warps = 128 rows x 128 columns.  Per block the scale's
// reciprocal RN(1 / RN(dec(S') g')) comes from a per-CTA table of the 127
// finite E4M3 values (g' is the entry's); the products are packed binary32
// multiplies; per-expert inputs take the block's amax from the exact f16
// products code * S (amax_i RN(cs_i g) = RN(amax_i cs_i * g), g > 0).  Codes
// and scales are staged in shared memory ([output row][16-row chunk], chunk
// XOR bits 3..5 of the row) and written as 16-byte pieces, four lanes per
// output row.
// Register targets (measured): 5 resident CTAs per SM for the per-group form
// (faster than 4 by 3 %; 6 spills and is 6 % slower), 4 for the per-row
// form, which would spill at 5.
#ifndef PMN_FP4RQ_MIN_BLOCKS
#define PMN_FP4RQ_MIN_BLOCKS 5
#endif
template <bool PER_ROW>
__global__ void __launch_bounds__(128, PER_ROW ? 4 : PMN_FP4RQ_MIN_BLOCKS) requant_transpose_nvfp4_kernel(
    const uint8_t *__restrict__ codes, const uint8_t *__restrict__ scales, const float *__restrict__ outer,
    int64_t rows, int64_t cols, uint64_t seed, uint32_t tag, int stochastic, const uint32_t *__restrict__ gmax,
    uint8_t *__restrict__ out, uint8_t *__restrict__ out_sc)
{
    __shared__ __align__(16) uint2 oS[128 * 8];     // [output row][chunk ^ swizzle]: 16 codes = 8 bytes
    __shared__ __align__(8) uint8_t scS[128 * 8];   // [output row][chunk]: E4M3 block scale
    __shared__ float rtab[128];                     // RN(1 / RN(dec(S) g')), 0 where that product is 0
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, q = lane & 15, hf = lane >> 4;
    const int64_t b = blockIdx.z;
    const int64_t r0 = (int64_t)blockIdx.y * 128, c0 = (int64_t)blockIdx.x * 128;
    const int64_t row0 = r0 + 32 * w + 16 * hf;
    const int64_t col0 = c0 + 8 * q;
    const float gp = nvfp4_outer_from_max(__ldg(gmax + b));
    if (threadIdx.x < 127) {
        const float sd = __fmul_rn(e4m3_to_f32(threadIdx.x), gp);
        rtab[threadIdx.x] = sd == 0.0f ? 0.0f : __frcp_rn(sd);
    }
    __syncthreads();
    if (row0 < rows && col0 < cols) {
    const int chunk = 2 * w + hf;  // the thread's 16-row chunk of the tile
    const int64_t cols2 = cols / 2, cols16 = cols / 16;
    const uint8_t *cp = codes + (b * rows + row0) * cols2 + col0 / 2;
    const uint8_t *sp = scales + (b * rows + row0) * cols16 + col0 / 16;
    uint32_t word[16], s2[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) word[i] = __ldg(reinterpret_cast<const uint32_t *>(cp + i * cols2));
#pragma unroll
    for (int i = 0; i < 16; ++i) s2[i] = e4m3_to_h2(__ldg(sp + i * cols16));
    float g[PER_ROW ? 16 : 1];
    if (PER_ROW) {
#pragma unroll
        for (int i = 0; i < 16; ++i) g[i] = __ldg(outer + b * rows + row0 + i);
    } else {
        g[0] = __ldg(outer + b);
    }
    const float six_g = __fmul_rn(6.0f, gp);
    const uint64_t j0 = (uint64_t)((b * cols + col0) * rows + row0) >> 4;
    const uint64_t jstep = (uint64_t)rows >> 4;
    const uint32_t jhi0 = (uint32_t)(j0 >> 32);
    const bool one_hi = (uint32_t)((j0 + 7 * jstep) >> 32) == jhi0;
    const PhiloxPrefix pre = philox_prefix(seed, tag, jhi0);
    auto column_pair = [&](auto kc) {
        constexpr int K = decltype(kc)::value;
        uint32_t cs[16];  // exact code * S of columns 2K (low halves) and 2K + 1 (high halves)
#pragma unroll
        for (int i = 0; i < 16; ++i) cs[i] = e2m1x2_byte_mul_h2<K>(word[i], s2[i]);
        uint32_t mm = 0u;
        if (!PER_ROW) {
            uint32_t m[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) m[i] = h2_absmax_xs(cs[2 * i], cs[2 * i + 1]);
#pragma unroll
            for (int hh = 4; hh >= 1; hh >>= 1)
#pragma unroll
                for (int i = 0; i < hh; ++i) m[i] = h2_absmax_xs(m[i], m[i + hh]);
            mm = m[0] & 0x7FFF7FFFu;
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int c = 2 * K + h;
            float d[16], amax = 0.0f;
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
                const float a0 = h ? h2_hi_to_f32(cs[i]) : h2_lo_to_f32(cs[i]);
                const float a1 = h ? h2_hi_to_f32(cs[i + 1]) : h2_lo_to_f32(cs[i + 1]);
                mul2(a0, a1, g[PER_ROW ? i : 0], g[PER_ROW ? i + 1 : 0], d[i], d[i + 1]);
                if (PER_ROW) amax = fmaxf(amax, fmaxf(fabsf(d[i]), fabsf(d[i + 1])));
            }
            if (!PER_ROW) amax = __fmul_rn(h ? h2_hi_to_f32(mm) : h2_lo_to_f32(mm), g[0]);
            const float sq = __fdiv_rn(amax, six_g);
            uint32_t S = cvt_e4m3(sq);
            if (e4m3_to_f32(S) < sq && S < 0x7Eu) ++S;  // round the scale up: no value clips
            const float r = rtab[S];
            float y[16];
#pragma unroll
            for (int i = 0; i < 16; i += 2) mul2(d[i], d[i + 1], r, r, y[i], y[i + 1]);
            uint32_t packed[2] = {0u, 0u};
            if (stochastic) {
                const uint64_t j = j0 + (uint64_t)c * jstep;
                const uint4 wd = one_hi ? philox_from_prefix(pre, (uint32_t)j) : sr_words16(seed, tag, j);
#if PMN_FP4_HW_SR
                const uint32_t wv[4] = {wd.x, wd.y, wd.z, wd.w};
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4)
                    packed[q4 >> 1] |= cvt_e2m1x4_rs(y[4 * q4], y[4 * q4 + 1], y[4 * q4 + 2], y[4 * q4 + 3], wv[q4])
                                       << (16 * (q4 & 1));
#else
#pragma unroll
                for (int i = 0; i < 16; ++i) packed[i >> 3] |= e2m1_sr(y[i], sr_bits_of(wd, i)) << (4 * (i & 7));
#endif
            } else {
#pragma unroll
                for (int i = 0; i < 16; i += 2) packed[i >> 3] |= cvt_e2m1x2(y[i], y[i + 1]) << (4 * (i & 7));
            }
            const int orow = 8 * q + c;  // output row within the tile; bits 3..5 = q & 7
            oS[orow * 8 + (chunk ^ (q & 7))] = make_uint2(packed[0], packed[1]);
            scS[orow * 8 + chunk] = (uint8_t)S;
        }
    };
    column_pair(std::integral_constant<int, 0>());
    column_pair(std::integral_constant<int, 1>());
    column_pair(std::integral_constant<int, 2>());
    column_pair(std::integral_constant<int, 3>());
    }
    __syncthreads();
    // write-out: four lanes per output row, 16 bytes (two chunks) each
    const int64_t vrows = min((int64_t)128, rows - r0), vcols = min((int64_t)128, cols - c0);
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const int orow = it * 32 + (threadIdx.x >> 2), seg = threadIdx.x & 3;
        if (orow >= vcols || 32 * seg >= vrows) continue;
        const int sw = (orow >> 3) & 7;
        const uint2 lo = oS[orow * 8 + ((2 * seg) ^ sw)], hi = oS[orow * 8 + ((2 * seg + 1) ^ sw)];
        const int64_t oc = b * cols + c0 + orow;
        *reinterpret_cast<uint4 *>(out + oc * (rows / 2) + r0 / 2 + 16 * seg) = make_uint4(lo.x, lo.y, hi.x, hi.y);
        *reinterpret_cast<uint16_t *>(out_sc + oc * (rows / 16) + r0 / 16 + 2 * seg) =
            (uint16_t)(scS[orow * 8 + 2 * seg] | (scS[orow * 8 + 2 * seg + 1] << 8));
    }
}

// ------------------------------------------------------------------ RHT + S2F6
__global__ void __launch_bounds__(256) rht_s2f6_kernel(const float *__restrict__ x, int64_t nblocks,
                                                       uint64_t seed, int8_t *__restrict__ out,
                                                       uint8_t *__restrict__ out_sc)
{
    int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= nblocks) return;
    const uint32_t sigma = rht_sigma(seed);
    float v[32];
    const float4 *p = reinterpret_cast<const float4 *>(x + t * 32);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float4 f = __ldg(p + i);
        v[4 * i] = f.x;
        v[4 * i + 1] = f.y;
        v[4 * i + 2] = f.z;
        v[4 * i + 3] = f.w;
    }
    uint32_t q[8];
    uint32_t sb = rht32_s2f6(v, sigma, q);
    uint4 *po = reinterpret_cast<uint4 *>(out + t * 32);
    po[0] = make_uint4(q[0], q[1], q[2], q[3]);
    po[1] = make_uint4(q[4], q[5], q[6], q[7]);
    out_sc[t] = (uint8_t)sb;
}

// ------------------------------------------------------------------ combine receive
// Receive side of the combine [NVLink], back in token order.  The back
// transform is linear, so the k choices are summed first and transformed once:
//   u = sum_i (gate_i * 2^(e_i - 6)) * k_i     (float32 fma, choices in order)
//   y = sigma . (FWHT32(u) * RN(1/sqrt(32)))
// which equals sum_i gate_i * sigma . H (k_i 2^(e_i - 6)) / sqrt(32) up to
// float32 rounding.  An S2F6 byte enters as float32 exactly: the byte plus 128
// becomes the low mantissa byte of 2^23, and 2^23 + 128 is subtracted.
// Thread = half of one 32-value block (values 16 h .. 16 h + 15, h = lane & 1):
// the butterfly stages of stride 1 .. 8 run in registers, the stride-16 stage
// pairs lanes l and l ^ 1 through one shuffle per value.  Packed float32x2
// arithmetic for the conversion, the sum and the in-lane butterflies.
__device__ __forceinline__ void add2(float a0, float a1, float b0, float b1, float &c0, float &c1)
{
    asm("{\n\t.reg .b64 a, b, c;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
        "add.rn.f32x2 c, a, b;\n\tmov.b64 {%0, %1}, c;\n\t}"
        : "=f"(c0), "=f"(c1) : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

__device__ __forceinline__ void sub2(float a0, float a1, float b0, float b1, float &c0, float &c1)
{
    asm("{\n\t.reg .b64 a, b, c;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
        "sub.rn.f32x2 c, a, b;\n\tmov.b64 {%0, %1}, c;\n\t}"
        : "=f"(c0), "=f"(c1) : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

__device__ __forceinline__ void fma2(float a0, float a1, float b0, float b1, float &c0, float &c1)
{
    asm("{\n\t.reg .b64 a, b, c;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\tmov.b64 c, {%0, %1};\n\t"
        "fma.rn.f32x2 c, a, b, c;\n\tmov.b64 {%0, %1}, c;\n\t}"
        : "+f"(c0), "+f"(c1) : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// u[0..3] += s * (4 S2F6 bytes of w)
__device__ __forceinline__ void s2f6_word_fma(uint32_t w, float s, float *u)
{
    const uint32_t x = w ^ 0x80808080u;  // k + 128 per byte
    const float c = 8388736.0f;          // 2^23 + 128
    float f[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) f[j] = __uint_as_float(__byte_perm(x, 0x4B000000u, 0x7540u + j));
    sub2(f[0], f[1], c, c, f[0], f[1]);
    sub2(f[2], f[3], c, c, f[2], f[3]);
    fma2(f[0], f[1], s, s, u[0], u[1]);
    fma2(f[2], f[3], s, s, u[2], u[3]);
}

__device__ __forceinline__ void s2f6_half_fma(const uint4 &w, float s, float (&u)[16])
{
    s2f6_word_fma(w.x, s, u);
    s2f6_word_fma(w.y, s, u + 4);
    s2f6_word_fma(w.z, s, u + 8);
    s2f6_word_fma(w.w, s, u + 12);
}

// KF > 0: the number of choices at compile time (all loads issued before the
// arithmetic); KF == 0: k_rt choices, one at a time.  A negative row index is
// a dropped choice; an index >= rows latches PMN_DEVERR_BAD_OFFSETS and is
// dropped too.
template <int KF, bool BF16>
__global__ void __launch_bounds__(256, 3) combine_receive_kernel(
    const int8_t *__restrict__ q, const uint8_t *__restrict__ sc, int64_t rows, int64_t nb, uint64_t seed,
    const int32_t *__restrict__ row_index, const float *__restrict__ gates, int64_t tokens, int k_rt,
    void *__restrict__ out)
{
    // CTA (t, y): token t, blocks 128 y .. 128 y + 127 of its row
    const int64_t t = blockIdx.x;
    const int64_t b = (int64_t)blockIdx.y * (blockDim.x / 2) + (threadIdx.x >> 1);
    const int hf = threadIdx.x & 1;
    // every lane stays for the stride-16 shuffle; lanes past the row's end load and store nothing
    const bool active = b < nb;
    const int64_t cols = nb * 32;
    const int k = KF > 0 ? KF : k_rt;
    const int32_t *ri = row_index + t * k;
    const float *gi = gates + t * k;
    // the sign-scaled normalisation sigma_j * RN(1/sqrt(32)) of the 32 positions, once per CTA
    __shared__ __align__(16) float sgn_rs[32];
    if (threadIdx.x < 32) {
        const uint32_t sigma = rht_sigma(seed);
        sgn_rs[threadIdx.x] = __uint_as_float(0x3E3504F3u ^ (((sigma >> threadIdx.x) & 1u) << 31));
    }
    float u[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) u[j] = 0.0f;
    auto row_ok = [&](int32_t r) {
        if (r >= rows) atomicOr(&g_pmn_quant_error, PMN_DEVERR_BAD_OFFSETS);
        return r >= 0 && r < rows;
    };
    // gate * 2^(e - 6) with e = byte - 127, as (g * 2^min(byte - 7, 0)) * 2^max(byte - 133, -126):
    // both factors are normal powers of two, so one rounding at most (below the normal range)
    auto row_scale = [&](float g, uint32_t e8) {
        const int e = (int)e8;
        const float lo = __uint_as_float((uint32_t)(min(e, 7) + 120) << 23);
        const float hi = __uint_as_float((uint32_t)max(e - 6, 1) << 23);
        return __fmul_rn(__fmul_rn(g, lo), hi);
    };
    const int64_t off = 32 * b + 16 * hf;
    if (active) {
        if (KF > 0) {
            constexpr int N = KF > 0 ? KF : 1;
            int32_t r[N];
            float g[N];
            uint4 w[N];
            uint32_t e8[N];
            if (N % 4 == 0 && ((reinterpret_cast<uintptr_t>(ri) | reinterpret_cast<uintptr_t>(gi)) & 15u) == 0) {
#pragma unroll
                for (int i = 0; i < N; i += 4) {  // 16-byte loads of the choices' indices and gates
                    const int4 rv = __ldg(reinterpret_cast<const int4 *>(ri + i));
                    const float4 gv = __ldg(reinterpret_cast<const float4 *>(gi + i));
                    r[i] = rv.x, r[i + 1] = rv.y, r[i + 2] = rv.z, r[i + 3] = rv.w;
                    g[i] = gv.x, g[i + 1] = gv.y, g[i + 2] = gv.z, g[i + 3] = gv.w;
                }
            } else {
#pragma unroll
                for (int i = 0; i < N; ++i) {
                    r[i] = __ldg(ri + i);
                    g[i] = __ldg(gi + i);
                }
            }
#pragma unroll
            for (int i = 0; i < N; ++i) {
                w[i] = make_uint4(0u, 0u, 0u, 0u);  // S2F6 zeros
                e8[i] = 0u;
                if (row_ok(r[i])) {
                    w[i] = __ldg(reinterpret_cast<const uint4 *>(q + (int64_t)r[i] * cols + off));
                    e8[i] = __ldg(sc + (int64_t)r[i] * nb + b);
                } else {
                    g[i] = 0.0f;
                }
            }
#pragma unroll
            for (int i = 0; i < N; ++i) s2f6_half_fma(w[i], row_scale(g[i], e8[i]), u);
        } else {
            for (int i = 0; i < k; ++i) {
                const int32_t r = __ldg(ri + i);
                if (!row_ok(r)) continue;
                const uint4 w = __ldg(reinterpret_cast<const uint4 *>(q + (int64_t)r * cols + off));
                s2f6_half_fma(w, row_scale(__ldg(gi + i), __ldg(sc + (int64_t)r * nb + b)), u);
            }
        }
    }
    // strides 1, 2, 4, 8 in registers
#pragma unroll
    for (int i = 0; i < 16; i += 2) {  // stride 1: (u[i], u[i+1])
        const float a = u[i], c = u[i + 1];
        u[i] = __fadd_rn(a, c);
        u[i + 1] = __fsub_rn(a, c);
    }
#pragma unroll
    for (int h = 2; h < 16; h <<= 1) {
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
            if ((i & h) == 0) {
                float s0, s1, d0, d1;
                add2(u[i], u[i + 1], u[i + h], u[i + h + 1], s0, s1);
                sub2(u[i], u[i + 1], u[i + h], u[i + h + 1], d0, d1);
                u[i] = s0;
                u[i + 1] = s1;
                u[i + h] = d0;
                u[i + h + 1] = d1;
            }
        }
    }
    // stride 16 across the lane pair: low half a + b, high half a - b (one rounding each)
    const float sgn = hf ? -1.0f : 1.0f;
    float p[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) p[j] = __shfl_xor_sync(0xFFFFFFFFu, u[j], 1);
#pragma unroll
    for (int j = 0; j < 16; j += 2) fma2(sgn, sgn, u[j], u[j + 1], p[j], p[j + 1]);
    __syncthreads();  // sgn_rs written
    const float4 *cr = reinterpret_cast<const float4 *>(sgn_rs + 16 * hf);
#pragma unroll
    for (int v = 0; v < 4; ++v) {  // times sigma_j RN(1/sqrt(32)): the sign is exact
        const float4 c = cr[v];
        mul2(p[4 * v], p[4 * v + 1], c.x, c.y, u[4 * v], u[4 * v + 1]);
        mul2(p[4 * v + 2], p[4 * v + 3], c.z, c.w, u[4 * v + 2], u[4 * v + 3]);
    }
    if (!active) return;
    if (BF16) {
        uint32_t o[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const __nv_bfloat162 h2 = __floats2bfloat162_rn(u[2 * j], u[2 * j + 1]);
            o[j] = *reinterpret_cast<const uint32_t *>(&h2);
        }
        uint4 *po = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(out) + t * cols + off);
        po[0] = make_uint4(o[0], o[1], o[2], o[3]);
        po[1] = make_uint4(o[4], o[5], o[6], o[7]);
    } else {
        float4 *po = reinterpret_cast<float4 *>(static_cast<float *>(out) + t * cols + off);
#pragma unroll
        for (int v = 0; v < 4; ++v) po[v] = make_float4(u[4 * v], u[4 * v + 1], u[4 * v + 2], u[4 * v + 3]);
    }
}

constexpr int MAX_DEVICES = 64;

// Resident CTAs of the per-group kernel on the current device (SMs x CTAs
// per SM), computed once per device under a lock.
pmn_status quant_groups_grid(int *out)
{
    static std::mutex mu;
    static int grid[MAX_DEVICES] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return PMN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    if (grid[dev] == 0) {
        int sms = 0, per_sm = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, nvfp4_quant_groups_kernel, QG_THREADS, 0) !=
                cudaSuccess)
            return PMN_ERR_CUDA;
        grid[dev] = std::max(1, sms * per_sm);
    }
    *out = grid[dev];
    return PMN_OK;
}

// Clears the scratch, then runs the per-group kernel on as many CTAs as fit.
pmn_status launch_quant_groups(const uint16_t *x, int64_t groups, int64_t blocks_per_group, int four_over_six,
                               uint8_t *codes, uint8_t *scales, float *outer, uint32_t *scratch, cudaStream_t s)
{
    int grid = 0;
    if (quant_groups_grid(&grid) != PMN_OK) return PMN_ERR_CUDA;
    if (cudaMemsetAsync(scratch, 0, quant_groups_scratch_bytes(groups), s) != cudaSuccess) return PMN_ERR_CUDA;
    const int64_t nch = (blocks_per_group + QG_CHUNK - 1) / QG_CHUNK;
    // Amax items lead the coding items of the same chunks by one group plus
    // three quarters of an item per CTA, capped at 45 MB of chunks (about a
    // third of L2) and never below one group: the chunks read for their amax
    // wait in L2 for their coding, so a longer lead pushes them out and a
    // shorter one makes coding items wait.  Measured (full-size step):
    // uncapped, quant_w1 2.536 ms; capped at 600 / 690 / 780 items of 64 KB,
    // 2.525 / 2.473 / 2.478 ms; quant_w2 (648 items) unchanged.
#ifndef PMN_QG_LEAD_Q  // the lead beyond one group, in quarters of an item per CTA
#define PMN_QG_LEAD_Q 3
#endif
#ifndef PMN_QG_LEAD_CAP_MB
#define PMN_QG_LEAD_CAP_MB 45
#endif
    const int64_t cap = ((int64_t)PMN_QG_LEAD_CAP_MB << 20) / ((int64_t)QG_CHUNK * 32);
    const int64_t lead = std::min(groups * nch, std::max(nch, std::min(nch + (int64_t)grid * PMN_QG_LEAD_Q / 4, cap)));
    nvfp4_quant_groups_kernel<<<(unsigned)grid, QG_THREADS, 0, s>>>(x, groups, blocks_per_group, nch, lead,
                                                                     four_over_six, codes, scales, outer, scratch,
                                                                     pmn_wait_limit_ns());
    return launch_status();
}

}  // namespace

// The h coding step of pmn_w1_gemm_swiglu_nvfp4 (gemm.cu): per-row NVFP4 of
// the GEMM's bf16 h, rows past the expert segments written as zero rows.
pmn_status pmn_quantize_h_rows(const uint16_t *h, int64_t rows, int cols, int fos, uint8_t *codes, uint8_t *scales,
                               float *outer, const int32_t *row_end, cudaStream_t s)
{
    return launch_rows_bf16(h, rows, cols, fos, codes, scales, outer, row_end, s);
}

// Reads and clears the quantisation kernels' device error bits (called by
// pmn_get_device_error, which owns the stream synchronisation).
pmn_status pmn_take_quant_device_error(cudaStream_t s, int *bits)
{
    int host = 0;
    if (cudaMemcpyFromSymbolAsync(&host, g_pmn_quant_error, sizeof(int), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return PMN_ERR_CUDA;
    if (host != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbolAsync(g_pmn_quant_error, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s) !=
                cudaSuccess ||
            cudaStreamSynchronize(s) != cudaSuccess)
            return PMN_ERR_CUDA;
    }
    *bits = host;
    return PMN_OK;
}

// Device address of the fixed scratch, looked up once per device.
pmn_status noalloc_scratch(uint32_t **out)
{
    static std::mutex mu;
    static void *addr[MAX_DEVICES] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return PMN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_qg_scratch) != cudaSuccess || !p) return PMN_ERR_CUDA;
        addr[dev] = p;
    }
    *out = static_cast<uint32_t *>(addr[dev]);
    return PMN_OK;
}

// ====================================================================== C ABI
extern "C" pmn_status pmn_wait_selftest(uint64_t limit_ns, void *stream)
{
    if (limit_ns > 2000000000ull) return PMN_ERR_INVALID_ARG;
    wait_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(limit_ns);
    return launch_status();
}

extern "C" pmn_status pmn_nvfp4_quantize_per_group_noalloc(const void *x, int64_t rows, int64_t cols,
                                                            int64_t rows_per_group, int four_over_six,
                                                            uint8_t *codes, uint8_t *scales, float *outer,
                                                            void *stream)
{
    if (rows < 0 || cols <= 0 || cols % 16 != 0 || cols > 8192) return PMN_ERR_INVALID_ARG;
    if (four_over_six != 0 && four_over_six != 1) return PMN_ERR_INVALID_ARG;
    if (rows_per_group <= 0 || rows % rows_per_group != 0) return PMN_ERR_INVALID_ARG;
    if (rows / rows_per_group > QG_NOALLOC_GROUPS) return PMN_ERR_INVALID_ARG;
    if (!x || !codes || !scales || !outer) return PMN_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(codes) || !aligned16(scales) || !aligned16(outer)) return PMN_ERR_INVALID_ARG;
    if (rows == 0) return PMN_OK;
    uint32_t *scratch = nullptr;
    if (noalloc_scratch(&scratch) != PMN_OK) return PMN_ERR_CUDA;
    return launch_quant_groups(reinterpret_cast<const uint16_t *>(x), rows / rows_per_group,
                               rows_per_group * (cols / 16), four_over_six, codes, scales, outer, scratch,
                               reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int64_t pmn_nvfp4_quantize_workspace_bytes(int outer_mode, int64_t rows, int64_t rows_per_group)
{
    if (outer_mode != PMN_OUTER_PER_GROUP) return outer_mode == PMN_OUTER_PER_ROW ? 0 : -1;
    if (rows < 0 || rows_per_group <= 0 || rows % rows_per_group != 0) return -1;
    return (int64_t)quant_groups_scratch_bytes(rows / rows_per_group);
}

extern "C" pmn_status pmn_nvfp4_quantize(const void *x, int64_t rows, int64_t cols, int64_t ldx, int in_mode,
                                         int outer_mode, int64_t rows_per_group, int four_over_six,
                                         uint8_t *codes, uint8_t *scales, float *outer, void *h_out,
                                         void *workspace, int64_t workspace_bytes, void *stream)
{
    if (rows < 0 || cols <= 0 || cols % 16 != 0 || cols > 8192) return PMN_ERR_INVALID_ARG;
    if (in_mode != PMN_IN_BF16 && in_mode != PMN_IN_BF16_SWIGLU) return PMN_ERR_INVALID_ARG;
    if (outer_mode != PMN_OUTER_PER_ROW && outer_mode != PMN_OUTER_PER_GROUP) return PMN_ERR_INVALID_ARG;
    if (four_over_six != 0 && four_over_six != 1) return PMN_ERR_INVALID_ARG;
    const bool swiglu = in_mode == PMN_IN_BF16_SWIGLU;
    if (ldx < (swiglu ? 2 * cols : cols) || ldx % 8 != 0) return PMN_ERR_INVALID_ARG;
    if (!x || !codes || !scales || !outer) return PMN_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(codes) || !aligned16(scales) || !aligned16(outer)) return PMN_ERR_INVALID_ARG;
    if (h_out && (!swiglu || !aligned16(h_out))) return PMN_ERR_INVALID_ARG;
    if (outer_mode == PMN_OUTER_PER_GROUP) {
        if (swiglu || rows_per_group <= 0 || rows % rows_per_group != 0 || ldx != cols) return PMN_ERR_INVALID_ARG;
        if (!workspace || !aligned16(workspace) ||
            workspace_bytes < (int64_t)quant_groups_scratch_bytes(rows / rows_per_group))
            return PMN_ERR_INVALID_ARG;
    }
    if (rows == 0) return PMN_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const uint16_t *xb = reinterpret_cast<const uint16_t *>(x);
    if (outer_mode == PMN_OUTER_PER_GROUP)
        return launch_quant_groups(xb, rows / rows_per_group, rows_per_group * (cols / 16), four_over_six, codes,
                                   scales, outer, static_cast<uint32_t *>(workspace), s);
    const int nb = (int)((cols / 16 + 31) / 32);
    dim3 block(256), grid((unsigned)((rows + 7) / 8));
    uint16_t *ho = reinterpret_cast<uint16_t *>(h_out);
    const int fos = four_over_six;
    if (nb <= 1) launch_rows<1>(swiglu, grid, block, s, xb, rows, (int)cols, ldx, fos, codes, scales, outer, ho);
    else if (nb <= 2) launch_rows<2>(swiglu, grid, block, s, xb, rows, (int)cols, ldx, fos, codes, scales, outer, ho);
    else if (nb <= 4) launch_rows<4>(swiglu, grid, block, s, xb, rows, (int)cols, ldx, fos, codes, scales, outer, ho);
    else if (nb <= 8) launch_rows<8>(swiglu, grid, block, s, xb, rows, (int)cols, ldx, fos, codes, scales, outer, ho);
    else launch_rows<16>(swiglu, grid, block, s, xb, rows, (int)cols, ldx, fos, codes, scales, outer, ho);
    return launch_status();
}

extern "C" pmn_status pmn_mxfp8_quantize(const void *x, int64_t rows, int64_t cols, int transpose, uint8_t *out,
                                         uint8_t *out_scales, void *stream)
{
    if (rows < 0 || cols < 0 || (transpose != 0 && transpose != 1)) return PMN_ERR_INVALID_ARG;
    if (!x || !out || !out_scales || !aligned16(x) || !aligned16(out)) return PMN_ERR_INVALID_ARG;
    if (transpose == 0 && cols % 32 != 0) return PMN_ERR_INVALID_ARG;
    if (transpose == 1 && (rows % 32 != 0 || cols % 8 != 0)) return PMN_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return PMN_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const uint16_t *xb = reinterpret_cast<const uint16_t *>(x);
    if (!transpose) {
        const int64_t nblocks = rows * cols / 32;
        mxfp8_quant_rowwise_kernel<<<(unsigned)((nblocks + 255) / 256), 256, 0, s>>>(xb, nblocks, cols / 32, out,
                                                                                     out_scales);
    } else {
        if ((rows + RQ_T - 1) / RQ_T > 65535) return PMN_ERR_UNSUPPORTED;  // grid.y: one row of CTAs per 128 rows
        dim3 grid((unsigned)((cols + RQ_T - 1) / RQ_T), (unsigned)((rows + RQ_T - 1) / RQ_T));
        mxfp8_quant_transposed_kernel<false><<<grid, 256, 0, s>>>(xb, rows, cols, out, out_scales, nullptr, nullptr);
    }
    return launch_status();
}

extern "C" pmn_status pmn_mxfp8_quantize_both(const void *x, int64_t rows, int64_t cols, uint8_t *out_rows,
                                              uint8_t *out_rows_scales, uint8_t *out_cols, uint8_t *out_cols_scales,
                                              void *stream)
{
    if (rows < 0 || cols < 0 || rows % 32 != 0 || cols % 32 != 0) return PMN_ERR_INVALID_ARG;
    if (!x || !out_rows || !out_rows_scales || !out_cols || !out_cols_scales) return PMN_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(out_rows) || !aligned16(out_cols)) return PMN_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return PMN_OK;
    if ((rows + RQ_T - 1) / RQ_T > 65535) return PMN_ERR_UNSUPPORTED;  // grid.y: one row of CTAs per 128 rows
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    dim3 grid((unsigned)((cols + RQ_T - 1) / RQ_T), (unsigned)((rows + RQ_T - 1) / RQ_T));
    mxfp8_quant_transposed_kernel<true><<<grid, 256, 0, s>>>(reinterpret_cast<const uint16_t *>(x), rows, cols,
                                                             out_cols, out_cols_scales, out_rows, out_rows_scales);
    return launch_status();
}

extern "C" pmn_status pmn_mxfp8_quantize_swiglu(const void *y, int64_t rows, int64_t f, uint8_t *out,
                                                uint8_t *out_scales, void *h_out, void *stream)
{
    if (rows < 0 || f < 0 || f % 32 != 0) return PMN_ERR_INVALID_ARG;
    if (rows == 0 || f == 0) return PMN_OK;
    if (!y || !out || !out_scales || !aligned16(y) || !aligned16(out)) return PMN_ERR_INVALID_ARG;
    if (h_out && !aligned16(h_out)) return PMN_ERR_INVALID_ARG;
    const int64_t nblocks = rows * (f / 32);
    if (nblocks > 0xFFFFFF00LL) return PMN_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    mxfp8_swiglu_rowwise_kernel<<<(unsigned)((nblocks + 255) / 256), 256, 0, s>>>(
        reinterpret_cast<const uint16_t *>(y), (uint32_t)nblocks, (uint32_t)(f / 32), out, out_scales,
        reinterpret_cast<uint16_t *>(h_out));
    return launch_status();
}

extern "C" pmn_status pmn_requant_transpose_sr_mxfp8(const uint8_t *codes, const uint8_t *scales,
                                                     const float *outer, int outer_mode, int64_t batch,
                                                     int64_t rows, int64_t cols, uint64_t seed, uint32_t tag,
                                                     int rounding, uint8_t *out, uint8_t *out_scales,
                                                     void *stream)
{
    if (batch < 0 || rows < 0 || cols < 0 || rows % 32 != 0 || cols % 32 != 0) return PMN_ERR_INVALID_ARG;
    if (outer_mode != PMN_OUTER_PER_ROW && outer_mode != PMN_OUTER_PER_GROUP) return PMN_ERR_INVALID_ARG;
    if (rounding != PMN_ROUND_SR && rounding != PMN_ROUND_RN) return PMN_ERR_INVALID_ARG;
    if (!codes || !scales || !outer || !out || !out_scales) return PMN_ERR_INVALID_ARG;
    if (!aligned16(codes) || !aligned16(scales) || !aligned16(out) || ((uintptr_t)outer & 3u)) return PMN_ERR_INVALID_ARG;
    if (batch == 0 || rows == 0 || cols == 0) return PMN_OK;
    if ((cols / 16) % 4 != 0) return PMN_ERR_INVALID_ARG;  // 4-byte scale words per 64 columns
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    dim3 grid((unsigned)((cols + 127) / 128), (unsigned)((rows + 127) / 128), (unsigned)batch);
    const bool per_row = outer_mode == PMN_OUTER_PER_ROW;
    const int sr = rounding == PMN_ROUND_SR;
#define PMN_RQ_LAUNCH(PR, C)                                                                                  \
    requant_transpose_kernel<PR, C><<<grid, 128, 0, s>>>(codes, scales, outer, rows, cols, seed, tag, sr, out, \
                                                         out_scales)
    // the expert layer's two row lengths (d_model, d_ff) get compile-time strides
    if (cols == 4096) {
        if (per_row) PMN_RQ_LAUNCH(true, 4096); else PMN_RQ_LAUNCH(false, 4096);
    } else if (cols == 1536) {
        if (per_row) PMN_RQ_LAUNCH(true, 1536); else PMN_RQ_LAUNCH(false, 1536);
    } else {
        if (per_row) PMN_RQ_LAUNCH(true, 0); else PMN_RQ_LAUNCH(false, 0);
    }
#undef PMN_RQ_LAUNCH
    return launch_status();
}

extern "C" pmn_status pmn_requant_transpose_sr_nvfp4(const uint8_t *codes, const uint8_t *scales,
                                                     const float *outer, int outer_mode, int64_t batch,
                                                     int64_t rows, int64_t cols, uint64_t seed, uint32_t tag,
                                                     int rounding, uint8_t *out, uint8_t *out_scales,
                                                     float *out_outer, void *stream)
{
    if (batch < 0 || rows < 0 || cols < 0 || rows % 32 != 0 || cols % 64 != 0) return PMN_ERR_INVALID_ARG;
    if (outer_mode != PMN_OUTER_PER_ROW && outer_mode != PMN_OUTER_PER_GROUP) return PMN_ERR_INVALID_ARG;
    if (rounding != PMN_ROUND_SR && rounding != PMN_ROUND_RN) return PMN_ERR_INVALID_ARG;
    if (batch == 0) return PMN_OK;
    if (!codes || !scales || !outer || !out || !out_scales || !out_outer) return PMN_ERR_INVALID_ARG;
    if (!aligned16(codes) || !aligned16(scales) || !aligned16(out) || ((uintptr_t)outer & 3u) ||
        ((uintptr_t)out_outer & 3u))
        return PMN_ERR_INVALID_ARG;
    if (batch > 65535 || rows * (cols / 64) >= 0xFFFFFF00LL) return PMN_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint32_t *gmax = reinterpret_cast<uint32_t *>(out_outer);  // the largest dec(S) * g, then g'
    if (cudaMemsetAsync(gmax, 0, (size_t)batch * sizeof(uint32_t), s) != cudaSuccess) return PMN_ERR_CUDA;
    const bool per_row = outer_mode == PMN_OUTER_PER_ROW;
    if (rows > 0 && cols > 0) {
        const uint32_t wpr = (uint32_t)(cols / 64), nw = (uint32_t)rows * wpr;
        const uint32_t per_cta = 256u * SMX_PIECES;  // 16-byte pieces per CTA
        nvfp4_scale_max_kernel<<<dim3((nw / 4u + per_cta - 1u) / per_cta, (unsigned)batch), 256, 0, s>>>(
            scales, outer, per_row, (uint32_t)rows, wpr, gmax);
        dim3 grid((unsigned)((cols + 127) / 128), (unsigned)((rows + 127) / 128), (unsigned)batch);
        const int sr = rounding == PMN_ROUND_SR;
        if (per_row)
            requant_transpose_nvfp4_kernel<true><<<grid, 128, 0, s>>>(codes, scales, outer, rows, cols, seed, tag,
                                                                      sr, gmax, out, out_scales);
        else
            requant_transpose_nvfp4_kernel<false><<<grid, 128, 0, s>>>(codes, scales, outer, rows, cols, seed, tag,
                                                                       sr, gmax, out, out_scales);
    }
    nvfp4_outer_finalize_kernel<<<(unsigned)((batch + 255) / 256), 256, 0, s>>>(out_outer, batch);
    return launch_status();
}

extern "C" pmn_status pmn_rht_s2f6_quantize(const float *x, int64_t rows, int64_t cols, uint64_t seed, int8_t *out,
                                            uint8_t *out_scales, void *stream)
{
    if (rows < 0 || cols < 0 || cols % 32 != 0) return PMN_ERR_INVALID_ARG;
    if (!x || !out || !out_scales || !aligned16(x) || !aligned16(out)) return PMN_ERR_INVALID_ARG;
    const int64_t nblocks = rows * cols / 32;
    if (nblocks == 0) return PMN_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    rht_s2f6_kernel<<<(unsigned)((nblocks + 255) / 256), 256, 0, s>>>(x, nblocks, seed, out, out_scales);
    return launch_status();
}

extern "C" pmn_status pmn_combine_receive_s2f6(const int8_t *q, const uint8_t *scales, int64_t rows, int64_t cols,
                                               uint64_t seed, const int32_t *row_index, const float *gates,
                                               int64_t tokens, int k, int out_kind, void *out, void *stream)
{
    if (rows < 0 || cols < 0 || tokens < 0 || cols % 32 != 0 || k < 1 || k > 64) return PMN_ERR_INVALID_ARG;
    if (out_kind != PMN_OUT_BF16 && out_kind != PMN_OUT_F32) return PMN_ERR_INVALID_ARG;
    if (tokens == 0 || cols == 0) return PMN_OK;  // nothing to read or write (empty buffers may be NULL)
    if (!q || !scales || !row_index || !gates || !out) return PMN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(out) || ((uintptr_t)row_index & 3u) || ((uintptr_t)gates & 3u))
        return PMN_ERR_INVALID_ARG;
    const int64_t nb = cols / 32, chunks = (2 * nb + 255) / 256;  // 128 blocks per CTA
    if (tokens > 0x7FFFFFFF || chunks > 65535) return PMN_ERR_INVALID_ARG;
    const dim3 grid((unsigned)tokens, (unsigned)chunks);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
#define PMN_CR_LAUNCH(KF, BF)                                                                           \
    combine_receive_kernel<KF, BF><<<grid, 256, 0, s>>>(q, scales, rows, nb, seed, row_index, gates, \
                                                                  tokens, k, out)
    const bool bf = out_kind == PMN_OUT_BF16;
    if (k == 8) {  // the layer's top-8
        if (bf) PMN_CR_LAUNCH(8, true); else PMN_CR_LAUNCH(8, false);
    } else {
        if (bf) PMN_CR_LAUNCH(0, true); else PMN_CR_LAUNCH(0, false);
    }
#undef PMN_CR_LAUNCH
    return launch_status();
}
