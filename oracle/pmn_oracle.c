/*
 * pmn_oracle.c -- CPU oracle for the block-scaled numerics of one MoE expert
 * layer (NVFP4 forward, MXFP8 backward requantisation with stochastic
 * rounding, RHT + S2F6 combine quantisation).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain definition that the
 * CUDA library is checked against.  Only the test-suite, the smoke check and
 * the benchmark's CPU-baseline leg may load it; the product path never does.
 * It shares no code, header, table or constant generator with the CUDA path.
 *
 * Every function follows one passage of the pages ("Thinking Machines on
 * training Inkling 2 Small with native 4-bit forward passes", arex-research.com,
 * and the lhc.media page that repeats it), cited by page and section:
 *   [Bits]   section "更少的比特换更快的算术" (fewer bits, faster arithmetic)
 *   [Layers] section "只把专家层的前向传播降到 4-bit" (only the expert forward in 4-bit)
 *   [SR]     section "转置打散分组,随机舍入保住期望值" (transpose regroups, SR keeps E)
 *   [NVLink] section "计算提速后,NVLink 通信成了新瓶颈" (dispatch / combine)
 *   [Cost]   section "配方的代价" (4/6, outer scales)
 * Where the pages are silent the plainest reading is taken; each such reading
 * is named in a comment starting with "Reading:".
 *
 * Arithmetic rules.  Every decision that produces an integer (a code, a scale
 * byte) is taken in IEEE binary32 with one rounding per operation, as the
 * kernels take it: compile with -ffp-contract=off, no fast-math.  Values that
 * the definition fixes exactly (a scaled value, a rounding fraction) are held
 * in binary64, where they are exact.  Grid rounding is written from the
 * definition (nearest grid point, ties to the even mantissa) on exact values.
 *
 * Parity status: every exported function is pinned by the oracle tests
 * (worked examples from the pages, closed forms, library codecs, brute force).
 */
#include <math.h>
#include <stdlib.h>
#include <stdint.h>
#include <string.h>
#include <omp.h>

#define ORC_API __attribute__((visibility("default")))

/* ------------------------------------------------------------------------ */
/* Philox4x32-10: Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As   */
/* Easy as 1, 2, 3", SC'11.  Ten rounds; each round multiplies words 0 and 2 */
/* by the two round multipliers, swaps the halves and mixes in the key; the  */
/* key is bumped by the two Weyl constants between rounds.                   */
/* ------------------------------------------------------------------------ */
ORC_API void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        uint64_t p0 = (uint64_t)0xD2511F53u * (uint64_t)c0;
        uint64_t p1 = (uint64_t)0xCD9E8D57u * (uint64_t)c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n1 = lo1;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        uint32_t n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* Random bits for element i of a tensor.  Reading (the pages say only that
 * SR is hardware-accelerated on Blackwell; this library takes the layout that
 * Blackwell's stochastic-rounding conversion consumes): four consecutive
 * elements share one 32-bit Philox word; element 4w+0 takes the word's low 16
 * bits, 4w+1 the same 16 bits in reversed bit order, 4w+2 the high 16 bits and
 * 4w+3 the high 16 bits reversed.  The Philox counter is (j lo32, j hi32, tag,
 * 0) with j = i / 16, the key (seed lo32, seed hi32); word (i / 4) % 4. */
static uint32_t rev16(uint32_t x)
{
    uint32_t r = 0;
    for (int b = 0; b < 16; ++b)
        if (x & (1u << b)) r |= 1u << (15 - b);
    return r;
}

ORC_API uint32_t orc_sr_bits16(uint64_t seed, uint32_t tag, uint64_t i)
{
    uint64_t j = i >> 4;
    uint32_t ctr[4] = {(uint32_t)j, (uint32_t)(j >> 32), tag, 0u};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t w[4];
    orc_philox4x32_10(ctr, key, w);
    uint32_t word = w[(i >> 2) & 3u];
    uint32_t half = (i & 2u) ? (word >> 16) : (word & 0xFFFFu);
    return (i & 1u) ? rev16(half) : half;
}

/* ------------------------------------------------------------------------ */
/* Element and scale formats.                                                */
/* E2M1 [SR]: 16 codes, sign bit 3, magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6.  */
/* E4M3 (OCP MX v1.0): bias 7, subnormals m/8 * 2^-6, max 448, S.1111.111   */
/* is NaN.  E8M0: 2^(b - 127), 0xFF is NaN.  S2F6 [NVLink]: int8 k -> k/64. */
/* ------------------------------------------------------------------------ */
ORC_API double orc_e2m1_value(uint32_t code)
{
    static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
    double v = mag[code & 7u];
    return (code & 8u) ? -v : v;
}

ORC_API double orc_e4m3_value(uint32_t b)
{
    uint32_t e = (b >> 3) & 15u, m = b & 7u;
    double v;
    if (e == 15u && m == 7u) return NAN;
    if (e == 0u) v = ldexp((double)m, -9);
    else v = ldexp((double)(8u + m), (int)e - 10);
    return (b & 0x80u) ? -v : v;
}

ORC_API double orc_e8m0_value(uint32_t b)
{
    if ((b & 0xFFu) == 0xFFu) return NAN;
    return ldexp(1.0, (int)(b & 0xFFu) - 127);
}

ORC_API double orc_s2f6_value(int32_t k) { return (double)(int8_t)k / 64.0; }

/* floor(log2(a)) for a finite a > 0, exactly */
static int ilog2_floor(double a)
{
    int E;
    (void)frexp(a, &E); /* a = f * 2^E, f in [0.5, 1) */
    return E - 1;
}

/* Nearest point of a binary minifloat grid (mbits mantissa bits, smallest
 * normal exponent emin, largest finite value maxv), ties to the even mantissa,
 * saturating above maxv.  a >= 0 and exact. */
static double rne_grid(double a, int mbits, int emin, double maxv)
{
    if (a == 0.0) return 0.0;
    if (isinf(a)) return maxv;
    int L = ilog2_floor(a);
    if (L < emin) L = emin;
    double ulp = ldexp(1.0, L - mbits);
    double q = a / ulp;       /* exact: ulp is a power of two */
    double n = nearbyint(q);  /* default rounding mode: nearest, ties to even */
    double r = n * ulp;
    return r > maxv ? maxv : r;
}

/* Stochastic rounding on the same grid [SR]: the two neighbours lo <= a < hi,
 * f = (a - lo) / (hi - lo).  Reading: 16 random bits are added to the leading
 * 16 bits of the fraction, f16 = floor(f * 2^16), and a carry rounds away from
 * zero: the result is hi iff rb16 + f16 >= 2^16.  So P(hi) = f16 / 2^16 and
 * E[result] = a to within 2^-16 of a grid step (2.25 between 2 and 3 goes to
 * 3 with p = 1/4 exactly, as in the pages' example). */
static double sr_grid(double a, uint32_t rb16, int mbits, int emin, double maxv)
{
    if (a == 0.0) return 0.0;
    int L = ilog2_floor(a);
    if (L < emin) L = emin;
    double ulp = ldexp(1.0, L - mbits);
    double lo = floor(a / ulp) * ulp;
    double f = (a - lo) / ulp;            /* exact */
    double f16 = floor(f * 65536.0);      /* exact */
    double r = ((double)(rb16 & 0xFFFFu) + f16 >= 65536.0) ? lo + ulp : lo;
    return r > maxv ? maxv : r;
}

static uint32_t e2m1_encode_mag(double v)
{
    static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
    for (uint32_t c = 0; c < 8; ++c)
        if (mag[c] == v) return c;
    return 0xFFu; /* not on the grid: caller bug */
}

static uint32_t e4m3_encode_mag(double v)
{
    if (v == 0.0) return 0u;
    if (v < ldexp(1.0, -6)) return (uint32_t)(v / ldexp(1.0, -9)); /* subnormal */
    int L = ilog2_floor(v);
    uint32_t m = (uint32_t)((v / ldexp(1.0, L) - 1.0) * 8.0);
    return ((uint32_t)(L + 7) << 3) | m;
}

/* binary32 value -> E2M1 code, round to nearest even, saturating (3.2 -> 3,
 * [Bits]; the value set of [SR]).  The sign is kept, so -0 and small negative
 * values give the code 0x8. */
ORC_API uint32_t orc_e2m1_rne(float v)
{
    double a = fabs((double)v);
    uint32_t s = signbit(v) ? 8u : 0u;
    return s | e2m1_encode_mag(rne_grid(a, 1, 0, 6.0));
}

/* binary32 value -> E4M3 byte, round to nearest even, saturating at 448. */
ORC_API uint32_t orc_e4m3_rne(float v)
{
    double a = fabs((double)v);
    uint32_t s = signbit(v) ? 0x80u : 0u;
    return s | e4m3_encode_mag(rne_grid(a, 3, -6, 448.0));
}

/* exact value y -> E4M3 byte by stochastic rounding with 16 random bits */
ORC_API uint32_t orc_e4m3_sr(double y, uint32_t rb16)
{
    uint32_t s = signbit(y) ? 0x80u : 0u;
    return s | e4m3_encode_mag(sr_grid(fabs(y), rb16, 3, -6, 448.0));
}

/* exact value y -> E2M1 code by stochastic rounding (used for the pages'
 * worked example: 2.25 on the FP4 grid goes to 2 with p = 3/4, 3 with 1/4) */
ORC_API uint32_t orc_e2m1_sr(double y, uint32_t rb16)
{
    uint32_t s = signbit(y) ? 8u : 0u;
    return s | e2m1_encode_mag(sr_grid(fabs(y), rb16, 1, 0, 6.0));
}

/* RN of an exact value to bfloat16 (bits) -- finite, normal range */
ORC_API uint32_t orc_bf16_rne(double v)
{
    double a = fabs(v);
    double r = rne_grid(a, 7, -126, ldexp(255.0, 120));
    float f = (float)r; /* exact: r is on the bfloat16 grid */
    uint32_t bits;
    memcpy(&bits, &f, 4);
    bits >>= 16;
    return signbit(v) ? (bits | 0x8000u) : bits;
}

static float bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* ------------------------------------------------------------------------ */
/* NVFP4 block quantisation [SR], [Cost].                                    */
/* One block = 16 contiguous values.  With outer scale g and candidate m:   */
/*   s  = amax_b / (m * g)            (binary32)                             */
/*   S  = RNE_E4M3(s)                 (scale byte)                           */
/*   sd = dec(S) * g                  (binary32)                             */
/*   r  = 1 / sd  (0 when sd == 0)    (binary32)                             */
/*   c_i = RNE_E2M1(x_i * r)          (codes)                                */
/* With g = 1 and amax -54 this gives code -6 and scale 9 ([SR] example).   */
/* 4/6 [Cost]: candidates m = 6 and m = 4; the one with the smaller sum of  */
/* squared dequantisation errors wins, ties to 6.  Reading: the error is     */
/* summed in binary32 with the tree t[i] = e[i] + e[i+8], then + [i+4],     */
/* + [i+2], + [i+1].                                                         */
/* ------------------------------------------------------------------------ */
static float deq_nvfp4(uint32_t code, uint32_t sbyte, float g)
{
    float cs = (float)(orc_e2m1_value(code) * orc_e4m3_value(sbyte)); /* exact */
    return cs * g;
}

static float block_try(const float x[16], float amax, float g, float m,
                       uint8_t codes[16], uint8_t *sbyte)
{
    float denom = m * g;
    float s = amax / denom;
    uint32_t S = orc_e4m3_rne(s);
    float sd = (float)orc_e4m3_value(S) * g;
    float r = (sd == 0.0f) ? 0.0f : 1.0f / sd;
    float e[16];
    for (int i = 0; i < 16; ++i) {
        float p = x[i] * r;
        codes[i] = (uint8_t)orc_e2m1_rne(p);
        float d = x[i] - deq_nvfp4(codes[i], S, g);
        e[i] = d * d;
    }
    for (int h = 8; h >= 1; h >>= 1)
        for (int i = 0; i < h; ++i) e[i] = e[i] + e[i + h];
    *sbyte = (uint8_t)S;
    return e[0];
}

ORC_API int orc_nvfp4_quantize_block(const float x[16], float g, int four_over_six,
                                     uint8_t codes[16], uint8_t *sbyte)
{
    float amax = 0.0f;
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
    uint8_t c6[16], s6;
    float err6 = block_try(x, amax, g, 6.0f, c6, &s6);
    if (four_over_six) {
        uint8_t c4[16], s4;
        float err4 = block_try(x, amax, g, 4.0f, c4, &s4);
        if (err4 < err6) {
            memcpy(codes, c4, 16);
            *sbyte = s4;
            return 4;
        }
    }
    memcpy(codes, c6, 16);
    *sbyte = s6;
    return 6;
}

/* Outer scale [Cost]: one binary32 scale per token (activations) or per
 * expert (weights), following the recipe the pages credit to Composer 2.
 * Reading (no formula on the pages): g = amax / (6 * 448), or amax / (4 * 448)
 * with 4/6 on, so that every candidate block scale fits E4M3; g = 1 when the
 * group is all zero. */
static float outer_from_amax(float amax, int four_over_six)
{
    float M = four_over_six ? 1792.0f : 2688.0f;
    return amax == 0.0f ? 1.0f : amax / M;
}

enum { ORC_OUTER_PER_ROW = 0, ORC_OUTER_PER_GROUP = 1, ORC_OUTER_GIVEN = 2 };
enum { ORC_IN_BF16 = 0 };

/* x: bf16 [rows, cols] with leading dimension ldx (elements).
 * outer_mode PER_ROW: one g per row (tokens).  PER_GROUP: one g per row range
 * [offsets[k], offsets[k+1]) (experts; one range = per tensor).  GIVEN: outer
 * holds one g per row on entry.  Outputs: codes [rows, cols/2] (element 2i in
 * the low nibble), scales [rows, cols/16], outer [rows] (PER_ROW/GIVEN) or
 * [num_groups] (PER_GROUP), choice [rows, cols/16] (4 or 6; may be NULL). */
ORC_API void orc_nvfp4_quantize(const uint16_t *x, int64_t rows, int64_t cols, int64_t ldx,
                                int outer_mode, const int64_t *offsets, int64_t num_groups,
                                int four_over_six, uint8_t *codes, uint8_t *scales,
                                float *outer, uint8_t *choice)
{
    if (outer_mode == ORC_OUTER_PER_GROUP) {
        #pragma omp parallel for schedule(dynamic)
        for (int64_t k = 0; k < num_groups; ++k) {
            float amax = 0.0f;
            for (int64_t r = offsets[k]; r < offsets[k + 1]; ++r)
                for (int64_t c = 0; c < cols; ++c)
                    amax = fmaxf(amax, fabsf(bf16_to_f32(x[r * ldx + c])));
            outer[k] = outer_from_amax(amax, four_over_six);
        }
    }
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        float g;
        if (outer_mode == ORC_OUTER_PER_ROW) {
            float amax = 0.0f;
            for (int64_t c = 0; c < cols; ++c)
                amax = fmaxf(amax, fabsf(bf16_to_f32(x[r * ldx + c])));
            g = outer_from_amax(amax, four_over_six);
            outer[r] = g;
        } else if (outer_mode == ORC_OUTER_PER_GROUP) {
            int64_t k = 0;
            while (k + 1 < num_groups && r >= offsets[k + 1]) ++k;
            g = outer[k];
        } else {
            g = outer[r];
        }
        for (int64_t b = 0; b < cols / 16; ++b) {
            float xb[16];
            uint8_t cb[16], sb;
            for (int i = 0; i < 16; ++i) xb[i] = bf16_to_f32(x[r * ldx + b * 16 + i]);
            int m = orc_nvfp4_quantize_block(xb, g, four_over_six, cb, &sb);
            for (int i = 0; i < 16; i += 2)
                codes[r * (cols / 2) + b * 8 + i / 2] = (uint8_t)(cb[i] | (cb[i + 1] << 4));
            scales[r * (cols / 16) + b] = sb;
            if (choice) choice[r * (cols / 16) + b] = (uint8_t)m;
        }
    }
}

/* Canonical binary32 dequantisation d = (dec(c) * dec(S)) * g; the first
 * product is exact. outer: one g per row, or per row-group of rows_per_outer */
ORC_API void orc_nvfp4_dequant_f32(const uint8_t *codes, const uint8_t *scales, const float *outer,
                                   int64_t rows_per_outer, int64_t rows, int64_t cols, float *out)
{
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        float g = outer ? outer[r / rows_per_outer] : 1.0f;
        for (int64_t c = 0; c < cols; ++c) {
            uint32_t byte = codes[r * (cols / 2) + c / 2];
            uint32_t code = (c & 1) ? (byte >> 4) : (byte & 15u);
            out[r * cols + c] = deq_nvfp4(code, scales[r * (cols / 16) + c / 16], g);
        }
    }
}

/* dec(c) * dec(S) in binary64, without the outer scale (GEMM operands) */
ORC_API void orc_nvfp4_dequant_f64(const uint8_t *codes, const uint8_t *scales,
                                   int64_t rows, int64_t cols, double *out)
{
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) {
            uint32_t byte = codes[r * (cols / 2) + c / 2];
            uint32_t code = (c & 1) ? (byte >> 4) : (byte & 15u);
            out[r * cols + c] = orc_e2m1_value(code) * orc_e4m3_value(scales[r * (cols / 16) + c / 16]);
        }
}

/* ------------------------------------------------------------------------ */
/* MXFP8 (E4M3 values, one E8M0 scale per 32) [Bits], [SR].                  */
/* Scale of a 32-block: the smallest integer e with amax <= 448 * 2^e,       */
/* clamped to [-127, 127]; e = -127 for an all-zero block; byte e + 127.     */
/* Reading: this is the rule that never clips, so SR stays unbiased [SR].   */
/* ------------------------------------------------------------------------ */
ORC_API int orc_e8m0_exponent(double amax, double top)
{
    if (amax == 0.0) return -127;
    int e = ilog2_floor(amax) - ilog2_floor(top);
    while (amax > ldexp(top, e)) ++e;
    while (amax <= ldexp(top, e - 1)) --e;
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return e;
}

/* Dequantise -> transpose -> requantise [SR].  Input: NVFP4 tensor [batch,
 * rows, cols] (codes [.., cols/2], scales [.., cols/16]) with binary32 outer
 * scale per row (outer_mode 0, outer[batch*rows]) or per batch entry
 * (outer_mode 1, outer[batch]).  rows must be a multiple of 32 (expert
 * segments padded with zero rows).  Output: E4M3 [batch, cols, rows] and E8M0
 * [batch, cols, rows/32]; 32-blocks run along the original rows.  rounding 0:
 * stochastic with orc_sr_bits16(seed, tag, i), i the row-major output index;
 * rounding 1: nearest even. */
ORC_API void orc_requant_transpose_mxfp8_window(const uint8_t *codes, const uint8_t *scales,
                                                const float *outer, int outer_mode, int64_t batch,
                                                int64_t rows, int64_t cols, uint64_t seed, uint32_t tag,
                                                int rounding, uint8_t *out, uint8_t *out_sc,
                                                int64_t b_begin, int64_t rows_total, int64_t r_begin);

ORC_API void orc_requant_transpose_mxfp8(const uint8_t *codes, const uint8_t *scales,
                                         const float *outer, int outer_mode, int64_t batch,
                                         int64_t rows, int64_t cols, uint64_t seed, uint32_t tag,
                                         int rounding, uint8_t *out, uint8_t *out_sc)
{
    orc_requant_transpose_mxfp8_window(codes, scales, outer, outer_mode, batch, rows, cols, seed, tag,
                                       rounding, out, out_sc, 0, rows, 0);
}

/* The same computation for a window of a larger tensor (sampled checks at
 * full size): the inputs hold batch entries b_begin .. b_begin+batch-1 and,
 * of each, rows r_begin .. r_begin+rows-1 of rows_total (r_begin and rows
 * multiples of 32).  The random bits use the element's index in the FULL
 * output [*, cols, rows_total].  Output: [batch, cols, rows] (+ scales). */
ORC_API void orc_requant_transpose_mxfp8_window(const uint8_t *codes, const uint8_t *scales,
                                                const float *outer, int outer_mode, int64_t batch,
                                                int64_t rows, int64_t cols, uint64_t seed, uint32_t tag,
                                                int rounding, uint8_t *out, uint8_t *out_sc,
                                                int64_t b_begin, int64_t rows_total, int64_t r_begin)
{
    #pragma omp parallel for collapse(2) schedule(static)
    for (int64_t b = 0; b < batch; ++b)
        for (int64_t c = 0; c < cols; ++c)
            for (int64_t rb = 0; rb < rows / 32; ++rb) {
                float d[32];
                double amax = 0.0;
                for (int j = 0; j < 32; ++j) {
                    int64_t r = rb * 32 + j;
                    int64_t src = b * rows + r;
                    float g = outer_mode == 0 ? outer[src] : outer[b];
                    uint32_t byte = codes[src * (cols / 2) + c / 2];
                    uint32_t code = (c & 1) ? (byte >> 4) : (byte & 15u);
                    d[j] = deq_nvfp4(code, scales[src * (cols / 16) + c / 16], g);
                    amax = fmax(amax, fabs((double)d[j]));
                }
                int e = orc_e8m0_exponent(amax, 448.0);
                int64_t orow = (b * cols + c) * rows;
                int64_t grow = ((b_begin + b) * cols + c) * rows_total + r_begin;
                for (int j = 0; j < 32; ++j) {
                    int64_t i = orow + rb * 32 + j;
                    int64_t gi = grow + rb * 32 + j;
                    double y = ldexp((double)d[j], -e); /* exact */
                    uint32_t q;
                    if (rounding == 0) q = orc_e4m3_sr(y, orc_sr_bits16(seed, tag, (uint64_t)gi));
                    else {
                        uint32_t sg = signbit(y) ? 0x80u : 0u;
                        q = sg | e4m3_encode_mag(rne_grid(fabs(y), 3, -6, 448.0));
                    }
                    out[i] = (uint8_t)q;
                }
                out_sc[(b * cols + c) * (rows / 32) + rb] = (uint8_t)(e + 127);
            }
}

/* Dequantise -> transpose -> requantise to NVFP4 with stochastic rounding:
 * the FP4 backward the pages name as future work, the same [SR] steps as the
 * MXFP8 requantisation above with the NVFP4 format of the forward pass.
 * Input as orc_requant_transpose_mxfp8; d = (code * S) * g in binary32.
 * Output per batch entry: codes [cols, rows/2] (element 2i in the low
 * nibble), E4M3 scales [cols, rows/16] (16-blocks along the original rows),
 * binary32 outer scale out_outer[b].
 * Reading (outer scale; the pages give none for the transposed tensor): the
 * entry's largest block scale times its outer scale, sd = dec(S) * g
 * (binary32), over every input block of the entry, divided by 448:
 * g' = max sd / 448 (binary32), g' = 1 when every scale is zero.  So every
 * |d| <= 6 * dec(S) * g fits under 6 * 448 * g', and zero (padding) blocks do
 * not count.
 * Reading (block scale; unbiased SR needs values that do not clip, as the
 * MXFP8 exponent rule): s = amax / RN(6 * g'), S' = the smallest E4M3 value
 * >= s (saturating at 448); sd' = dec(S') * g'; r = 1 / sd' (0 if sd' = 0);
 * y = d * r (all binary32); code = SR_E2M1(y) with orc_sr_bits16(seed, tag,
 * i), i the element's row-major index in the output [batch, cols, rows] of
 * the full tensor (b_begin shifts the entries), or RNE_E2M1(y) (rounding 1).
 * The sign is kept, as in the forward codes. */
static double ru_e4m3(double s)
{
    if (s <= 0.0) return 0.0;
    if (s >= 448.0) return 448.0;
    int L = ilog2_floor(s);
    if (L < -6) L = -6;
    double ulp = ldexp(1.0, L - 3);
    return ceil(s / ulp) * ulp; /* exact: ulp is a power of two */
}

ORC_API void orc_requant_transpose_nvfp4(const uint8_t *codes, const uint8_t *scales, const float *outer,
                                         int outer_mode, int64_t batch, int64_t rows, int64_t cols,
                                         uint64_t seed, uint32_t tag, int rounding, uint8_t *out_codes,
                                         uint8_t *out_sc, float *out_outer, int64_t b_begin)
{
    for (int64_t b = 0; b < batch; ++b) {
        float m = 0.0f;
        for (int64_t r = 0; r < rows; ++r) {
            int64_t src = b * rows + r;
            float g = outer_mode == 0 ? outer[src] : outer[b];
            for (int64_t k = 0; k < cols / 16; ++k) {
                float sd = (float)orc_e4m3_value(scales[src * (cols / 16) + k]) * g;
                if (sd > m) m = sd;
            }
        }
        out_outer[b] = m == 0.0f ? 1.0f : m / 448.0f;
    }
    #pragma omp parallel for collapse(2) schedule(static)
    for (int64_t b = 0; b < batch; ++b)
        for (int64_t c = 0; c < cols; ++c) {
            const float gp = out_outer[b];
            const float six_g = 6.0f * gp;
            for (int64_t rb = 0; rb < rows / 16; ++rb) {
                float d[16];
                float amax = 0.0f;
                for (int j = 0; j < 16; ++j) {
                    int64_t src = b * rows + rb * 16 + j;
                    float g = outer_mode == 0 ? outer[src] : outer[b];
                    uint32_t byte = codes[src * (cols / 2) + c / 2];
                    uint32_t code = (c & 1) ? (byte >> 4) : (byte & 15u);
                    d[j] = deq_nvfp4(code, scales[src * (cols / 16) + c / 16], g);
                    amax = fmaxf(amax, fabsf(d[j]));
                }
                float s = amax / six_g;
                uint32_t S = e4m3_encode_mag(ru_e4m3((double)s));
                float sd = (float)orc_e4m3_value(S) * gp;
                float r = sd == 0.0f ? 0.0f : 1.0f / sd;
                int64_t orow = (b * cols + c) * rows;
                int64_t grow = ((b_begin + b) * cols + c) * rows;
                for (int j = 0; j < 16; j += 2) {
                    uint32_t q[2];
                    for (int t = 0; t < 2; ++t) {
                        float y = d[j + t] * r;
                        if (rounding == 0)
                            q[t] = orc_e2m1_sr((double)y, orc_sr_bits16(seed, tag, (uint64_t)(grow + rb * 16 + j + t)));
                        else
                            q[t] = orc_e2m1_rne(y);
                    }
                    out_codes[(orow + rb * 16 + j) / 2] = (uint8_t)(q[0] | (q[1] << 4));
                }
                out_sc[(b * cols + c) * (rows / 16) + rb] = (uint8_t)S;
            }
        }
}

/* bf16 -> MXFP8 with round to nearest even (used for dY).  Reading: the pages
 * ask for SR on the saved forward tensors only; gradients take RN.
 * transpose 0: out [rows, cols], scales [rows, cols/32] (blocks along cols).
 * transpose 1: out [cols, rows], scales [cols, rows/32] (blocks along rows). */
ORC_API void orc_mxfp8_quantize(const uint16_t *x, int64_t rows, int64_t cols, int transpose,
                                uint8_t *out, uint8_t *out_sc)
{
    int64_t outer_n = transpose ? cols : rows;
    int64_t inner_n = transpose ? rows : cols;
    #pragma omp parallel for schedule(static)
    for (int64_t o = 0; o < outer_n; ++o)
        for (int64_t ib = 0; ib < inner_n / 32; ++ib) {
            float v[32];
            double amax = 0.0;
            for (int j = 0; j < 32; ++j) {
                int64_t in = ib * 32 + j;
                v[j] = transpose ? bf16_to_f32(x[in * cols + o]) : bf16_to_f32(x[o * cols + in]);
                amax = fmax(amax, fabs((double)v[j]));
            }
            int e = orc_e8m0_exponent(amax, 448.0);
            for (int j = 0; j < 32; ++j) {
                double y = ldexp((double)v[j], -e);
                uint32_t s = signbit(y) ? 0x80u : 0u;
                out[o * inner_n + ib * 32 + j] = (uint8_t)(s | e4m3_encode_mag(rne_grid(fabs(y), 3, -6, 448.0)));
            }
            out_sc[o * (inner_n / 32) + ib] = (uint8_t)(e + 127);
        }
}

/* E4M3 * 2^(E8M0) in binary64: MXFP8 dequantisation along the last axis */
ORC_API void orc_mxfp8_dequant_f64(const uint8_t *q, const uint8_t *sc, int64_t rows, int64_t cols,
                                   double *out)
{
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c)
            out[r * cols + c] = orc_e4m3_value(q[r * cols + c]) * orc_e8m0_value(sc[r * (cols / 32) + c / 32]);
}

/* ------------------------------------------------------------------------ */
/* Combine quantisation [NVLink]: 32-point randomised Hadamard transform,    */
/* then block-scaled S2F6 (int8 k, value k/64, one scale per 32 values).     */
/* Reading: sigma in {+-1}^32 is bit j of Philox word 0 at counter           */
/* (0, 0, 5, 0) with key = seed (bit set -> -1), one sigma for every block;  */
/* z = RN(1/sqrt(32)) * FWHT(sigma * x), butterflies h = 1, 2, 4, 8, 16 in   */
/* binary32; scale exponent = smallest e with amax <= (127/64) * 2^e, byte   */
/* e + 127 (E8M0); k = RNE(z * 2^(6 - e)).                                   */
/* ------------------------------------------------------------------------ */
ORC_API uint32_t orc_rht_sign_word(uint64_t seed)
{
    uint32_t ctr[4] = {0u, 0u, 5u, 0u};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t w[4];
    orc_philox4x32_10(ctr, key, w);
    return w[0];
}

ORC_API float orc_rsqrt32(void) { return (float)(1.0 / sqrt(32.0)); }

/* One 32-block: sign flip, fast Walsh-Hadamard transform, normalisation. */
ORC_API void orc_rht32(const float x[32], uint32_t sigma, float z[32])
{
    float v[32];
    for (int j = 0; j < 32; ++j) v[j] = ((sigma >> j) & 1u) ? -x[j] : x[j];
    for (int h = 1; h < 32; h <<= 1)
        for (int i = 0; i < 32; i += 2 * h)
            for (int j = i; j < i + h; ++j) {
                float a = v[j], b = v[j + h];
                v[j] = a + b;
                v[j + h] = a - b;
            }
    float rs = orc_rsqrt32();
    for (int j = 0; j < 32; ++j) z[j] = v[j] * rs;
}

/* x: binary32 [rows, cols] (cols % 32 == 0) -> int8 [rows, cols], E8M0
 * [rows, cols/32] */
ORC_API void orc_rht_s2f6(const float *x, int64_t rows, int64_t cols, uint64_t seed,
                          int8_t *out, uint8_t *out_sc)
{
    uint32_t sigma = orc_rht_sign_word(seed);
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < cols / 32; ++b) {
            float z[32];
            orc_rht32(x + r * cols + b * 32, sigma, z);
            double amax = 0.0;
            for (int j = 0; j < 32; ++j) amax = fmax(amax, fabs((double)z[j]));
            int e = orc_e8m0_exponent(amax, 127.0 / 64.0);
            for (int j = 0; j < 32; ++j) {
                double k = nearbyint(ldexp((double)z[j], 6 - e));
                if (k > 127.0) k = 127.0;
                if (k < -128.0) k = -128.0;
                out[r * cols + b * 32 + j] = (int8_t)k;
            }
            out_sc[r * (cols / 32) + b] = (uint8_t)(e + 127);
        }
}

/* Receive side of the combine (the inverse the pages call exact): decode
 * k/64 * 2^e, apply H/sqrt(32) again (it is its own inverse) and the signs.
 * Binary64 throughout. */
ORC_API void orc_s2f6_dequant_inverse_rht(const int8_t *q, const uint8_t *sc, int64_t rows,
                                          int64_t cols, uint64_t seed, double *out)
{
    uint32_t sigma = orc_rht_sign_word(seed);
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < cols / 32; ++b) {
            double v[32];
            double s = orc_e8m0_value(sc[r * (cols / 32) + b]);
            for (int j = 0; j < 32; ++j) v[j] = orc_s2f6_value(q[r * cols + b * 32 + j]) * s;
            for (int h = 1; h < 32; h <<= 1)
                for (int i = 0; i < 32; i += 2 * h)
                    for (int j = i; j < i + h; ++j) {
                        double a = v[j], c = v[j + h];
                        v[j] = a + c;
                        v[j + h] = a - c;
                    }
            for (int j = 0; j < 32; ++j) {
                double y = v[j] / sqrt(32.0);
                out[r * cols + b * 32 + j] = ((sigma >> j) & 1u) ? -y : y;
            }
        }
}

/* Element-wise orc_bf16_rne over an array (binary64 in, bfloat16 bits out). */
/* Receive side of the combine, gathered back into token order [NVLink]: each
 * token t sums, over its k expert choices i = 0 .. k-1 in order,
 *   gate[t, i] * R(row_index[t, i])
 * where R(r) is routed row r decoded and transformed back as in
 * orc_s2f6_dequant_inverse_rht.  Binary64 throughout; out double [tokens, cols].
 * Reading: the pages send each expert output back to the token's GPU and do
 * not say how the k results are merged; the plainest reading is the weighted
 * sum of an MoE combine, with the router's gate weights passed in as inputs.
 * A negative row index is a dropped choice and adds nothing. */
ORC_API void orc_combine_receive(const int8_t *q, const uint8_t *sc, int64_t rows, int64_t cols,
                                 uint64_t seed, const int64_t *row_index, const float *gates,
                                 int64_t tokens, int64_t k, double *out)
{
    (void)rows;
    #pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < tokens; ++t) {
        double *y = out + t * cols;
        double *row = (double *)malloc((size_t)cols * sizeof(double));
        for (int64_t c = 0; c < cols; ++c) y[c] = 0.0;
        for (int64_t i = 0; i < k; ++i) {
            int64_t r = row_index[t * k + i];
            if (r < 0) continue;
            orc_s2f6_dequant_inverse_rht(q + r * cols, sc + r * (cols / 32), 1, cols, seed, row);
            double g = (double)gates[t * k + i];
            for (int64_t c = 0; c < cols; ++c) y[c] += g * row[c];
        }
        free(row);
    }
}

ORC_API void orc_bf16_rne_array(const double *v, int64_t n, uint16_t *out)
{
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = (uint16_t)orc_bf16_rne(v[i]);
}

/* Threads of the oracle's OpenMP loops (the CPU baseline times all host
 * cores and one thread); no effect on any result. */
ORC_API void orc_set_num_threads(int n) { omp_set_num_threads(n > 0 ? n : 1); }
ORC_API int orc_max_threads(void) { return omp_get_max_threads(); }
