// numerics.cuh -- device-side format codecs, rounding and random bits for the
// block-scaled MoE numerics (GB300, sm_103a).
//
// Formats (page "Thinking Machines ... Inkling 2 Small", arex-research.com):
//   E2M1 codes {+-0, 0.5, 1, 1.5, 2, 3, 4, 6}       section [SR], first paragraph
//   E4M3 block scales of NVFP4, E8M0 scales of MXFP8  section [SR] / [Bits]
//   S2F6 combine format, int8 k = value * 64           section [NVLink]
// E4M3 / E8M0 bit layouts follow the OCP Microscaling spec v1.0.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace pmn {

// ---------------------------------------------------------------- SwiGLU
// h = silu(a) * b = a * b / (1 + e^-a) in binary32, with the hardware's
// approximate exponential and division (the __expf / __fdividef intrinsics:
// a few dozen binary32 ulps at most for |a| <= 40; for a < -87 the quotient
// is 0, against a true |silu(a)| < 2^-120 |a|).  Every SwiGLU of the library
// (the w1 GEMM epilogue, the row quantisers' SwiGLU input modes) uses this
// one function, so they give the same h bit for bit; h is rounded to bf16
// afterwards, a step of 2^-8 relative.
__device__ __forceinline__ float silu_mul(float a, float b)
{
    return __fmul_rn(__fdividef(a, __fadd_rn(1.0f, __expf(-a))), b);
}

// ---------------------------------------------------------------- decoders
// E2M1 magnitude code m (0..7): e = m >> 1, mantissa bit m & 1; e == 0 is the
// subnormal 0 / 0.5, otherwise (1 + mant/2) * 2^(e-1).  Built as float bits.
__device__ __forceinline__ float e2m1_to_f32(uint32_t code)
{
    uint32_t m = code & 7u;
    uint32_t bits = (m >= 2u) ? ((((m >> 1) + 126u) << 23) | ((m & 1u) << 22))
                              : (m == 1u ? 0x3F000000u : 0u);
    return __uint_as_float(bits | ((code & 8u) << 28));
}

// Two E2M1 codes (one byte; bits 3:0 = element 0, in the low half) decoded
// by the hardware to f16x2 and multiplied by an E4M3 scale held as f16x2:
// e2m1 (2 significant bits) x E4M3 (4 bits) is exact in f16 (range 2^-10 ..
// 2688).  Returns the two exact products as f16x2 bits.
__device__ __forceinline__ uint32_t e2m1x2_mul_h2(uint32_t byte, uint32_t scale_h2)
{
    uint32_t h2, p;
    const uint16_t b16 = (uint16_t)(byte & 0xFFu);
    asm("{\n\t.reg .b8 lo, hi;\n\tmov.b16 {lo, hi}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, lo;\n\t}" : "=r"(h2) : "h"(b16));
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(p) : "r"(h2), "r"(scale_h2));
    return p;
}

// The four bytes of a code word at once (element 2k, 2k+1 of byte k in the
// low, high half of out[k]), each times the f16x2 scale: exact as above.
__device__ __forceinline__ void e2m1x8_mul_h2(uint32_t word, uint32_t scale_h2, uint32_t (&out)[4])
{
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t.reg .b32 t0, t1, t2, t3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 t0, b0;\n\tcvt.rn.f16x2.e2m1x2 t1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 t2, b2;\n\tcvt.rn.f16x2.e2m1x2 t3, b3;\n\t"
        "mul.rn.f16x2 %0, t0, %5;\n\tmul.rn.f16x2 %1, t1, %5;\n\t"
        "mul.rn.f16x2 %2, t2, %5;\n\tmul.rn.f16x2 %3, t3, %5;\n\t}"
        : "=r"(out[0]), "=r"(out[1]), "=r"(out[2]), "=r"(out[3])
        : "r"(word), "r"(scale_h2));
}

// max(|a|, |b|) per f16 half with the sign bit the XOR of the inputs' signs
// (finite inputs); clear the sign bits to read a magnitude.
__device__ __forceinline__ uint32_t h2_absmax_xs(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("max.xorsign.abs.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Word i (0..3) of a 16-byte vector (i a compile-time constant after unrolling).
__device__ __forceinline__ uint32_t u4_word(const uint4 &v, int i)
{
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// The low / high f16 of an f16x2 word as binary32 (exact).
__device__ __forceinline__ float h2_lo_to_f32(uint32_t h2)
{
    float f;
    asm("{\n\t.reg .f16 a, b;\n\tmov.b32 {a, b}, %1;\n\tcvt.f32.f16 %0, a;\n\t}" : "=f"(f) : "r"(h2));
    return f;
}

__device__ __forceinline__ float h2_hi_to_f32(uint32_t h2)
{
    float f;
    asm("{\n\t.reg .f16 a, b;\n\tmov.b32 {a, b}, %1;\n\tcvt.f32.f16 %0, b;\n\t}" : "=f"(f) : "r"(h2));
    return f;
}

// E4M3 byte -> the same value twice as f16x2 (exact: E4M3 is a subset of f16).
__device__ __forceinline__ uint32_t e4m3_to_h2(uint32_t b)
{
    uint32_t h2;
    const uint16_t b16 = (uint16_t)(((b & 0xFFu) << 8) | (b & 0xFFu));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(b16));
    return h2;
}

// E4M3 (bias 7, subnormal m * 2^-9); NaN (S.1111.111) never reaches here.
__device__ __forceinline__ float e4m3_to_f32(uint32_t b)
{
    uint32_t e = (b >> 3) & 15u, m = b & 7u;
    float v = (e == 0u) ? (float)m * 0.001953125f : __uint_as_float(((e + 120u) << 23) | (m << 20));
    return (b & 0x80u) ? -v : v;
}

// 2^(b - 127) for an E8M0 byte b in [0, 254].
__device__ __forceinline__ float e8m0_to_f32(uint32_t b)
{
    return b == 0u ? __uint_as_float(0x00400000u) : __uint_as_float(b << 23);
}

// ---------------------------------------------------------------- hardware RN
// Two binary32 values -> two E2M1 codes, round to nearest even, saturating;
// `lo` lands in bits 3:0, `hi` in bits 7:4.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi)
{
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %2, %1;\n\tcvt.u32.u8 %0, t;\n\t}"
        : "=r"(r) : "f"(lo), "f"(hi));
    return r;
}

// One binary32 value -> E4M3 byte, round to nearest even, saturating at 448.
__device__ __forceinline__ uint32_t cvt_e4m3(float v)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %2, %1;" : "=h"(r) : "f"(v), "f"(0.0f));
    return (uint32_t)r & 0xFFu;
}

// ---------------------------------------------------------------- E8M0 exponents
// Smallest integer e with a <= 448 * 2^e (448 = 1.75 * 2^8), clamped to
// [-127, 127]; -127 for a == 0.  a is a finite non-negative binary32.
__device__ __forceinline__ int mx_exponent_448(float a)
{
    uint32_t bits = __float_as_uint(a);
    uint32_t E = bits >> 23, m = bits & 0x7FFFFFu;
    if (E == 0u) return -127;  // zero or subnormal: 2^-126 <= 448 * 2^-127
    int e = (m <= 0x600000u) ? (int)E - 135 : (int)E - 134;
    return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// Smallest integer e with a <= (127/64) * 2^e (127/64 = 1.984375), clamped.
__device__ __forceinline__ int mx_exponent_s2f6(float a)
{
    uint32_t bits = __float_as_uint(a);
    uint32_t E = bits >> 23, m = bits & 0x7FFFFFu;
    if (E == 0u) return (m <= 0x7F0000u) ? -127 : -126;
    int e = (m <= 0x7E0000u) ? (int)E - 127 : (int)E - 126;
    return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// ---------------------------------------------------------------- E4M3 from y = d * 2^-e
// 2^-e as binary32 for the MX exponents that finite inputs produce (e <= 120).
__device__ __forceinline__ float exp2_neg(int e) { return __uint_as_float((uint32_t)(127 - e) << 23); }

// Two binary32 values -> two E4M3 bytes (lo in byte 0), nearest even, saturating.
__device__ __forceinline__ uint32_t cvt_e4m3x2_rn(float lo, float hi)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %2, %1;" : "=h"(r) : "f"(lo), "f"(hi));
    return (uint32_t)r;
}

// Four binary32 values -> four E4M3 bytes (element k in byte k) by the
// hardware's stochastic rounding: each element adds a 16-bit random value to
// the leading 16 bits of its discarded fraction and rounds away from zero on
// carry.  Elements 0 / 1 take rbits[15:0] / the same bits reversed, elements
// 2 / 3 take rbits[31:16] / reversed.  The sign is kept.
__device__ __forceinline__ uint32_t cvt_e4m3x4_rs(float e0, float e1, float e2, float e3, uint32_t rbits)
{
    uint32_t r;
    asm("cvt.rs.satfinite.e4m3x4.f32 %0, {%1, %2, %3, %4}, %5;"
        : "=r"(r)
        : "f"(e3), "f"(e2), "f"(e1), "f"(e0), "r"(rbits));
    return r;
}

// ---------------------------------------------------------------- Philox4x32-10
// Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3",
// SC'11: ten rounds of two 32x32->64 multiplies (multipliers 0xD2511F53,
// 0xCD9E8D57) with the key added by xor and bumped by the Weyl constants
// (0x9E3779B9, 0xBB67AE85) between rounds.
// One Philox round: the 32 x 32 -> 64-bit products as separate high and low
// 32-bit multiplies (measured 6 % faster in the requantisation kernels than
// one 64-bit product; the same bits).
__device__ __forceinline__ uint4 philox_round(uint4 c, uint32_t k0, uint32_t k1)
{
    const uint32_t h0 = __umulhi(0xD2511F53u, c.x), l0 = 0xD2511F53u * c.x;
    const uint32_t h1 = __umulhi(0xCD9E8D57u, c.z), l1 = 0xCD9E8D57u * c.z;
    return make_uint4(h1 ^ c.y ^ k0, l1, h0 ^ c.w ^ k1, l0);
}

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1)
{
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        c = philox_round(c, k0, k1);
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return c;
}

// The 4 random words for output elements 16j .. 16j+15 of a tensor (tag
// selects the tensor): counter (j lo, j hi, tag, 0), key (seed lo, seed hi);
// word k serves elements 16j + 4k .. 16j + 4k + 3.
__device__ __forceinline__ uint4 sr_words16(uint64_t seed, uint32_t tag, uint64_t j)
{
    return philox4x32_10(make_uint4((uint32_t)j, (uint32_t)(j >> 32), tag, 0u), (uint32_t)seed,
                         (uint32_t)(seed >> 32));
}

// ---------------------------------------------------------------- RHT + S2F6
// In-register 32-point randomised Hadamard transform and S2F6 block
// quantisation [NVLink]: v = sigma . x; butterflies (a, b) -> (a + b, a - b)
// for strides 1, 2, 4, 8, 16; z = v * RN(1/sqrt(32)); e = smallest exponent
// with amax <= (127/64) 2^e; k = rint(z * 2^(6 - e)).  The block functions
// return the E8M0 byte and write 32 int8 codes packed little-endian into q[8].

// Packed binary32 product (each lane rounded to nearest even).  Used only
// where the product feeds a conversion: measured on sm_103a, a packed multiply
// whose result feeds a packed add is contracted into a fused multiply-add
// despite the .rn modifiers, so sums of products stay on the scalar
// intrinsics, which are never contracted.
__device__ __forceinline__ void mul2(float a0, float a1, float b0, float b1, float &c0, float &c1)
{
    asm("{\n\t.reg .b64 a, b, c;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
        "mul.rn.f32x2 c, a, b;\n\tmov.b64 {%0, %1}, c;\n\t}"
        : "=f"(c0), "=f"(c1) : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// (a, b) -> (a + b, a - b) on two lanes at once (each lane rounded to nearest
// even, exactly the scalar __fadd_rn / __fsub_rn).  Only for sums whose inputs
// are themselves sums, so no product can be contracted into them.
__device__ __forceinline__ void add_sub2(float &a0, float &a1, float &b0, float &b1)
{
    asm("{\n\t.reg .b64 a, b, s, d;\n\tmov.b64 a, {%0, %1};\n\tmov.b64 b, {%2, %3};\n\t"
        "add.rn.f32x2 s, a, b;\n\tsub.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, s;\n\tmov.b64 {%2, %3}, d;\n\t}"
        : "+f"(a0), "+f"(a1), "+f"(b0), "+f"(b1));
}

// RN(a * s + c) on two lanes.
__device__ __forceinline__ void fma2(float a0, float a1, float s, float c, float &r0, float &r1)
{
    asm("{\n\t.reg .b64 a, b, c, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %4};\n\tmov.b64 c, {%5, %5};\n\t"
        "fma.rn.f32x2 d, a, b, c;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(r0), "=f"(r1)
        : "f"(a0), "f"(a1), "f"(s), "f"(c));
}

// The RHT-32 + S2F6 of a block whose signs sigma have already been applied:
// butterflies, z = v * RN(1/sqrt(32)), e from max |z|, k = RNE(z * 2^(6-e)).
// The exponent is chosen so that |z| * 2^(6-e) <= 127; the product by the
// power of two is exact (or far below 1/2, where it is rounded once), so
// RN(z * 2^(6-e) + 1.5 * 2^23) holds rint(z * 2^(6-e)) in its low mantissa
// bits: its low byte is k's two's-complement byte.  A block at the clamped
// exponent 127 (an amax of 2^127 or more, or not finite) takes the general
// ldexp / convert / clamp path instead.
__device__ __forceinline__ uint32_t rht32_s2f6_signed(float (&v)[32], uint32_t (&q)[8])
{
#pragma unroll
    for (int i = 0; i < 32; i += 2) {  // stride 1: inputs may be products, scalar sums
        const float a = v[i], b = v[i + 1];
        v[i] = __fadd_rn(a, b);
        v[i + 1] = __fsub_rn(a, b);
    }
#pragma unroll
    for (int h = 2; h < 32; h <<= 1) {
#pragma unroll
        for (int i = 0; i < 32; i += 2)
            if ((i & h) == 0) add_sub2(v[i], v[i + 1], v[i + h], v[i + h + 1]);
    }
    const float rs = __uint_as_float(0x3E3504F3u);  // RN(1/sqrt(32))
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        v[j] = __fmul_rn(v[j], rs);
        amax = fmaxf(amax, fabsf(v[j]));
    }
    const int e = mx_exponent_s2f6(amax);
    if (e < 127) {
        int n = 6 - e;  // -120 .. 133
        if (n > 127) {  // 2^n is not a binary32 value: scale by 2^64 first (exact: |v| < 2^-120)
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __fmul_rn(v[j], 18446744073709551616.0f);
            n -= 64;
        }
        const float sc = __uint_as_float((uint32_t)(n + 127) << 23), magic = 12582912.0f;  // 2^n, 1.5 * 2^23
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            float t[4];
            fma2(v[4 * w], v[4 * w + 1], sc, magic, t[0], t[1]);
            fma2(v[4 * w + 2], v[4 * w + 3], sc, magic, t[2], t[3]);
            q[w] = __byte_perm(__byte_perm(__float_as_uint(t[0]), __float_as_uint(t[1]), 0x0040u),
                               __byte_perm(__float_as_uint(t[2]), __float_as_uint(t[3]), 0x0040u), 0x5410u);
        }
    } else {
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            uint32_t packed = 0u;
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                int k = __float2int_rn(ldexpf(v[4 * w + t], 6 - e));
                k = k > 127 ? 127 : (k < -128 ? -128 : k);
                packed |= ((uint32_t)k & 0xFFu) << (8 * t);
            }
            q[w] = packed;
        }
    }
    return (uint32_t)(e + 127);
}

// In-register 32-point randomised Hadamard transform and S2F6 block
// quantisation [NVLink] of x: v = sigma . x, then rht32_s2f6_signed.
__device__ __forceinline__ uint32_t rht32_s2f6(float (&v)[32], uint32_t sigma, uint32_t (&q)[8])
{
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(__float_as_uint(v[j]) ^ (((sigma >> j) & 1u) << 31));
    return rht32_s2f6_signed(v, q);
}

__device__ __forceinline__ uint32_t rht_sigma(uint64_t seed)
{
    return philox4x32_10(make_uint4(0u, 0u, 5u, 0u), (uint32_t)seed, (uint32_t)(seed >> 32)).x;
}

}  // namespace pmn
