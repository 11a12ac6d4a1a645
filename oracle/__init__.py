"""CPU oracle for block-scaled MoE expert-layer numerics.

TEST INFRASTRUCTURE ONLY.  The slow, plain definition of what the CUDA library
computes.  Only tests/, the smoke check and the benchmark's CPU-baseline leg
may import this package; the product path must never route through it.  It
shares no code with the CUDA path.

Element-wise and block-wise steps (codecs, quantisers, stochastic rounding,
Philox, RHT + S2F6) live in pmn_oracle.c and are reached through ctypes.  The
GEMMs are written here: a binary64 matrix product over the dequantised
operands (a library matmul serves as the step), then the outer scales.

Sections of the pages cited below (page "Thinking Machines ... Inkling 2 Small",
arex-research.com): [Bits] fewer bits / faster arithmetic, [Layers] expert
forward in 4-bit, [SR] transpose regrouping and stochastic rounding, [NVLink]
dispatch and combine, [Cost] the recipe's costs (4/6, outer scales).

Parity status: pinned -- see tests/test_oracle_*.py.
"""
import ctypes
import os

import numpy as np

from .build import build_oracle

_lib = None

OUTER_PER_ROW = 0
OUTER_PER_GROUP = 1
OUTER_GIVEN = 2

TAG_X, TAG_H, TAG_W1, TAG_W2, TAG_RHT = 1, 2, 3, 4, 5


def lib():
    global _lib
    if _lib is None:
        path = build_oracle()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i64, u64, u32, i32 = ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int
        L.orc_philox4x32_10.argtypes = [P, P, P]
        L.orc_set_num_threads.argtypes = [i32]
        L.orc_set_num_threads.restype = None
        L.orc_max_threads.restype = i32
        L.orc_sr_bits16.argtypes = [u64, u32, u64]
        L.orc_sr_bits16.restype = u32
        for n in ("orc_e2m1_value", "orc_e4m3_value", "orc_e8m0_value"):
            getattr(L, n).argtypes = [u32]
            getattr(L, n).restype = ctypes.c_double
        L.orc_s2f6_value.argtypes = [ctypes.c_int32]
        L.orc_s2f6_value.restype = ctypes.c_double
        L.orc_e2m1_rne.argtypes = [ctypes.c_float]
        L.orc_e2m1_rne.restype = u32
        L.orc_e4m3_rne.argtypes = [ctypes.c_float]
        L.orc_e4m3_rne.restype = u32
        L.orc_e4m3_sr.argtypes = [ctypes.c_double, u32]
        L.orc_e4m3_sr.restype = u32
        L.orc_e2m1_sr.argtypes = [ctypes.c_double, u32]
        L.orc_e2m1_sr.restype = u32
        L.orc_bf16_rne.argtypes = [ctypes.c_double]
        L.orc_bf16_rne.restype = u32
        L.orc_nvfp4_quantize_block.argtypes = [P, ctypes.c_float, i32, P, P]
        L.orc_nvfp4_quantize_block.restype = i32
        L.orc_nvfp4_quantize.argtypes = [P, i64, i64, i64, i32, P, i64, i32, P, P, P, P]
        L.orc_nvfp4_dequant_f32.argtypes = [P, P, P, i64, i64, i64, P]
        L.orc_nvfp4_dequant_f64.argtypes = [P, P, i64, i64, P]
        L.orc_e8m0_exponent.argtypes = [ctypes.c_double, ctypes.c_double]
        L.orc_e8m0_exponent.restype = i32
        L.orc_requant_transpose_mxfp8.argtypes = [P, P, P, i32, i64, i64, i64, u64, u32, i32, P, P]
        L.orc_requant_transpose_mxfp8_window.argtypes = [P, P, P, i32, i64, i64, i64, u64, u32, i32, P, P,
                                                         i64, i64, i64]
        L.orc_mxfp8_quantize.argtypes = [P, i64, i64, i32, P, P]
        L.orc_requant_transpose_nvfp4.argtypes = [P, P, P, i32, i64, i64, i64, u64, u32, i32, P, P, P, i64]
        L.orc_mxfp8_dequant_f64.argtypes = [P, P, i64, i64, P]
        L.orc_rht_sign_word.argtypes = [u64]
        L.orc_rht_sign_word.restype = u32
        L.orc_rsqrt32.restype = ctypes.c_float
        L.orc_rht32.argtypes = [P, u32, P]
        L.orc_rht_s2f6.argtypes = [P, i64, i64, u64, P, P]
        L.orc_s2f6_dequant_inverse_rht.argtypes = [P, P, i64, i64, u64, P]
        L.orc_combine_receive.argtypes = [P, P, i64, i64, u64, P, P, i64, i64, P]
        L.orc_bf16_rne_array.argtypes = [P, i64, P]
        _lib = L
    return _lib


def _p(a):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else None


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- primitives
def philox4x32_10(ctr, key):
    """Philox4x32-10 (Salmon et al., SC'11) of one counter block."""
    c = _c(ctr, np.uint32)
    k = _c(key, np.uint32)
    out = np.zeros(4, np.uint32)
    lib().orc_philox4x32_10(_p(c), _p(k), _p(out))
    return out


def sr_bits16(seed, tag, i):
    return lib().orc_sr_bits16(seed, tag, i)


def e2m1_value(code):
    return lib().orc_e2m1_value(code)


def e4m3_value(b):
    return lib().orc_e4m3_value(b)


def e8m0_value(b):
    return lib().orc_e8m0_value(b)


def s2f6_value(k):
    return lib().orc_s2f6_value(k)


def e2m1_rne(v):
    return lib().orc_e2m1_rne(float(np.float32(v)))


def e4m3_rne(v):
    return lib().orc_e4m3_rne(float(np.float32(v)))


def e4m3_sr(y, rb16):
    return lib().orc_e4m3_sr(float(y), rb16)


def e2m1_sr(y, rb16):
    return lib().orc_e2m1_sr(float(y), rb16)


def bf16_rne(v):
    return lib().orc_bf16_rne(float(v))


def set_num_threads(n):
    """Threads of the oracle's OpenMP loops (timing only; results do not depend on it)."""
    lib().orc_set_num_threads(int(n))


def max_threads():
    return int(lib().orc_max_threads())


def e8m0_exponent(amax, top=448.0):
    return lib().orc_e8m0_exponent(float(amax), float(top))


def rsqrt32():
    return np.float32(lib().orc_rsqrt32())


def rht_sign_word(seed):
    return lib().orc_rht_sign_word(seed)


def rht32(x, sigma):
    x = _c(x, np.float32)
    z = np.zeros(32, np.float32)
    lib().orc_rht32(_p(x), sigma, _p(z))
    return z


# ---------------------------------------------------------------- NVFP4 [SR], [Cost]
def nvfp4_quantize_block(x16, g, four_over_six=False):
    """One 16-value block with outer scale g: (codes[16], scale byte, chosen m)."""
    x = _c(x16, np.float32)
    codes = np.zeros(16, np.uint8)
    sb = np.zeros(1, np.uint8)
    m = lib().orc_nvfp4_quantize_block(_p(x), float(np.float32(g)), int(four_over_six), _p(codes), _p(sb))
    return codes, int(sb[0]), m


def nvfp4_quantize(x_bf16_bits, outer_mode=OUTER_PER_ROW, group_offsets=None, four_over_six=False,
                   outer=None, want_choice=False):
    """bf16 bits [rows, cols] -> (codes [rows, cols/2] u8, scales [rows, cols/16] u8, outer f32).

    outer_mode OUTER_PER_ROW: g per row (tokens); OUTER_PER_GROUP: g per row range
    group_offsets[k]..group_offsets[k+1] (experts, or one range for a tensor);
    OUTER_GIVEN: `outer` holds g per row.
    """
    x = _c(x_bf16_bits, np.uint16)
    rows, cols = x.shape
    assert cols % 16 == 0
    codes = np.zeros((rows, cols // 2), np.uint8)
    scales = np.zeros((rows, cols // 16), np.uint8)
    offs = None
    ng = 0
    if outer_mode == OUTER_PER_GROUP:
        offs = _c(group_offsets, np.int64)
        ng = len(offs) - 1
        out_outer = np.zeros(ng, np.float32)
    elif outer_mode == OUTER_GIVEN:
        out_outer = _c(outer, np.float32).copy()
        assert out_outer.shape == (rows,)
    else:
        out_outer = np.zeros(rows, np.float32)
    choice = np.zeros((rows, cols // 16), np.uint8) if want_choice else None
    lib().orc_nvfp4_quantize(_p(x), rows, cols, cols, outer_mode, _p(offs), ng, int(four_over_six),
                             _p(codes), _p(scales), _p(out_outer), _p(choice))
    if want_choice:
        return codes, scales, out_outer, choice
    return codes, scales, out_outer


def nvfp4_dequant_f32(codes, scales, outer, rows_per_outer=1):
    """Canonical binary32 dequantisation (dec(c) * dec(S)) * g."""
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    rows = codes.shape[0]
    cols = codes.shape[1] * 2
    out = np.zeros((rows, cols), np.float32)
    o = _c(outer, np.float32) if outer is not None else None
    lib().orc_nvfp4_dequant_f32(_p(codes), _p(scales), _p(o), rows_per_outer, rows, cols, _p(out))
    return out


def nvfp4_dequant_f64(codes, scales):
    """dec(c) * dec(S) in binary64 (no outer scale)."""
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    rows = codes.shape[0]
    cols = codes.shape[1] * 2
    out = np.zeros((rows, cols), np.float64)
    lib().orc_nvfp4_dequant_f64(_p(codes), _p(scales), rows, cols, _p(out))
    return out


# ---------------------------------------------------------------- MXFP8 [SR]
def requant_transpose_mxfp8(codes, scales, outer, outer_per_row, batch, rows, cols, seed, tag,
                            stochastic=True, b_begin=0, rows_total=None, r_begin=0):
    """NVFP4 [batch, rows, cols] -> dequant -> transpose -> MXFP8 [batch, cols, rows].

    With b_begin / rows_total / r_begin the inputs are a window of a larger
    tensor and the random bits follow the element's index in the full output."""
    codes = _c(codes, np.uint8).reshape(batch * rows, cols // 2)
    scales = _c(scales, np.uint8).reshape(batch * rows, cols // 16)
    outer = _c(outer, np.float32)
    assert rows % 32 == 0 and r_begin % 32 == 0
    out = np.zeros((batch, cols, rows), np.uint8)
    out_sc = np.zeros((batch, cols, rows // 32), np.uint8)
    lib().orc_requant_transpose_mxfp8_window(_p(codes), _p(scales), _p(outer), 0 if outer_per_row else 1,
                                             batch, rows, cols, seed, tag, 0 if stochastic else 1,
                                             _p(out), _p(out_sc), b_begin, rows if rows_total is None else rows_total,
                                             r_begin)
    return out, out_sc


def requant_transpose_nvfp4(codes, scales, outer, outer_per_row, batch, rows, cols, seed, tag,
                            stochastic=True, b_begin=0):
    """NVFP4 [batch, rows, cols] -> dequant -> transpose -> NVFP4 [batch, cols,
    rows] with stochastic (or nearest) rounding: (codes [batch, cols, rows/2],
    E4M3 scales [batch, cols, rows/16], outer [batch]).  b_begin: index of
    the first entry in the full tensor (random bits follow the full index)."""
    codes = _c(codes, np.uint8).reshape(batch * rows, cols // 2)
    scales = _c(scales, np.uint8).reshape(batch * rows, cols // 16)
    outer = _c(outer, np.float32)
    assert rows % 16 == 0 and cols % 16 == 0
    out = np.zeros((batch, cols, rows // 2), np.uint8)
    out_sc = np.zeros((batch, cols, rows // 16), np.uint8)
    out_g = np.zeros(batch, np.float32)
    lib().orc_requant_transpose_nvfp4(_p(codes), _p(scales), _p(outer), 0 if outer_per_row else 1, batch, rows,
                                      cols, seed, tag, 0 if stochastic else 1, _p(out), _p(out_sc), _p(out_g),
                                      b_begin)
    return out, out_sc, out_g


def mxfp8_quantize(x_bf16_bits, transpose=False):
    """bf16 -> MXFP8 with round to nearest even (gradients)."""
    x = _c(x_bf16_bits, np.uint16)
    rows, cols = x.shape
    if transpose:
        assert rows % 32 == 0
        out = np.zeros((cols, rows), np.uint8)
        sc = np.zeros((cols, rows // 32), np.uint8)
    else:
        assert cols % 32 == 0
        out = np.zeros((rows, cols), np.uint8)
        sc = np.zeros((rows, cols // 32), np.uint8)
    lib().orc_mxfp8_quantize(_p(x), rows, cols, int(transpose), _p(out), _p(sc))
    return out, sc


def mxfp8_dequant_f64(q, sc):
    q = _c(q, np.uint8)
    sc = _c(sc, np.uint8)
    rows, cols = q.shape
    out = np.zeros((rows, cols), np.float64)
    lib().orc_mxfp8_dequant_f64(_p(q), _p(sc), rows, cols, _p(out))
    return out


# ---------------------------------------------------------------- RHT + S2F6 [NVLink]
def rht_s2f6(x_f32, seed):
    x = _c(x_f32, np.float32)
    rows, cols = x.shape
    assert cols % 32 == 0
    out = np.zeros((rows, cols), np.int8)
    sc = np.zeros((rows, cols // 32), np.uint8)
    lib().orc_rht_s2f6(_p(x), rows, cols, seed, _p(out), _p(sc))
    return out, sc


def s2f6_dequant_inverse_rht(q, sc, seed):
    q = _c(q, np.int8)
    sc = _c(sc, np.uint8)
    rows, cols = q.shape
    out = np.zeros((rows, cols), np.float64)
    lib().orc_s2f6_dequant_inverse_rht(_p(q), _p(sc), rows, cols, seed, _p(out))
    return out


def combine_receive(q, sc, seed, row_index, gates):
    """Receive side of the combine [NVLink]: out[t] = sum_i gates[t, i] *
    (routed row row_index[t, i] decoded and transformed back), binary64
    [tokens, cols]; a negative index adds nothing."""
    q = _c(q, np.int8)
    sc = _c(sc, np.uint8)
    idx = _c(row_index, np.int64)
    g = _c(gates, np.float32)
    rows, cols = q.shape
    tokens, k = idx.shape
    assert g.shape == (tokens, k) and cols % 32 == 0 and sc.shape == (rows, cols // 32)
    assert np.all(idx < rows)
    out = np.zeros((tokens, cols), np.float64)
    lib().orc_combine_receive(_p(q), _p(sc), rows, cols, seed, _p(idx), _p(g), tokens, k, _p(out))
    return out


# ---------------------------------------------------------------- GEMMs [Layers], [SR]
def grouped_gemm_nvfp4(a_codes, a_scales, a_outer, b_codes, b_scales, b_outer, offsets, rows=None):
    """Z[m, n] = (sum_k A[m, k] * B_e[n, k]) * gA[m] * gB[e] in binary64 for the
    rows m of expert e = offsets[e]..offsets[e+1]; A and B are dequantised
    exactly (code * E4M3 scale).  `rows` may restrict the output to a subset of
    row indices (sampled parity at full size).

    b_codes: [E, N, K/2], b_scales: [E, N, K/16], b_outer: [E]."""
    offsets = np.asarray(offsets, np.int64)
    E = len(offsets) - 1
    N = b_codes.shape[1]
    sel = np.arange(offsets[-1]) if rows is None else np.asarray(rows, np.int64)
    out = np.zeros((len(sel), N), np.float64)
    expert_of = np.searchsorted(offsets, sel, side="right") - 1
    for e in np.unique(expert_of):
        idx = np.nonzero(expert_of == e)[0]
        A = nvfp4_dequant_f64(a_codes[sel[idx]], a_scales[sel[idx]])
        B = nvfp4_dequant_f64(b_codes[e], b_scales[e])
        out[idx] = (A @ B.T) * np.asarray(a_outer, np.float64)[sel[idx], None] * float(b_outer[e])
    return out


def gemm_nvfp4(a_codes, a_scales, a_outer, b_codes, b_scales, b_outer):
    """Single GEMM: A [M, K] (outer per row), B [N, K] (one outer)."""
    M = a_codes.shape[0]
    return grouped_gemm_nvfp4(a_codes, a_scales, a_outer, b_codes[None], b_scales[None],
                              np.asarray([b_outer], np.float32), [0, M])


def gemm_mxfp8_mgrouped(a, a_sc, b, b_sc, offsets, rows=None):
    """C[m, n] = sum_k A[m, k] B_e[n, k], rows m of group e; A [M, K], B [E, N, K]."""
    offsets = np.asarray(offsets, np.int64)
    N = b.shape[1]
    sel = np.arange(offsets[-1]) if rows is None else np.asarray(rows, np.int64)
    out = np.zeros((len(sel), N), np.float64)
    expert_of = np.searchsorted(offsets, sel, side="right") - 1
    for e in np.unique(expert_of):
        idx = np.nonzero(expert_of == e)[0]
        A = mxfp8_dequant_f64(a[sel[idx]], a_sc[sel[idx]])
        B = mxfp8_dequant_f64(b[e], b_sc[e])
        out[idx] = A @ B.T
    return out


def gemm_mxfp8_kgrouped(a, a_sc, b, b_sc, offsets, groups=None):
    """C_e[m, n] = sum_{k in segment e} A[m, k] B[n, k]; A [M, Ktot], B [N, Ktot]
    with 32-blocks along K (segments are multiples of 32)."""
    offsets = np.asarray(offsets, np.int64)
    E = len(offsets) - 1
    groups = range(E) if groups is None else groups
    M, N = a.shape[0], b.shape[0]
    out = {}
    for e in groups:
        k0, k1 = int(offsets[e]), int(offsets[e + 1])
        if k1 == k0:
            out[e] = np.zeros((M, N))
            continue
        A = mxfp8_dequant_f64(a[:, k0:k1], a_sc[:, k0 // 32:k1 // 32])
        B = mxfp8_dequant_f64(b[:, k0:k1], b_sc[:, k0 // 32:k1 // 32])
        out[e] = A @ B.T
    return out


def swiglu_bf16(y_bf16_bits, f):
    """h = silu(gate) * up in binary64, rounded once to bfloat16.

    Reading (not on the pages; the w1 shape [2F, D] fixes that the layer is
    gated): gate = columns [0, F), up = columns [F, 2F)."""
    y = _c(y_bf16_bits, np.uint16)
    yf = (y.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    a = yf[:, :f]
    b = yf[:, f:2 * f]
    h = a * b / (1.0 + np.exp(-a))
    return bf16_rne_array(h)


def swiglu_bf16_from_f64(y, f):
    """h = silu(gate) * up from binary64 gate | up values [rows, 2F] (a GEMM's
    exact result, not rounded to bf16 first), rounded once to bfloat16.
    Reading, for an epilogue that forms h from the GEMM's accumulator: the
    unfused path rounds Y to bf16 before the SwiGLU, the fused one does not."""
    yf = _c(y, np.float64)
    a = yf[:, :f]
    b = yf[:, f:2 * f]
    return bf16_rne_array(a * b / (1.0 + np.exp(-a)))


def bf16_rne_array(v):
    """Round binary64 values to bfloat16 bits (nearest even), element by element."""
    v = _c(v, np.float64)
    out = np.empty(v.shape, np.uint16)
    lib().orc_bf16_rne_array(_p(v), v.size, _p(out))
    return out
