"""Thin Python binding of the C ABI declared in include/pmn.h.

Each function here has the name of its C entry point without the `pmn_`
prefix and does argument marshalling only: it allocates outputs with torch
(device memory), passes raw device pointers and the current CUDA stream to
libpmn.so, and raises on a non-zero status.  Every step of the computation
runs in the library's CUDA kernels; there is no fallback path -- if the
library is missing or fails to load, every call raises.
"""
import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpmn.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT = 0, 1, 2, 3, 4
IN_BF16, IN_BF16_SWIGLU = 0, 1
OUTER_PER_ROW, OUTER_PER_GROUP = 0, 1
ROUND_SR, ROUND_RN = 0, 1
OUT_BF16, OUT_F32, OUT_RHT_S2F6, OUT_SWIGLU_BF16 = 0, 1, 2, 3
GROUP_M, GROUP_K = 0, 1
DEVERR_WAIT_TIMEOUT = 1
DEVERR_BAD_OFFSETS = 2

# Stochastic-rounding stream tags of the expert layer's saved tensors.
TAG_X, TAG_H, TAG_W1, TAG_W2 = 1, 2, 3, 4

_P, _I64, _U64, _U32, _I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int

SIGNATURES = {
    "pmn_version": ([], _I),
    "pmn_status_string": ([_I], ctypes.c_char_p),
    "pmn_get_device_error": ([_P, _P], _I),
    "pmn_set_wait_limit_ns": ([_U64], _U64),
    "pmn_wait_selftest": ([_U64, _P], _I),
    "pmn_nvfp4_quantize": ([_P, _I64, _I64, _I64, _I, _I, _I64, _I, _P, _P, _P, _P, _P, _I64, _P], _I),
    "pmn_nvfp4_quantize_workspace_bytes": ([_I, _I64, _I64], _I64),
    "pmn_nvfp4_quantize_per_group_noalloc": ([_P, _I64, _I64, _I64, _I, _P, _P, _P, _P], _I),
    "pmn_requant_transpose_sr_mxfp8": ([_P, _P, _P, _I, _I64, _I64, _I64, _U64, _U32, _I, _P, _P, _P], _I),
    "pmn_mxfp8_quantize_both": ([_P, _I64, _I64, _P, _P, _P, _P, _P], _I),
    "pmn_requant_transpose_sr_nvfp4": ([_P, _P, _P, _I, _I64, _I64, _I64, _U64, _U32, _I, _P, _P, _P, _P], _I),
    "pmn_mxfp8_quantize": ([_P, _I64, _I64, _I, _P, _P, _P], _I),
    "pmn_mxfp8_quantize_swiglu": ([_P, _I64, _I64, _P, _P, _P, _P], _I),
    "pmn_grouped_gemm_nvfp4": ([_P, _P, _P, _P, _P, _P, _P, _I, _I64, _I64, _I64, _I, _P, _P], _I),
    "pmn_w1_gemm_swiglu_nvfp4": ([_P, _P, _P, _P, _P, _P, _P, _I, _I64, _I64, _I64, _I, _P, _P, _P, _P, _P], _I),
    "pmn_w2_gemm_rht_s2f6": ([_P, _P, _P, _P, _P, _P, _P, _I, _I64, _I64, _I64, _U64, _P, _P, _P, _P], _I),
    "pmn_rht_s2f6_quantize": ([_P, _I64, _I64, _U64, _P, _P, _P], _I),
    "pmn_combine_receive_s2f6": ([_P, _P, _I64, _I64, _U64, _P, _P, _I64, _I, _I, _P, _P], _I),
    "pmn_gemm_mxfp8": ([_P, _P, _P, _P, _P, _I, _I, _I64, _I64, _I64, _I, _P, _P], _I),
}

_lib = None


class PmnError(RuntimeError):
    pass


def lib():
    """The loaded libpmn.so (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise PmnError("libpmn.so not built: run precision_moe_numerics_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in SIGNATURES.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def _check(st, what):
    if st != OK:
        msg = lib().pmn_status_string(st).decode()
        raise PmnError("%s failed: %s (%d)" % (what, msg, st))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dev(t, dtype=None):
    if not t.is_cuda:
        raise PmnError("tensor must live on the GPU")
    if not t.is_contiguous():
        raise PmnError("tensor must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise PmnError("expected %s, got %s" % (dtype, t.dtype))
    return t


def version():
    return lib().pmn_version()


def get_device_error(stream=None):
    err = ctypes.c_int32(0)
    _check(lib().pmn_get_device_error(_stream(stream), ctypes.byref(err)), "get_device_error")
    return err.value


def set_wait_limit_ns(ns):
    """Sets the limit of the library's bounded device waits; returns the previous one."""
    return lib().pmn_set_wait_limit_ns(int(ns))


def wait_selftest(limit_ns, stream=None):
    _check(lib().pmn_wait_selftest(int(limit_ns), _stream(stream)), "wait_selftest")


def nvfp4_quantize_workspace_bytes(outer_mode, rows, rows_per_group=0):
    n = lib().pmn_nvfp4_quantize_workspace_bytes(outer_mode, rows, rows_per_group)
    if n < 0:
        raise PmnError("nvfp4_quantize_workspace_bytes: invalid arguments")
    return n


# ------------------------------------------------------------------ quantisation
def nvfp4_quantize(x, cols=None, four_over_six=False, outer_mode=OUTER_PER_ROW, rows_per_group=None,
                   swiglu=False, want_h=False, out=None, workspace=None, stream=None):
    """bf16 [rows, ldx] -> (codes u8 [rows, cols/2], scales u8 [rows, cols/16], outer f32[, h bf16]).

    swiglu: x holds gate | up halves of width `cols`; h = silu(gate) * up is quantised.
    workspace: the per-group kernel's scratch (uint8 device tensor of at least
    nvfp4_quantize_workspace_bytes(...) bytes); allocated here when None."""
    _dev(x, torch.bfloat16)
    rows, ldx = x.shape
    if cols is None:
        cols = ldx // 2 if swiglu else ldx
    dev = x.device
    if out is None:
        codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device=dev)
        scales = torch.empty((rows, cols // 16), dtype=torch.uint8, device=dev)
        n_outer = rows if outer_mode == OUTER_PER_ROW else rows // rows_per_group
        outer = torch.empty((n_outer,), dtype=torch.float32, device=dev)
    else:
        codes, scales, outer = out
    h = torch.empty((rows, cols), dtype=torch.bfloat16, device=dev) if want_h else None
    if workspace is None and outer_mode == OUTER_PER_GROUP:
        workspace = torch.empty((max(1, nvfp4_quantize_workspace_bytes(outer_mode, rows, rows_per_group or 0)),),
                                dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().pmn_nvfp4_quantize(_ptr(x), rows, cols, ldx, IN_BF16_SWIGLU if swiglu else IN_BF16, outer_mode,
                                  rows_per_group or 0, int(four_over_six), _ptr(codes), _ptr(scales), _ptr(outer),
                                  _ptr(h), _ptr(workspace), ws_bytes, _stream(stream))
    _check(st, "nvfp4_quantize")
    return (codes, scales, outer, h) if want_h else (codes, scales, outer)


def nvfp4_quantize_per_group_noalloc(x, rows_per_group, four_over_six=False, out=None, stream=None):
    """As nvfp4_quantize(x, outer_mode=OUTER_PER_GROUP, ...), through the entry point whose scratch is a
    fixed device array (no allocation inside the call)."""
    _dev(x, torch.bfloat16)
    rows, cols = x.shape
    dev = x.device
    if out is None:
        codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device=dev)
        scales = torch.empty((rows, cols // 16), dtype=torch.uint8, device=dev)
        outer = torch.empty((rows // rows_per_group,), dtype=torch.float32, device=dev)
    else:
        codes, scales, outer = out
    st = lib().pmn_nvfp4_quantize_per_group_noalloc(_ptr(x), rows, cols, rows_per_group, int(four_over_six),
                                                    _ptr(codes), _ptr(scales), _ptr(outer), _stream(stream))
    _check(st, "nvfp4_quantize_per_group_noalloc")
    return codes, scales, outer


def requant_transpose_sr_mxfp8(codes, scales, outer, outer_per_row, batch, rows, cols, seed, tag,
                               stochastic=True, out=None, stream=None):
    """NVFP4 [batch, rows, cols] -> MXFP8 transposed (u8 [batch, cols, rows], u8 [batch, cols, rows/32])."""
    _dev(codes, torch.uint8)
    _dev(scales, torch.uint8)
    _dev(outer, torch.float32)
    if out is None:
        q = torch.empty((batch, cols, rows), dtype=torch.uint8, device=codes.device)
        sc = torch.empty((batch, cols, rows // 32), dtype=torch.uint8, device=codes.device)
    else:
        q, sc = out
    st = lib().pmn_requant_transpose_sr_mxfp8(_ptr(codes), _ptr(scales), _ptr(outer),
                                              OUTER_PER_ROW if outer_per_row else OUTER_PER_GROUP, batch, rows,
                                              cols, seed, tag, ROUND_SR if stochastic else ROUND_RN, _ptr(q),
                                              _ptr(sc), _stream(stream))
    _check(st, "requant_transpose_sr_mxfp8")
    return q, sc


def requant_transpose_sr_nvfp4(codes, scales, outer, outer_per_row, batch, rows, cols, seed, tag,
                               stochastic=True, out=None, stream=None):
    """NVFP4 [batch, rows, cols] -> NVFP4 of the transpose with stochastic
    rounding (u8 codes [batch, cols, rows/2], u8 E4M3 [batch, cols, rows/16],
    f32 outer [batch]): the FP4 backward's requantisation."""
    _dev(codes, torch.uint8)
    _dev(scales, torch.uint8)
    _dev(outer, torch.float32)
    if out is None:
        q = torch.empty((batch, cols, rows // 2), dtype=torch.uint8, device=codes.device)
        sc = torch.empty((batch, cols, rows // 16), dtype=torch.uint8, device=codes.device)
        g = torch.empty((batch,), dtype=torch.float32, device=codes.device)
    else:
        q, sc, g = out
    st = lib().pmn_requant_transpose_sr_nvfp4(_ptr(codes), _ptr(scales), _ptr(outer),
                                              OUTER_PER_ROW if outer_per_row else OUTER_PER_GROUP, batch, rows,
                                              cols, seed, tag, ROUND_SR if stochastic else ROUND_RN, _ptr(q),
                                              _ptr(sc), _ptr(g), _stream(stream))
    _check(st, "requant_transpose_sr_nvfp4")
    return q, sc, g


def mxfp8_quantize(x, transpose=False, out=None, stream=None):
    """bf16 [rows, cols] -> MXFP8 with RN (u8 values, u8 E8M0 scales), optionally transposed."""
    _dev(x, torch.bfloat16)
    rows, cols = x.shape
    if out is None:
        shp = (cols, rows) if transpose else (rows, cols)
        q = torch.empty(shp, dtype=torch.uint8, device=x.device)
        sc = torch.empty((shp[0], shp[1] // 32), dtype=torch.uint8, device=x.device)
    else:
        q, sc = out
    _check(lib().pmn_mxfp8_quantize(_ptr(x), rows, cols, int(transpose), _ptr(q), _ptr(sc), _stream(stream)),
           "mxfp8_quantize")
    return q, sc


def mxfp8_quantize_both(x, out=None, out_t=None, stream=None):
    """bf16 [rows, cols] -> (MXFP8 rowwise (u8 [rows, cols], u8 [rows, cols/32]),
    MXFP8 of the transpose (u8 [cols, rows], u8 [cols, rows/32])) in one pass."""
    _dev(x, torch.bfloat16)
    rows, cols = x.shape
    dev = x.device
    if out is None:
        out = (torch.empty((rows, cols), dtype=torch.uint8, device=dev),
               torch.empty((rows, cols // 32), dtype=torch.uint8, device=dev))
    if out_t is None:
        out_t = (torch.empty((cols, rows), dtype=torch.uint8, device=dev),
                 torch.empty((cols, rows // 32), dtype=torch.uint8, device=dev))
    st = lib().pmn_mxfp8_quantize_both(_ptr(x), rows, cols, _ptr(out[0]), _ptr(out[1]), _ptr(out_t[0]),
                                       _ptr(out_t[1]), _stream(stream))
    _check(st, "mxfp8_quantize_both")
    return out, out_t


def mxfp8_quantize_swiglu(y, want_h=False, out=None, stream=None):
    """bf16 y [rows, 2f] (gate | up) -> MXFP8 (RN) of h = silu(gate) * up
    (u8 values [rows, f], u8 E8M0 scales [rows, f/32][, bf16 h])."""
    _dev(y, torch.bfloat16)
    rows, f2 = y.shape
    f = f2 // 2
    if out is None:
        q = torch.empty((rows, f), dtype=torch.uint8, device=y.device)
        sc = torch.empty((rows, f // 32), dtype=torch.uint8, device=y.device)
    else:
        q, sc = out
    h = torch.empty((rows, f), dtype=torch.bfloat16, device=y.device) if want_h else None
    _check(lib().pmn_mxfp8_quantize_swiglu(_ptr(y), rows, f, _ptr(q), _ptr(sc), _ptr(h), _stream(stream)),
           "mxfp8_quantize_swiglu")
    return (q, sc, h) if want_h else (q, sc)


def rht_s2f6_quantize(x, seed, out=None, stream=None):
    _dev(x, torch.float32)
    rows, cols = x.shape
    if out is None:
        q = torch.empty((rows, cols), dtype=torch.int8, device=x.device)
        sc = torch.empty((rows, cols // 32), dtype=torch.uint8, device=x.device)
    else:
        q, sc = out
    _check(lib().pmn_rht_s2f6_quantize(_ptr(x), rows, cols, seed, _ptr(q), _ptr(sc), _stream(stream)),
           "rht_s2f6_quantize")
    return q, sc


def combine_receive_s2f6(payload, seed, row_index, gates, out_dtype=torch.bfloat16, out=None, stream=None):
    """payload = (int8 [rows, cols], E8M0 uint8 [rows, cols/32]) in routed
    order; row_index int32 [tokens, k], gates float32 [tokens, k] -> the
    token rows [tokens, cols] (bf16 or float32)."""
    q, sc = payload
    _dev(q, torch.int8)
    _dev(sc, torch.uint8)
    _dev(row_index, torch.int32)
    _dev(gates, torch.float32)
    rows, cols = q.shape
    tokens, k = row_index.shape
    if tuple(gates.shape) != (tokens, k) or tuple(sc.shape) != (rows, cols // 32):
        raise PmnError("combine_receive_s2f6: shape mismatch")
    kind = {torch.bfloat16: OUT_BF16, torch.float32: OUT_F32}[out_dtype]
    if out is None:
        out = torch.empty((tokens, cols), dtype=out_dtype, device=q.device)
    _check(lib().pmn_combine_receive_s2f6(_ptr(q), _ptr(sc), rows, cols, seed, _ptr(row_index), _ptr(gates),
                                          tokens, k, kind, _ptr(out), _stream(stream)),
           "combine_receive_s2f6")
    return out


# ------------------------------------------------------------------ GEMMs
def grouped_gemm_nvfp4(a, b, offsets, out_dtype=torch.bfloat16, swiglu=False, out=None, stream=None):
    """a = (codes [T, K/2], scales [T, K/16], outer [T]); b = (codes [E, N, K/2],
    scales [E, N, K/16], outer [E]); offsets int32 [E+1] on the device.
    swiglu: the bf16 h = silu(gate) * up [T, N/2] of the float32 product
    (gate = the first N/2 rows of each B_e, up = the last N/2)."""
    ac, asc, ao = a
    bc, bsc, bo = b
    _dev(offsets, torch.int32)
    T = ac.shape[0]
    E, N = bc.shape[0], bc.shape[1]
    K = ac.shape[1] * 2
    kind = OUT_SWIGLU_BF16 if swiglu else (OUT_BF16 if out_dtype == torch.bfloat16 else OUT_F32)
    if out is None:
        out = torch.empty((T, N // 2 if swiglu else N), dtype=torch.bfloat16 if swiglu else out_dtype,
                          device=ac.device)
    st = lib().pmn_grouped_gemm_nvfp4(_ptr(ac), _ptr(asc), _ptr(ao), _ptr(bc), _ptr(bsc), _ptr(bo), _ptr(offsets),
                                      E, T, N, K, kind, _ptr(out), _stream(stream))
    _check(st, "grouped_gemm_nvfp4")
    return out


def w1_gemm_swiglu_nvfp4(a, b, offsets, four_over_six=True, out=None, h=None, stream=None):
    """w1 GEMM with SwiGLU in its epilogue, then NVFP4 (per token, 4/6) of h.
    a = NVFP4 rows (codes [T, K/2], scales [T, K/16], outer [T]); b = NVFP4 W1
    (codes [E, 2F, K/2], scales [E, 2F, K/16], outer [E]) with gate rows first.
    Returns (codes u8 [T, F/2], scales u8 [T, F/16], outer f32 [T]); `h` (bf16
    [T, F], allocated here when None) receives h itself."""
    ac, asc, ao = a
    bc, bsc, bo = b
    _dev(offsets, torch.int32)
    T = ac.shape[0]
    E, F2 = bc.shape[0], bc.shape[1]
    F = F2 // 2
    K = ac.shape[1] * 2
    dev = ac.device
    if out is None:
        out = (torch.empty((T, F // 2), dtype=torch.uint8, device=dev),
               torch.empty((T, F // 16), dtype=torch.uint8, device=dev),
               torch.empty((T,), dtype=torch.float32, device=dev))
    if h is None:
        h = torch.empty((T, F), dtype=torch.bfloat16, device=dev)
    _dev(h, torch.bfloat16)
    c, sc, g = out
    st = lib().pmn_w1_gemm_swiglu_nvfp4(_ptr(ac), _ptr(asc), _ptr(ao), _ptr(bc), _ptr(bsc), _ptr(bo), _ptr(offsets),
                                        E, T, F, K, int(four_over_six), _ptr(h), _ptr(c), _ptr(sc), _ptr(g),
                                        _stream(stream))
    _check(st, "w1_gemm_swiglu_nvfp4")
    return out


def w2_gemm_rht_s2f6(a, b, offsets, seed, out=None, debug_acc=None, stream=None):
    """(q int8 [T, N], scales u8 [T, N/32]); debug_acc: optional float32 [T, N] that receives the
    epilogue's input (the scaled accumulator) on the expert segments' rows."""
    ac, asc, ao = a
    bc, bsc, bo = b
    _dev(offsets, torch.int32)
    T = ac.shape[0]
    E, N = bc.shape[0], bc.shape[1]
    K = ac.shape[1] * 2
    if out is None:
        q = torch.empty((T, N), dtype=torch.int8, device=ac.device)
        sc = torch.empty((T, N // 32), dtype=torch.uint8, device=ac.device)
    else:
        q, sc = out
    if debug_acc is not None:
        _dev(debug_acc, torch.float32)
    st = lib().pmn_w2_gemm_rht_s2f6(_ptr(ac), _ptr(asc), _ptr(ao), _ptr(bc), _ptr(bsc), _ptr(bo), _ptr(offsets), E,
                                    T, N, K, seed, _ptr(q), _ptr(sc),
                                    _ptr(debug_acc) if debug_acc is not None else None, _stream(stream))
    _check(st, "w2_gemm_rht_s2f6")
    return q, sc


def gemm_mxfp8(a, a_sc, b, b_sc, offsets, group_mode, out_dtype=torch.float32, out=None, stream=None):
    """GROUP_M: a [M, K], b [G, N, K] -> [M, N];  GROUP_K: a [M, Kt], b [N, Kt] -> [G, M, N]."""
    _dev(offsets, torch.int32)
    G = offsets.numel() - 1
    M, K = a.shape
    N = b.shape[-2]
    kind = OUT_BF16 if out_dtype == torch.bfloat16 else OUT_F32
    if out is None:
        shp = (M, N) if group_mode == GROUP_M else (G, M, N)
        out = torch.empty(shp, dtype=out_dtype, device=a.device)
    st = lib().pmn_gemm_mxfp8(_ptr(a), _ptr(a_sc), _ptr(b), _ptr(b_sc), _ptr(offsets), G, group_mode, M, N, K, kind,
                              _ptr(out), _stream(stream))
    _check(st, "gemm_mxfp8")
    return out
