"""Checks shared by the SwiGLU parity tests: the bound on h from the fused w1
GEMM epilogue against the oracle's binary64 SwiGLU of the binary64 product,
and the byte check of the NVFP4 coding of h against the plain per-row
quantiser on the kernel's h."""
import numpy as np
import torch

import oracle
from precision_moe_numerics_gb300 import workloads as W


def f64(bits):
    return W.bf16_bits_to_f32(bits).astype(np.float64)


def gemm_ref(ac, asc, ag, bc, bsc, bg, offs):
    """binary64 product and (|A| |B|) with the outer scales, rows of the segments"""
    ref = oracle.grouped_gemm_nvfp4(ac, asc, ag, bc, bsc, bg, offs)
    absab = np.zeros_like(ref)
    for e in range(len(offs) - 1):
        lo, hi = int(offs[e]), int(offs[e + 1])
        if hi > lo:
            A = np.abs(oracle.nvfp4_dequant_f64(ac[lo:hi], asc[lo:hi]))
            B = np.abs(oracle.nvfp4_dequant_f64(bc[e], bsc[e]))
            absab[lo:hi] = (A @ B.T) * np.abs(ag[lo:hi, None].astype(np.float64)) * abs(float(bg[e]))
    return ref, absab


def swiglu_bound(y, absab, f):
    """2 (|dh/da| tau_a + |dh/db| tau_b) at the binary64 point, with tau the bf16
    GEMM tolerance of y: 2^-8 |y| (y is rounded to bf16 before the SwiGLU) +
    1e-3 (|A||B|)"""
    a, b = y[:, :f], y[:, f:2 * f]
    tau = 2.0 ** -8 * np.abs(y) + 1e-3 * absab
    with np.errstate(over="ignore"):
        sig = 1.0 / (1.0 + np.exp(-a))
    dha = np.abs(b * sig * (1.0 + a * (1.0 - sig)))
    dhb = np.abs(a * sig)
    return 2.0 * (dha * tau[:, :f] + dhb * tau[:, f:2 * f])


def check_h(h_bits, y_ref, absab, f, what):
    hr = f64(oracle.swiglu_bf16_from_f64(y_ref, f))
    hg = f64(h_bits)
    tol = np.abs(hr) * (2.0 ** -7 + 2.0 ** -16) + swiglu_bound(y_ref, absab, f) + 1e-30
    bad = np.abs(hg - hr) > tol
    assert not bad.any(), "%s: %d of %d h values beyond the bound, first at %s" % (
        what, int(bad.sum()), bad.size, np.argwhere(bad)[0])


def check_h_coding(P, h, codes, scales, outer, row_end, what):
    """every row: the plain per-row quantiser on the kernel's h gives the same bytes;
    rows at or past row_end: a zero row's quantisation"""
    pc, ps, pg = P.nvfp4_quantize(h, four_over_six=True)
    for got, want, name in ((codes, pc, "codes"), (scales, ps, "scales"), (outer, pg, "outer")):
        g, w = got[:row_end], want[:row_end]
        assert torch.equal(g.view(torch.uint8), w.view(torch.uint8)), "%s: h %s differ" % (what, name)
    if row_end < codes.shape[0]:
        assert torch.all(codes[row_end:] == 0) and torch.all(scales[row_end:] == 0), what
        assert torch.all(outer[row_end:] == 1.0), what
