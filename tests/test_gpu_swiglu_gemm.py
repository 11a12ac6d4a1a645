"""GPU parity of the w1 GEMM with SwiGLU in its epilogue followed by the NVFP4
coding of h (pmn_w1_gemm_swiglu_nvfp4), and of the single-expert forward at
T = 4096 tokens (X -> NVFP4 with 4/6 -> w1 GEMM + SwiGLU -> NVFP4 of h -> w2
GEMM -> bf16).

h.  The epilogue rounds y = acc * g_t * g_e to bf16 (as the bf16 GEMM output
does), then forms h = silu(gate) * up in binary32 and rounds h to bf16: the
arithmetic of the unfused path (bf16 GEMM output, then the row quantiser's
SwiGLU input mode), so h must equal that path's h bit for bit.  Against the
oracle (swiglu_bf16_from_f64 of the binary64 product): per element
|h - h_ref| <= 2^-7 |h_ref| (two roundings to bf16, half a step each)
+ 2^-16 |h_ref| (the float32 SwiGLU with the approximate exponential and
division, a few dozen float32 ulps) + 2 (|dh/da| tau_a + |dh/db| tau_b), the
bf16 GEMM tolerance of y, tau = 2^-8 |y| + 1e-3 (|A||B|) (outer scales
included), carried through the SwiGLU to first order with a factor of two.

NVFP4 of h.  Codes, scales and outer scales equal, byte for byte on every row,
those of the plain per-row quantiser (pmn_nvfp4_quantize, PER_ROW, 4/6) run on
the kernel's own h; that quantiser is pinned byte for byte to the oracle on
seeded inputs (test_gpu_quant.py).  Rows past the last expert segment are the
quantisation of a zero row.

GEMM outputs in bf16: within 2^-8 relative (half a bf16 step) plus
1e-3 (|A||B|) of the binary64 product of the same quantised operands.
"""
import numpy as np
import pytest
import torch

import oracle
from precision_moe_numerics_gb300 import workloads as W
from swiglu_checks import check_h, check_h_coding, f64, gemm_ref

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pmn():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from precision_moe_numerics_gb300 import build, pmn as P
    build.build()
    return P


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def dev_bf16(bits):
    return dev(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def host_bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def run_case(P, x_bits, w1_bits, offs, f, extra_rows=0, what=""):
    """quantise with the oracle, run the fused call on those bytes, check h and its coding"""
    E = len(offs) - 1
    d = x_bits.shape[1]
    ac, asc, ag = oracle.nvfp4_quantize(x_bits, oracle.OUTER_PER_ROW, four_over_six=True)
    bq = oracle.nvfp4_quantize(w1_bits.reshape(E * 2 * f, d), oracle.OUTER_PER_GROUP,
                               group_offsets=np.arange(E + 1) * 2 * f)
    bc, bsc, bg = bq[0].reshape(E, 2 * f, d // 2), bq[1].reshape(E, 2 * f, d // 16), bq[2]
    rows = int(offs[-1])
    T = rows + extra_rows
    pad = lambda a, v: np.concatenate([a, np.full((extra_rows,) + a.shape[1:], v, a.dtype)])
    A = (dev(pad(ac, 0)), dev(pad(asc, 0)), dev(pad(ag, 1.0)))
    B = (dev(bc), dev(bsc), dev(bg))
    doffs = dev(np.asarray(offs, np.int32))
    h = torch.full((T, f), 7.0, dtype=torch.bfloat16, device="cuda")  # rows past the segments stay 7.0
    codes, scales, outer = P.w1_gemm_swiglu_nvfp4(A, B, doffs, True, h=h)
    torch.cuda.synchronize()
    assert P.get_device_error() == 0
    y_ref, absab = gemm_ref(ac, asc, ag, bc, bsc, bg, offs)
    check_h(host_bits(h[:rows]), y_ref, absab, f, what)
    assert torch.all(h[rows:] == 7.0), what + ": rows outside the segments were written"
    check_h_coding(P, h, codes, scales, outer, rows, what)
    return A, B, doffs, h, (codes, scales, outer)


def test_swiglu_gemm_small_moe(pmn):
    P = pmn
    E, d, f = 8, 512, 256
    m = W.small_moe(0, tokens=256, experts=E, k=2, d=d, f=f)
    r = m["routing"]
    A, B, offs, h, hq = run_case(P, m["x"], m["w1"], r.offsets, f, extra_rows=40, what="small MoE")
    # the GEMM's SwiGLU output alone (out_kind PMN_OUT_SWIGLU_BF16) is the h of the fused call
    h2 = torch.full_like(h, 7.0)
    P.grouped_gemm_nvfp4(A, B, offs, swiglu=True, out=h2)
    assert torch.equal(h.view(torch.int16), h2.view(torch.int16))
    # the unfused path (bf16 Y, then the row quantiser's SwiGLU input mode) gives the same h and bytes
    rows = int(r.offsets[-1])
    y = P.grouped_gemm_nvfp4(A, B, offs, out_dtype=torch.bfloat16)
    uc, us, ug, uh = P.nvfp4_quantize(y[:rows], cols=f, swiglu=True, four_over_six=True, want_h=True)
    assert torch.equal(uh.view(torch.int16), h[:rows].view(torch.int16))
    for a, b in zip((uc, us, ug), hq):
        assert torch.equal(a.view(torch.uint8), b[:rows].view(torch.uint8))
    # run to run: same bytes
    again = P.w1_gemm_swiglu_nvfp4(A, B, offs, True)
    for a, b in zip(hq, again):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))


def test_swiglu_gemm_edge_offsets(pmn):
    """empty experts, a 1-row expert, ragged tails, rows not a multiple of 32,
    segments that start inside a 128-row tile; one 128-wide tile of h (f = 128)"""
    rng = np.random.default_rng(41)
    d, f = 512, 128
    counts = [0, 1, 129, 0, 31, 300]
    E = len(counts)
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    x = W.normal_bf16_host(rng, (int(offs[-1]), d), 1.0, 0.01, 30.0)
    x[5] = 0  # an all-zero row: h = 0, outer 1
    w1 = W.normal_bf16_host(rng, (E, 2 * f, d), 0.02)
    run_case(pmn, x, w1, offs, f, extra_rows=3, what="edge offsets")


def test_swiglu_gemm_short_segments(pmn):
    """a decode-like batch (16 or fewer rows per expert on average, where the
    library takes 32-row tiles): empty experts, 1..5-row segments, and 33- and
    70-row segments that need several 32-row tiles"""
    rng = np.random.default_rng(42)
    d, f = 512, 256
    counts = [1, 2, 0, 70, 3, 0, 5, 1, 0, 2, 33, 4]
    E = len(counts)
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    assert offs[-1] <= 16 * E
    x = W.normal_bf16_host(rng, (int(offs[-1]), d), 1.0, 0.01, 30.0)
    w1 = W.normal_bf16_host(rng, (E, 2 * f, d), 0.02)
    run_case(pmn, x, w1, offs, f, extra_rows=5, what="short segments")


def test_swiglu_gemm_rejects_bad_arguments(pmn):
    z8 = torch.zeros((128, 128), dtype=torch.uint8, device="cuda")
    A = (z8, torch.zeros((128, 16), dtype=torch.uint8, device="cuda"), torch.ones(128, device="cuda"))
    # f = 192 is not a multiple of 128
    B = (torch.zeros((1, 384, 128), dtype=torch.uint8, device="cuda"),
         torch.zeros((1, 384, 16), dtype=torch.uint8, device="cuda"), torch.ones(1, device="cuda"))
    offs = torch.tensor([0, 128], dtype=torch.int32, device="cuda")
    with pytest.raises(pmn.PmnError):
        pmn.w1_gemm_swiglu_nvfp4(A, B, offs, True)


def test_single_expert_forward(pmn):
    """The single-expert forward at T = 4096 tokens (d_model 4096, d_ff 1536):
    every step checked element by element.
      X (4/6, per token), W1, W2 (per expert): bytes equal the oracle's.
      w1 GEMM + SwiGLU: h within the bound above, against the oracle's h from
        its own quantised operands (the same bytes, checked first).
      NVFP4 of h: equal to the plain per-row quantiser on the kernel's h.
      w2 GEMM (bf16 out): on the oracle's NVFP4 of its own h, within the bf16
        GEMM tolerance of the oracle's binary64 product."""
    P = pmn
    d = W.expert(0)
    x, w1, w2 = d["x"], d["w1"], d["w2"]
    T, D = x.shape
    F = w2.shape[1]
    xq = P.nvfp4_quantize(dev_bf16(x), four_over_six=True)
    w1q = P.nvfp4_quantize(dev_bf16(w1), outer_mode=P.OUTER_PER_GROUP, rows_per_group=2 * F)
    w2q = P.nvfp4_quantize(dev_bf16(w2), outer_mode=P.OUTER_PER_GROUP, rows_per_group=D)
    offs = dev(np.array([0, T], np.int32))
    h = torch.empty((T, F), dtype=torch.bfloat16, device="cuda")
    w1q3 = (w1q[0].view(1, 2 * F, D // 2), w1q[1].view(1, 2 * F, D // 16), w1q[2])
    hq = P.w1_gemm_swiglu_nvfp4(xq, w1q3, offs, True, h=h)
    w2q3 = (w2q[0].view(1, D, F // 2), w2q[1].view(1, D, F // 16), w2q[2])
    torch.cuda.synchronize()
    assert P.get_device_error() == 0

    rx = oracle.nvfp4_quantize(x, oracle.OUTER_PER_ROW, four_over_six=True)
    rw1 = oracle.nvfp4_quantize(w1, oracle.OUTER_PER_GROUP, group_offsets=[0, 2 * F])
    rw2 = oracle.nvfp4_quantize(w2, oracle.OUTER_PER_GROUP, group_offsets=[0, D])
    for got, want, what in ((xq, rx, "X"), (w1q, rw1, "W1"), (w2q, rw2, "W2")):
        for g, w, part in zip(got, want, ("codes", "scales", "outer")):
            g = g.cpu().numpy()
            if g.dtype == np.float32:
                g, w = g.view(np.uint32), np.asarray(w, np.float32).view(np.uint32)
            assert np.array_equal(g, w), "%s %s differ from the oracle's" % (what, part)

    b1 = (rw1[0].reshape(1, 2 * F, D // 2), rw1[1].reshape(1, 2 * F, D // 16), rw1[2])
    y_ref, absab = gemm_ref(rx[0], rx[1], rx[2], *b1, [0, T])
    check_h(host_bits(h), y_ref, absab, F, "single expert")
    check_h_coding(P, h, *hq, T, "single expert")

    # w2 GEMM on the oracle's own NVFP4 of its own h (the SwiGLU of the product rounded to bf16)
    h_ref = oracle.swiglu_bf16(oracle.bf16_rne_array(y_ref), F)
    rh = oracle.nvfp4_quantize(h_ref, oracle.OUTER_PER_ROW, four_over_six=True)
    b2 = (rw2[0].reshape(1, D, F // 2), rw2[1].reshape(1, D, F // 16), rw2[2])
    z = P.grouped_gemm_nvfp4((dev(rh[0]), dev(rh[1]), dev(rh[2])), tuple(dev(a) for a in b2), offs,
                             out_dtype=torch.bfloat16)
    z_ref, zab = gemm_ref(rh[0], rh[1], rh[2], *b2, [0, T])
    zg = f64(host_bits(z))
    bad = np.abs(zg - z_ref) > np.abs(z_ref) * 2.0 ** -8 + 1e-3 * zab + 1e-30
    assert not bad.any(), "w2 GEMM: %d elements beyond the bf16 GEMM tolerance" % int(bad.sum())
    # and the chain through the GPU's own h runs: the same call on the kernel's h coding
    z2 = P.grouped_gemm_nvfp4(hq, w2q3, offs, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert torch.isfinite(z2.float()).all()
    assert P.get_device_error() == 0
