"""GPU parity of the MXFP8 forward (the precision the pages keep for the last
16.6 % of layers): MXFP8 (round to nearest) quantisation of X, W1, W2 and of
h after SwiGLU, both grouped FP8 GEMMs with bf16 outputs.

Bytes of every quantisation whose input comes from the oracle's side match
the oracle exactly.  GEMM outputs (one rounding of the float32 accumulator to
bf16) are within 2^-8 relative, half a bf16 step, plus 1e-3 (|A| |B|) of the
binary64 product of the same quantised operands.  h from the kernel's
float32 SiLU is within one bf16 step (at most 2^-7 relative) of the binary64
SwiGLU: float32 rounding can move a value across a bf16 midpoint.  On every
row, the MXFP8 bytes of h equal those of the plain MXFP8 quantiser run on the
kernel's own h (that quantiser is pinned byte for byte to the oracle in
test_gpu_quant.py).  The second GEMM runs on the oracle's MXFP8 of the
oracle's own h and is checked element by element like the first.
"""
import numpy as np
import pytest
import torch

import oracle
from precision_moe_numerics_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def P():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from precision_moe_numerics_gb300 import build, pmn
    build.build()
    return pmn


def bf16_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def host_bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def f64(bits):
    return W.bf16_bits_to_f32(bits).astype(np.float64)


def check_gemm_bf16(got_bits, a, a_sc, b, b_sc, what):
    A, B = oracle.mxfp8_dequant_f64(a, a_sc), oracle.mxfp8_dequant_f64(b, b_sc)
    ref = A @ B.T
    absab = np.abs(A) @ np.abs(B).T
    bad = np.abs(f64(got_bits) - ref) > np.abs(ref) * 2.0 ** -8 + 1e-3 * absab + 1e-30
    assert not bad.any(), "%s: %d elements beyond one bf16 step" % (what, int(bad.sum()))
    return ref


def check_swiglu_quant(P, got_q, got_sc, got_h, y_bits, f, what):
    """h within one bf16 step of binary64 everywhere; the MXFP8 bytes of h equal, on every row, the
    plain (oracle-pinned) quantiser's on the kernel's own h"""
    h_ref = oracle.swiglu_bf16(y_bits, f)
    hv, rv = f64(host_bits(got_h)), f64(h_ref)
    # one bf16 step, 2^(floor(log2 |h|) - 7), is at most |h| 2^-7
    assert np.all(np.abs(hv - rv) <= np.abs(rv) * 2.0 ** -7 + 1e-30), what + ": h beyond one bf16 step"
    pq, psc = P.mxfp8_quantize(got_h)
    assert torch.equal(got_q, pq), what + ": MXFP8 values of h differ from the plain quantiser's"
    assert torch.equal(got_sc, psc), what + ": MXFP8 scales of h differ from the plain quantiser's"
    return h_ref


@pytest.mark.parametrize("rows,f", [(96, 64), (257, 1536)])
def test_mxfp8_quantize_swiglu(P, rows, f):
    rng = np.random.default_rng(rows + f)
    y = W.normal_bf16_host(rng, (rows, 2 * f), 1.0, 0.01, 20.0)
    y[3, :] = 0                              # an all-zero row: scale byte of the smallest exponent
    q, sc, h = P.mxfp8_quantize_swiglu(bf16_dev(y), want_h=True)
    check_swiglu_quant(P, q, sc, h, y, f, "swiglu mxfp8")
    assert np.all(q.cpu().numpy()[3] == 0)
    q2, sc2 = P.mxfp8_quantize_swiglu(bf16_dev(y))  # without h: same bytes
    assert torch.equal(q, q2) and torch.equal(sc, sc2)


def test_mxfp8_quantize_swiglu_arguments(P):
    with pytest.raises(P.PmnError):      # f % 32 != 0
        P.mxfp8_quantize_swiglu(torch.zeros((4, 96), dtype=torch.bfloat16, device="cuda"))
    q, sc = P.mxfp8_quantize_swiglu(torch.zeros((0, 128), dtype=torch.bfloat16, device="cuda"))
    assert q.shape == (0, 64)


def test_mxfp8_forward_small_moe(P):
    from precision_moe_numerics_gb300 import layer
    E, d, f = 8, 512, 512
    m = W.small_moe(0, tokens=256, experts=E, k=2, d=d, f=f)
    r = m["routing"]
    offs = torch.from_numpy(r.offsets.astype(np.int32)).cuda()
    fw = layer.MXFP8Forward(bf16_dev(m["x"]), bf16_dev(m["w1"]), bf16_dev(m["w2"]), offs)
    fw.forward()
    torch.cuda.synchronize()
    assert P.get_device_error() == 0
    xq, xs = oracle.mxfp8_quantize(m["x"])
    w1q, w1s = oracle.mxfp8_quantize(m["w1"].reshape(E * 2 * f, d))
    w2q, w2s = oracle.mxfp8_quantize(m["w2"].reshape(E * d, f))
    for got, want, what in ((fw.xq, (xq, xs), "X"), (fw.w1q, (w1q, w1s), "W1"), (fw.w2q, (w2q, w2s), "W2")):
        assert np.array_equal(got[0].cpu().numpy(), want[0]) and np.array_equal(got[1].cpu().numpy(), want[1]), what
    y = host_bits(fw.y)
    y_ref = np.zeros((r.rows, 2 * f), np.uint16)
    for e in range(E):
        lo, hi = int(r.offsets[e]), int(r.offsets[e + 1])
        if hi == lo:
            continue
        rows = slice(lo, hi)
        ref = check_gemm_bf16(y[rows], xq[rows], xs[rows], w1q[e * 2 * f:(e + 1) * 2 * f],
                              w1s[e * 2 * f:(e + 1) * 2 * f], "Y expert %d" % e)
        y_ref[rows] = oracle.bf16_rne_array(ref)
    # h and its MXFP8 bytes from the layer's own Y, on every row
    qh, sch, hh = P.mxfp8_quantize_swiglu(fw.y, want_h=True)
    assert torch.equal(qh, fw.hq[0]) and torch.equal(sch, fw.hq[1])
    pq, psc = P.mxfp8_quantize(hh)
    assert torch.equal(fw.hq[0], pq) and torch.equal(fw.hq[1], psc)
    # the second GEMM on the oracle's MXFP8 of the oracle's own h, element by element
    hq_r, hs_r = oracle.mxfp8_quantize(oracle.swiglu_bf16(y_ref, f))
    z_or = P.gemm_mxfp8(torch.from_numpy(hq_r).cuda(), torch.from_numpy(hs_r).cuda(), fw.w2q[0].view(E, d, f),
                        fw.w2q[1].view(E, d, f // 32), offs, P.GROUP_M, torch.bfloat16)
    zb = host_bits(z_or)
    for e in range(E):
        lo, hi = int(r.offsets[e]), int(r.offsets[e + 1])
        if hi > lo:
            check_gemm_bf16(zb[lo:hi], hq_r[lo:hi], hs_r[lo:hi], w2q[e * d:(e + 1) * d], w2s[e * d:(e + 1) * d],
                            "Z expert %d" % e)


def test_mxfp8_forward_fullsize_sampled(P):
    """The bench's configuration (384 experts, top-8 of 16384 tokens, d_model
    4096, d_ff 1536): the quantised bytes of three experts' weights and their
    routed rows exactly, their Y rows within the GEMM tolerance."""
    from precision_moe_numerics_gb300 import layer
    inp = W.moe_device(0, device="cuda", with_backward=False)
    r = inp["routing"]
    offs = torch.from_numpy(r.offsets.astype(np.int32)).cuda()
    fw = layer.MXFP8Forward(inp["x"], inp["w1"], inp["w2"], offs)
    fw.forward()
    torch.cuda.synchronize()
    assert P.get_device_error() == 0
    E, F2, D = inp["w1"].shape
    nz = [e for e in range(E) if r.counts[e] > 0]
    for e in sorted({nz[0], nz[-1], nz[len(nz) // 2]}):
        lo, hi = int(r.offsets[e]), int(r.offsets[e + 1])
        x_e = host_bits(inp["x"][lo:hi])
        w_e = host_bits(inp["w1"][e])
        xq, xs = oracle.mxfp8_quantize(x_e)
        wq, ws = oracle.mxfp8_quantize(w_e)
        assert np.array_equal(fw.xq[0][lo:hi].cpu().numpy(), xq) and np.array_equal(fw.xq[1][lo:hi].cpu().numpy(), xs)
        assert np.array_equal(fw.w1q[0][e * F2:(e + 1) * F2].cpu().numpy(), wq)
        assert np.array_equal(fw.w1q[1][e * F2:(e + 1) * F2].cpu().numpy(), ws)
        check_gemm_bf16(host_bits(fw.y[lo:hi]), xq, xs, wq, ws, "full-size Y expert %d" % e)
