"""GPU parity of the MXFP8 forward (the precision the pages keep for the last
16.6 % of layers): MXFP8 (round to nearest) quantisation of X, W1, W2 and of
h after SwiGLU, both grouped FP8 GEMMs with bf16 outputs.

Bytes of every quantisation whose input comes from the oracle's side match
the oracle exactly.  GEMM outputs (one rounding of the float32 accumulator to
bf16) are within 2^-8 relative, half a bf16 step, plus 1e-3 (|A| |B|) of the
binary64 product of the same quantised operands.  h from the kernel's
float32 SiLU is within one bf16 step (at most 2^-7 relative) of the binary64
SwiGLU: float32 rounding can move a value across a bf16 midpoint.  Rows whose
h equals the oracle's bit for bit quantise bit for bit.
The second GEMM's output, whose input passes through the first GEMM's
rounding, is compared with the oracle's own chain within 2 % (relative
Frobenius).
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


def check_swiglu_quant(got_q, got_sc, got_h, y_bits, f, what):
    h_ref = oracle.swiglu_bf16(y_bits, f)
    hv, rv = f64(got_h), f64(h_ref)
    # one bf16 step, 2^(floor(log2 |h|) - 7), is at most |h| 2^-7
    assert np.all(np.abs(hv - rv) <= np.abs(rv) * 2.0 ** -7 + 1e-30), what + ": h beyond one bf16 step"
    same = np.all(got_h == h_ref, axis=1)
    assert same.mean() > 0.5, what + ": too few rows with h equal to the oracle's"
    rq, rsc = oracle.mxfp8_quantize(h_ref)
    assert np.array_equal(got_q[same], rq[same]) and np.array_equal(got_sc[same], rsc[same]), what
    return h_ref


@pytest.mark.parametrize("rows,f", [(96, 64), (257, 1536)])
def test_mxfp8_quantize_swiglu(P, rows, f):
    rng = np.random.default_rng(rows + f)
    y = W.normal_bf16_host(rng, (rows, 2 * f), 1.0, 0.01, 20.0)
    y[3, :] = 0                              # an all-zero row: scale byte of the smallest exponent
    q, sc, h = P.mxfp8_quantize_swiglu(bf16_dev(y), want_h=True)
    check_swiglu_quant(q.cpu().numpy(), sc.cpu().numpy(), host_bits(h), y, f, "swiglu mxfp8")
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
    z = f64(host_bits(fw.z))
    y_ref = np.zeros((r.rows, 2 * f), np.uint16)
    z_ref = np.zeros((r.rows, d))
    for e in range(E):
        lo, hi = int(r.offsets[e]), int(r.offsets[e + 1])
        if hi == lo:
            continue
        rows = slice(lo, hi)
        ref = check_gemm_bf16(y[rows], xq[rows], xs[rows], w1q[e * 2 * f:(e + 1) * 2 * f],
                              w1s[e * 2 * f:(e + 1) * 2 * f], "Y expert %d" % e)
        y_ref[rows] = oracle.bf16_rne_array(ref)
    # h and its MXFP8 bytes: test_mxfp8_quantize_swiglu checks the kernel on the oracle's inputs;
    # here the oracle runs its own chain from its own Y
    hq_r, hs_r = oracle.mxfp8_quantize(oracle.swiglu_bf16(y_ref, f))
    for e in range(E):
        lo, hi = int(r.offsets[e]), int(r.offsets[e + 1])
        if hi > lo:
            z_ref[lo:hi] = oracle.mxfp8_dequant_f64(hq_r[lo:hi], hs_r[lo:hi]) @ \
                oracle.mxfp8_dequant_f64(w2q[e * d:(e + 1) * d], w2s[e * d:(e + 1) * d]).T
    real = r.row_token >= 0
    rel = np.linalg.norm(z[real] - z_ref[real]) / np.linalg.norm(z_ref[real])
    assert rel < 0.02, rel


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
