"""Parity at the full MoE-layer size, in the launch configuration bench.py
times (384 experts, top-8 of 16384 tokens, d_model 4096, d_ff 1536, one step
of layer.ExpertLayerStep).

The oracle recomputes sampled outputs one by one from host copies of the same
seeded inputs: sampled routed rows and sampled experts.  Bytes (codes,
scales, outer scales, MXFP8 values) must match exactly; GEMM outputs within
the stated tolerances (fp32: relative Frobenius 1e-5 and |err| <= 1e-3 (|A||B|);
bf16: additionally one bf16 step).  Outputs whose inputs are themselves GEMM
results (h, the combine payload, dW2) are checked by properties against the
oracle's own binary64 pipeline, since the oracle never takes inputs from the
CUDA path.
"""
import numpy as np
import pytest
import torch

import oracle
from precision_moe_numerics_gb300 import workloads as W

pytestmark = pytest.mark.gpu

SEED = 0


@pytest.fixture(scope="module")
def run():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from precision_moe_numerics_gb300 import build, layer, pmn
    build.build()
    inp = W.moe_device(SEED, device="cuda")
    r = inp["routing"]
    offs = torch.from_numpy(r.offsets.astype(np.int32)).cuda()
    L = layer.ExpertLayerStep(inp["x"], inp["w1"], inp["w2"], inp["dy"], inp["dy1"], offs, r.real_rows, seed=SEED)
    L.step()
    torch.cuda.synchronize()
    assert pmn.get_device_error() == 0
    rng = np.random.default_rng(1)
    nz = [e for e in range(len(r.counts)) if r.counts[e] > 0]
    experts = sorted({nz[0], nz[-1], int(rng.choice(nz))})
    return {"L": L, "inp": inp, "r": r, "experts": experts, "rng": rng}


def hb(t):
    """device bf16 -> host uint16 bits"""
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def hu(t):
    return t.cpu().numpy()


def same(a, b, what):
    a = np.asarray(a)
    b = np.asarray(b)
    if a.dtype == np.float32:
        a, b = a.view(np.uint32), b.astype(np.float32).view(np.uint32)
    bad = np.argwhere(a != b)
    assert bad.size == 0, "%s: %d mismatches, first at %s" % (what, len(bad), bad[0])


def seg(r, e):
    return int(r.offsets[e]), int(r.offsets[e + 1])


def check_f32(got, ref, absab, what):
    got = np.asarray(got, np.float64)
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    assert rel <= 1e-5, "%s: relative Frobenius error %.3e" % (what, rel)
    assert np.all(np.abs(got - ref) <= 1e-3 * absab + 1e-30), what


def check_bf16(got_bits, ref, absab, what):
    g = W.bf16_bits_to_f32(got_bits).astype(np.float64)
    bad = np.abs(g - ref) > np.abs(ref) * 2.0 ** -8 + 1e-3 * absab + 1e-30
    assert not bad.any(), "%s: %d elements beyond one bf16 step" % (what, bad.sum())


def oracle_w(run, which, e):
    """oracle NVFP4 of one expert's weight matrix (outer scale over the expert)"""
    w = hb(run["inp"][which][e])
    return oracle.nvfp4_quantize(w, oracle.OUTER_PER_GROUP, group_offsets=[0, w.shape[0]])


def test_fullsize_quantise_activation_rows(run):
    L, r = run["L"], run["r"]
    rows = np.sort(np.concatenate([run["rng"].choice(r.rows, 96, replace=False),
                                   [0, r.rows - 1, int(r.offsets[run["experts"][1]])]]))
    x = hb(L.x[torch.from_numpy(rows).cuda()])
    c, s, g = oracle.nvfp4_quantize(x, oracle.OUTER_PER_ROW, four_over_six=True)
    idx = torch.from_numpy(rows).cuda()
    same(hu(L.xq[0][idx]), c, "X codes")
    same(hu(L.xq[1][idx]), s, "X scales")
    same(hu(L.xq[2][idx]), g, "X outer")


def test_fullsize_quantise_weights(run):
    L = run["L"]
    E, F2, D = L.w1.shape
    for e in run["experts"][:2]:
        c, s, g = oracle_w(run, "w1", e)
        same(hu(L.w1q[0][e * F2:(e + 1) * F2]), c, "W1 codes e=%d" % e)
        same(hu(L.w1q[1][e * F2:(e + 1) * F2]), s, "W1 scales e=%d" % e)
        same(hu(L.w1q[2][e:e + 1]), g, "W1 outer e=%d" % e)
        c, s, g = oracle_w(run, "w2", e)
        same(hu(L.w2q[0][e * D:(e + 1) * D]), c, "W2 codes e=%d" % e)
        same(hu(L.w2q[2][e:e + 1]), g, "W2 outer e=%d" % e)


def test_fullsize_requant_weights_and_activations(run):
    L, r = run["L"], run["r"]
    E, F2, D = L.w1.shape
    e = run["experts"][1]
    c, s, g = oracle_w(run, "w1", e)
    q, qs = oracle.requant_transpose_mxfp8(c, s, g, False, 1, F2, D, SEED, oracle.TAG_W1, b_begin=e)
    same(hu(L.w1t[0][e]), q[0], "W1^T values")
    same(hu(L.w1t[1][e]), qs[0], "W1^T scales")
    lo, hi = seg(r, e)
    x = hb(L.x[lo:hi])
    xc, xs, xg = oracle.nvfp4_quantize(x, oracle.OUTER_PER_ROW, four_over_six=True)
    q, qs = oracle.requant_transpose_mxfp8(xc, xs, xg, True, 1, hi - lo, D, SEED, oracle.TAG_X,
                                          rows_total=L.shape.rows, r_begin=lo)
    same(hu(L.xt[0][0][:, lo:hi]), q[0], "X^T values")
    same(hu(L.xt[1][0][:, lo // 32:hi // 32]), qs[0], "X^T scales")


def test_fullsize_requant_nvfp4_weights(run):
    """The FP4 backward's requantisation of all 384 experts' w1 in one call;
    two experts compared byte for byte with the oracle's requantisation of
    its own NVFP4 of the same bf16 weights (random bits by the full index)."""
    from precision_moe_numerics_gb300 import pmn
    L = run["L"]
    E, F2, D = L.w1.shape
    q, qs, qg = pmn.requant_transpose_sr_nvfp4(L.w1q[0], L.w1q[1], L.w1q[2], False, E, F2, D, SEED, oracle.TAG_W1)
    torch.cuda.synchronize()
    assert pmn.get_device_error() == 0
    for e in run["experts"][:2]:
        c, s, g = oracle_w(run, "w1", e)
        rc, rs, rg = oracle.requant_transpose_nvfp4(c, s, g, False, 1, F2, D, SEED, oracle.TAG_W1, b_begin=e)
        same(hu(q[e]), rc[0], "W1^T NVFP4 codes")
        same(hu(qs[e]), rs[0], "W1^T NVFP4 scales")
        same(hu(qg[e:e + 1]), rg, "W1^T NVFP4 outer")
    del q, qs, qg


def test_fullsize_gradient_quantisation(run):
    L, r = run["L"], run["r"]
    lo, hi = seg(r, run["experts"][1])
    dy = hb(L.dy[lo:hi])
    q, qs = oracle.mxfp8_quantize(dy)
    same(hu(L.dy_r[0][lo:hi]), q, "dY rows")
    same(hu(L.dy_r[1][lo:hi]), qs, "dY row scales")
    qt, qts = oracle.mxfp8_quantize(dy, transpose=True)
    same(hu(L.dy_t[0][:, lo:hi]), qt, "dY^T")
    same(hu(L.dy_t[1][:, lo // 32:hi // 32]), qts, "dY^T scales")


def test_fullsize_forward_w1_gemm(run):
    L, r = run["L"], run["r"]
    E, F2, D = L.w1.shape
    e = run["experts"][2]
    lo, hi = seg(r, e)
    rows = np.arange(lo, min(hi, lo + 64))
    x = hb(L.x[lo:lo + len(rows)])
    xc, xs, xg = oracle.nvfp4_quantize(x, oracle.OUTER_PER_ROW, four_over_six=True)
    wc, ws, wg = oracle_w(run, "w1", e)
    ref = oracle.gemm_nvfp4(xc, xs, xg, wc, ws, wg[0])
    A = np.abs(oracle.nvfp4_dequant_f64(xc, xs)) * np.abs(xg[:, None].astype(np.float64))
    B = np.abs(oracle.nvfp4_dequant_f64(wc, ws)) * abs(float(wg[0]))
    check_bf16(hb(L.y[lo:lo + len(rows)]), ref, A @ B.T, "Y rows of expert %d" % e)


def test_fullsize_backward_dx_gemm(run):
    L, r = run["L"], run["r"]
    E, F2, D = L.w1.shape
    e = run["experts"][0]
    lo, hi = seg(r, e)
    n = min(hi - lo, 64)
    dq, dqs = oracle.mxfp8_quantize(hb(L.dy1[lo:lo + n]))
    c, s, g = oracle_w(run, "w1", e)
    wt, wts = oracle.requant_transpose_mxfp8(c, s, g, False, 1, F2, D, SEED, oracle.TAG_W1, b_begin=e)
    ref = oracle.gemm_mxfp8_mgrouped(dq, dqs, wt, wts, [0, n])
    absab = np.abs(oracle.mxfp8_dequant_f64(dq, dqs)) @ np.abs(oracle.mxfp8_dequant_f64(wt[0], wts[0])).T
    check_bf16(hb(L.dx[lo:lo + n]), ref, absab, "dX rows of expert %d" % e)


def test_fullsize_backward_dw1_gemm(run):
    L, r = run["L"], run["r"]
    E, F2, D = L.w1.shape
    e = run["experts"][1]
    lo, hi = seg(r, e)
    dq, dqs = oracle.mxfp8_quantize(hb(L.dy1[lo:hi]), transpose=True)  # [F2, n]
    xc, xs, xg = oracle.nvfp4_quantize(hb(L.x[lo:hi]), oracle.OUTER_PER_ROW, four_over_six=True)
    xt, xts = oracle.requant_transpose_mxfp8(xc, xs, xg, True, 1, hi - lo, D, SEED, oracle.TAG_X,
                                            rows_total=L.shape.rows, r_begin=lo)
    A = oracle.mxfp8_dequant_f64(dq, dqs)
    B = oracle.mxfp8_dequant_f64(xt[0], xts[0])
    ref = A @ B.T
    check_f32(hu(L.dw1[e]), ref, np.abs(A) @ np.abs(B).T, "dW1 of expert %d" % e)


def test_fullsize_combine_and_dw2_properties(run):
    """h, the combine payload and dW2 take GPU GEMM results as inputs, so they
    are compared with the oracle's own binary64 pipeline by loose properties:
    decoded combine output and dW2 within 2 % relative Frobenius error."""
    L, r = run["L"], run["r"]
    E, F2, D = L.w1.shape
    F = F2 // 2
    e = run["experts"][2]
    lo, hi = seg(r, e)
    n = hi - lo
    xc, xs, xg = oracle.nvfp4_quantize(hb(L.x[lo:hi]), oracle.OUTER_PER_ROW, four_over_six=True)
    w1c, w1s, w1g = oracle_w(run, "w1", e)
    y = oracle.bf16_rne_array(oracle.gemm_nvfp4(xc, xs, xg, w1c, w1s, w1g[0]))
    h = oracle.swiglu_bf16(y, F)
    hc, hs, hg = oracle.nvfp4_quantize(h, oracle.OUTER_PER_ROW, four_over_six=True)
    w2c, w2s, w2g = oracle_w(run, "w2", e)
    z = oracle.gemm_nvfp4(hc, hs, hg, w2c, w2s, w2g[0])
    zq = oracle.s2f6_dequant_inverse_rht(hu(L.z[0][lo:hi]), hu(L.z[1][lo:hi]), SEED)
    real = int(r.counts[e])
    rel = np.linalg.norm(zq[:real] - z[:real]) / np.linalg.norm(z[:real])
    assert rel < 0.02, rel
    ht, hts = oracle.requant_transpose_mxfp8(hc, hs, hg, True, 1, n, F, SEED, oracle.TAG_H,
                                            rows_total=L.shape.rows, r_begin=lo)
    dq, dqs = oracle.mxfp8_quantize(hb(L.dy[lo:hi]), transpose=True)
    ref = oracle.mxfp8_dequant_f64(dq, dqs) @ oracle.mxfp8_dequant_f64(ht[0], hts[0]).T
    got = hu(L.dw2[e]).astype(np.float64)
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert rel < 0.02, rel


def test_fullsize_step_is_deterministic(run):
    L = run["L"]
    before = [t.clone() for t in (L.z[0], L.dw1[:2], L.dx[:512], L.w1t[0][:2])]
    L.step()
    torch.cuda.synchronize()
    after = (L.z[0], L.dw1[:2], L.dx[:512], L.w1t[0][:2])
    for a, b in zip(before, after):
        assert torch.equal(a, b)


def test_decode_forward_against_oracle(run):
    """Decode batch: 64 tokens, top-8 of the 384 experts, segments of 1-5 rows
    (not padded), against the step's NVFP4 weights of every expert.  The
    activation codes and scales are bytes; Y rows of the first, the last and
    the most-used hit expert within the GEMM tolerance; the combine payload of
    the most-used one by the step's property."""
    from precision_moe_numerics_gb300 import layer
    L = run["L"]
    E, F2, D = L.w1.shape
    F = F2 // 2
    r = W.decode_routing(SEED)
    xb = W.decode_x(r, SEED, D)
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
    offs = torch.from_numpy(r.offsets.astype(np.int32)).cuda()
    dec = layer.DecodeForward(x, L.w1q3(), L.w2q3(), offs, seed=SEED)
    dec.forward()
    torch.cuda.synchronize()
    xc, xs, xg = oracle.nvfp4_quantize(xb, oracle.OUTER_PER_ROW, four_over_six=True)
    same(hu(dec.xq[0]), xc, "decode X codes")
    same(hu(dec.xq[1]), xs, "decode X scales")
    same(hu(dec.xq[2]), xg, "decode X outer")
    hit = [e for e in range(E) if r.counts[e] > 0]
    top = int(np.argmax(r.counts))
    for e in sorted({hit[0], hit[-1], top}):
        lo, hi = seg(r, e)
        wc, ws, wg = oracle_w(run, "w1", e)
        ref = oracle.gemm_nvfp4(xc[lo:hi], xs[lo:hi], xg[lo:hi], wc, ws, wg[0])
        A = np.abs(oracle.nvfp4_dequant_f64(xc[lo:hi], xs[lo:hi])) * np.abs(xg[lo:hi, None].astype(np.float64))
        B = np.abs(oracle.nvfp4_dequant_f64(wc, ws)) * abs(float(wg[0]))
        check_bf16(hb(dec.y[lo:hi]), ref, A @ B.T, "decode Y rows of expert %d" % e)
    lo, hi = seg(r, top)
    w1c, w1s, w1g = oracle_w(run, "w1", top)
    y = oracle.bf16_rne_array(oracle.gemm_nvfp4(xc[lo:hi], xs[lo:hi], xg[lo:hi], w1c, w1s, w1g[0]))
    h = oracle.swiglu_bf16(y, F)
    hc, hs, hg = oracle.nvfp4_quantize(h, oracle.OUTER_PER_ROW, four_over_six=True)
    w2c, w2s, w2g = oracle_w(run, "w2", top)
    z = oracle.gemm_nvfp4(hc, hs, hg, w2c, w2s, w2g[0])
    zq = oracle.s2f6_dequant_inverse_rht(hu(dec.z[0][lo:hi]), hu(dec.z[1][lo:hi]), SEED)
    rel = np.linalg.norm(zq - z) / np.linalg.norm(z)
    assert rel < 0.02, rel
