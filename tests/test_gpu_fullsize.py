"""Parity at the full MoE-layer size, in the launch configuration bench.py
times (384 experts, top-8 of 16384 tokens, d_model 4096, d_ff 1536, one step
of layer.ExpertLayerStep).

The oracle recomputes sampled outputs one by one from host copies of the same
seeded inputs: sampled routed rows and sampled experts.  Bytes (codes,
scales, outer scales, MXFP8 values) must match exactly; GEMM outputs within
the stated tolerances (fp32: relative Frobenius 1e-5 and |err| <= 1e-3 (|A||B|);
bf16: additionally one bf16 step); h within the bound of test_gpu_swiglu_gemm.
The oracle never takes an input from the CUDA path.  Where a step's input is
itself a GEMM result (the w2 GEMM's h, the dW2 GEMM's H^T), the step is run a
second time, in the same launch configuration, with the sampled expert's
operand replaced by the oracle's own bytes, and checked element by element;
the step's own outputs are checked against the library's pinned standalone
kernels on every row (the combine payload against the standalone RHT + S2F6
kernel on the fused epilogue's input, the coding of h against the plain
row quantiser on the kernel's h).
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


def oracle_h(run, x_bits, e):
    """the oracle's chain for rows of expert e: NVFP4 of X (4/6), the binary64 w1
    product, |A||B|, h (SwiGLU of the product rounded to bf16, as the layer
    computes it) and its NVFP4 (4/6)"""
    xc, xs, xg = oracle.nvfp4_quantize(x_bits, oracle.OUTER_PER_ROW, four_over_six=True)
    wc, ws, wg = oracle_w(run, "w1", e)
    y = oracle.gemm_nvfp4(xc, xs, xg, wc, ws, wg[0])
    A = np.abs(oracle.nvfp4_dequant_f64(xc, xs)) * np.abs(xg[:, None].astype(np.float64))
    B = np.abs(oracle.nvfp4_dequant_f64(wc, ws)) * abs(float(wg[0]))
    F = wc.shape[0] // 2
    h = oracle.swiglu_bf16(oracle.bf16_rne_array(y), F)
    return y, A @ B.T, h, oracle.nvfp4_quantize(h, oracle.OUTER_PER_ROW, four_over_six=True)


def test_fullsize_forward_w1_gemm_swiglu(run):
    """h rows of a sampled expert against the oracle's chain; the NVFP4 of h on
    every row against the plain per-row quantiser on the layer's own h."""
    from swiglu_checks import check_h, check_h_coding
    from precision_moe_numerics_gb300 import pmn
    L, r = run["L"], run["r"]
    E, F2, D = L.w1.shape
    e = run["experts"][2]
    lo, hi = seg(r, e)
    n = min(hi - lo, 64)
    y, absab, _, _ = oracle_h(run, hb(L.x[lo:lo + n]), e)
    check_h(hb(L.h[lo:lo + n]), y, absab, F2 // 2, "h rows of expert %d" % e)
    check_h_coding(pmn, L.h, *L.hq, int(r.offsets[-1]), "full-size h")


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


def test_fullsize_combine_payload(run):
    """The w2 GEMM + RHT + S2F6 at full size.  (a) The step's payload on every
    row equals the standalone RHT + S2F6 kernel's bytes on the fused
    epilogue's input (read back through debug_acc).  (b) With the sampled
    expert's rows of h replaced by the oracle's NVFP4 of the oracle's own h,
    the epilogue's input on those rows is within the float32 GEMM tolerance
    of the binary64 product, and its bytes again equal the standalone
    kernel's."""
    from precision_moe_numerics_gb300 import pmn
    L, r = run["L"], run["r"]
    E, F2, D = L.w1.shape
    e = run["experts"][2]
    lo, hi = seg(r, e)
    rows = L.shape.rows
    acc = torch.empty((rows, D), dtype=torch.float32, device="cuda")
    q, sc = pmn.w2_gemm_rht_s2f6(L.hq, L.w2q3(), L.offsets, SEED, debug_acc=acc)
    end = int(r.offsets[-1])
    assert torch.equal(q[:end], L.z[0][:end]) and torch.equal(sc[:end], L.z[1][:end])
    sq, ssc = pmn.rht_s2f6_quantize(acc[:end], SEED)
    assert torch.equal(sq, q[:end]), "payload codes differ from the standalone kernel's"
    assert torch.equal(ssc, sc[:end]), "payload scales differ from the standalone kernel's"
    # (b) the oracle's h for expert e
    _, _, _, (hc, hs, hg) = oracle_h(run, hb(L.x[lo:hi]), e)
    hq = tuple(t.clone() for t in L.hq)
    hq[0][lo:hi] = torch.from_numpy(hc).cuda()
    hq[1][lo:hi] = torch.from_numpy(hs).cuda()
    hq[2][lo:hi] = torch.from_numpy(hg).cuda()
    q, sc = pmn.w2_gemm_rht_s2f6(hq, L.w2q3(), L.offsets, SEED, debug_acc=acc)
    w2c, w2s, w2g = oracle_w(run, "w2", e)
    z = oracle.gemm_nvfp4(hc, hs, hg, w2c, w2s, w2g[0])
    A = np.abs(oracle.nvfp4_dequant_f64(hc, hs)) * np.abs(hg[:, None].astype(np.float64))
    B = np.abs(oracle.nvfp4_dequant_f64(w2c, w2s)) * abs(float(w2g[0]))
    check_f32(hu(acc[lo:hi]), z, A @ B.T, "w2 accumulator of expert %d" % e)
    sq, ssc = pmn.rht_s2f6_quantize(acc[lo:hi], SEED)
    assert torch.equal(sq, q[lo:hi]) and torch.equal(ssc, sc[lo:hi])
    del acc


def test_fullsize_backward_dw2_gemm(run):
    """dW2 of a sampled expert: the K-grouped GEMM over all 384 experts, run
    with the expert's columns of H^T replaced by the oracle's SR requantisation
    of the oracle's NVFP4 of its own h, against dY^T . H^T of the oracle's
    operands in binary64, element by element."""
    from precision_moe_numerics_gb300 import pmn
    L, r = run["L"], run["r"]
    E, F2, D = L.w1.shape
    F = F2 // 2
    e = run["experts"][2]
    lo, hi = seg(r, e)
    _, _, _, (hc, hs, hg) = oracle_h(run, hb(L.x[lo:hi]), e)
    ht, hts = oracle.requant_transpose_mxfp8(hc, hs, hg, True, 1, hi - lo, F, SEED, oracle.TAG_H,
                                            rows_total=L.shape.rows, r_begin=lo)
    hq = L.ht[0][0].clone()
    hqs = L.ht[1][0].clone()
    hq[:, lo:hi] = torch.from_numpy(ht[0]).cuda()
    hqs[:, lo // 32:hi // 32] = torch.from_numpy(hts[0]).cuda()
    dw2 = pmn.gemm_mxfp8(L.dy_t[0], L.dy_t[1], hq, hqs, L.offsets, pmn.GROUP_K, torch.float32)
    torch.cuda.synchronize()
    assert pmn.get_device_error() == 0
    dq, dqs = oracle.mxfp8_quantize(hb(L.dy[lo:hi]), transpose=True)
    A = oracle.mxfp8_dequant_f64(dq, dqs)
    B = oracle.mxfp8_dequant_f64(ht[0], hts[0])
    check_f32(hu(dw2[e]), A @ B.T, np.abs(A) @ np.abs(B).T, "dW2 of expert %d" % e)
    # the step's own dW2 of that expert is the same GEMM on the step's H^T
    assert torch.equal(pmn.gemm_mxfp8(L.dy_t[0], L.dy_t[1], L.ht[0][0], L.ht[1][0], L.offsets, pmn.GROUP_K,
                                      torch.float32)[e], L.dw2[e])
    del dw2


def test_fullsize_step_is_deterministic(run):
    L = run["L"]
    before = [t.clone() for t in (L.z[0], L.dw1[:2], L.dx[:512], L.w1t[0][:2], L.h, L.hq[0], L.hq[2])]
    L.step()
    torch.cuda.synchronize()
    after = (L.z[0], L.dw1[:2], L.dx[:512], L.w1t[0][:2], L.h, L.hq[0], L.hq[2])
    for a, b in zip(before, after):
        assert torch.equal(a, b)


def test_decode_forward_against_oracle(run):
    """Decode batch: 64 tokens, top-8 of the 384 experts, segments of 1-5 rows
    (not padded), against the step's NVFP4 weights of every expert.  The
    activation codes and scales are bytes; h rows of the first, the last and
    the most-used hit expert within the SwiGLU bound, and the NVFP4 of h on
    every row equal to the plain quantiser's on the kernel's h; the combine
    payload on every row equal to the standalone RHT + S2F6 kernel's bytes on
    the fused epilogue's input, and that input, on the most-used expert's rows
    with h replaced by the oracle's own NVFP4 of its h, within the float32
    GEMM tolerance of the binary64 product."""
    from swiglu_checks import check_h, check_h_coding
    from precision_moe_numerics_gb300 import layer, pmn
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
        y, absab, _, _ = oracle_h(run, xb[lo:hi], e)
        check_h(hb(dec.h[lo:hi]), y, absab, F, "decode h rows of expert %d" % e)
    check_h_coding(pmn, dec.h, *dec.hq, int(r.offsets[-1]), "decode h")
    T = xb.shape[0]
    acc = torch.empty((T, D), dtype=torch.float32, device="cuda")
    q, sc = pmn.w2_gemm_rht_s2f6(dec.hq, L.w2q3(), offs, SEED, debug_acc=acc)
    assert torch.equal(q, dec.z[0]) and torch.equal(sc, dec.z[1])
    sq, ssc = pmn.rht_s2f6_quantize(acc, SEED)
    assert torch.equal(sq, q) and torch.equal(ssc, sc)
    lo, hi = seg(r, top)
    _, _, _, (hc, hs, hg) = oracle_h(run, xb[lo:hi], top)
    hq = tuple(t.clone() for t in dec.hq)
    for t, v in zip(hq, (hc, hs, hg)):
        t[lo:hi] = torch.from_numpy(v).cuda()
    q, sc = pmn.w2_gemm_rht_s2f6(hq, L.w2q3(), offs, SEED, debug_acc=acc)
    w2c, w2s, w2g = oracle_w(run, "w2", top)
    z = oracle.gemm_nvfp4(hc, hs, hg, w2c, w2s, w2g[0])
    A = np.abs(oracle.nvfp4_dequant_f64(hc, hs)) * np.abs(hg[:, None].astype(np.float64))
    B = np.abs(oracle.nvfp4_dequant_f64(w2c, w2s)) * abs(float(w2g[0]))
    check_f32(hu(acc[lo:hi]), z, A @ B.T, "decode w2 accumulator of expert %d" % top)
    sq, ssc = pmn.rht_s2f6_quantize(acc[lo:hi], SEED)
    assert torch.equal(sq, q[lo:hi]) and torch.equal(ssc, sc[lo:hi])
    assert pmn.get_device_error() == 0
