"""Pins for the oracle's requantisation, dY quantisation, RHT + S2F6 and GEMMs
(no GPU).  Checks use brute force over the code tables, exact rational
arithmetic, explicit Hadamard matrices and statistical invariants."""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from precision_moe_numerics_gb300 import workloads as W

E4M3_FINITE = [(b, oracle.e4m3_value(b)) for b in range(256) if not np.isnan(oracle.e4m3_value(b))]


def _brute_e4m3_rn(y):
    """nearest finite E4M3 value (ties to the even mantissa), sign kept"""
    a = abs(y)
    best = min((b for b, v in E4M3_FINITE if not (b & 0x80)),
               key=lambda b: (abs(oracle.e4m3_value(b) - a), b & 1))
    return best | (0x80 if np.signbit(y) else 0)


def _brute_exponent(amax, top=448.0):
    if amax == 0:
        return -127
    e = -127
    while amax > top * 2.0 ** e:
        e += 1
    return min(e, 127)


def _random_nvfp4(rng, rows, cols):
    x = W.normal_bf16_host(rng, (rows, cols), 1.0, 0.02, 30.0)
    return oracle.nvfp4_quantize(x, oracle.OUTER_PER_ROW)


def test_requant_rn_is_transpose_with_brute_force_rounding():
    rng = np.random.default_rng(0)
    rows, cols = 64, 48
    c, s, g = _random_nvfp4(rng, rows, cols)
    d = oracle.nvfp4_dequant_f32(c, s, g).astype(np.float64)
    q, qs = oracle.requant_transpose_mxfp8(c, s, g, True, 1, rows, cols, 0, 1, stochastic=False)
    assert q.shape == (1, cols, rows) and qs.shape == (1, cols, rows // 32)
    for cc in range(0, cols, 5):
        for rb in range(rows // 32):
            blk = d[rb * 32:(rb + 1) * 32, cc]
            e = _brute_exponent(np.abs(blk).max())
            assert qs[0, cc, rb] == e + 127
            for j in range(0, 32, 3):
                assert q[0, cc, rb * 32 + j] == _brute_e4m3_rn(blk[j] / 2.0 ** e)


def test_requant_sr_index_mapping_and_padding():
    rng = np.random.default_rng(1)
    batch, rows, cols = 2, 64, 32
    x = W.normal_bf16_host(rng, (batch * rows, cols))
    x[rows - 32:rows] = 0  # a zero (padding) segment
    c, s, g = oracle.nvfp4_quantize(x, oracle.OUTER_PER_GROUP, group_offsets=[0, rows, 2 * rows])
    seed, tag = 77, 3
    q, qs = oracle.requant_transpose_mxfp8(c, s, g, False, batch, rows, cols, seed, tag)
    d = oracle.nvfp4_dequant_f32(c, s, g, rows_per_outer=rows).astype(np.float64)
    for b in range(batch):
        for cc in (0, 7, 31):
            for r in (0, 5, 33, 63):
                e = int(qs[b, cc, r // 32]) - 127
                y = d[b * rows + r, cc] / 2.0 ** e
                i = (b * cols + cc) * rows + r
                assert q[b, cc, r] == oracle.e4m3_sr(y, oracle.sr_bits16(seed, tag, i))
    assert np.all(q[0, :, 32:64] == 0) and np.all(qs[0, :, 1] == 0)


def test_requant_sr_expectation_equals_transposed_dequant():
    """E[w_q] = E[(w_q^T)^T]: the mean over seeds of the requantised transpose
    tends to the transpose of the forward dequantisation."""
    rng = np.random.default_rng(2)
    rows, cols = 32, 32
    c, s, g = _random_nvfp4(rng, rows, cols)
    d = oracle.nvfp4_dequant_f32(c, s, g).astype(np.float64)
    n = 400
    acc = np.zeros((cols, rows))
    for seed in range(n):
        q, qs = oracle.requant_transpose_mxfp8(c, s, g, True, 1, rows, cols, seed, 1)
        acc += oracle.mxfp8_dequant_f64(q[0], qs[0])
    mean = acc / n
    # grid step at each element: E4M3 ulp of |y| (>= 2^-9) times the block scale
    e = np.repeat(qs[0].astype(np.int64) - 127, 32, axis=1).astype(np.float64)
    y = np.abs(d.T) / 2.0 ** e
    k = np.floor(np.log2(np.maximum(y, 2.0 ** -6)))
    step = 2.0 ** (k - 3) * 2.0 ** e
    tol = 6 * step * np.sqrt(0.25 / n) + step * 2.0 ** -16
    assert np.all(np.abs(mean - d.T) <= tol)
    assert np.abs(mean - d.T).mean() < 0.1 * step.mean()
    # and SR differs from RN somewhere (it is not a deterministic rounding)
    q0, _ = oracle.requant_transpose_mxfp8(c, s, g, True, 1, rows, cols, 0, 1, stochastic=False)
    q1, _ = oracle.requant_transpose_mxfp8(c, s, g, True, 1, rows, cols, 1, 1)
    assert not np.array_equal(q0, q1)


def test_mxfp8_quantize_rn_brute_force_both_orientations():
    rng = np.random.default_rng(3)
    x = W.normal_bf16_host(rng, (64, 96), 1e-3)
    xf = W.bf16_bits_to_f32(x).astype(np.float64)
    q, qs = oracle.mxfp8_quantize(x, transpose=False)
    qt, qts = oracle.mxfp8_quantize(x, transpose=True)
    for r in range(0, 64, 7):
        for b in range(3):
            blk = xf[r, b * 32:(b + 1) * 32]
            e = _brute_exponent(np.abs(blk).max())
            assert qs[r, b] == e + 127
            for j in range(0, 32, 4):
                assert q[r, b * 32 + j] == _brute_e4m3_rn(blk[j] / 2.0 ** e)
    q2, qs2 = oracle.mxfp8_quantize(np.ascontiguousarray(x.T), transpose=False)
    assert np.array_equal(qt, q2) and np.array_equal(qts, qs2)


# ------------------------------------------------------------------ RHT + S2F6 [NVLink]
def _sylvester(n):
    H = np.array([[1]], np.int64)
    while H.shape[0] < n:
        H = np.block([[H, H], [H, -H]])
    return H


def test_rht_matrix_is_hadamard_and_orthogonal():
    cols = np.stack([oracle.rht32(np.eye(32, dtype=np.float32)[j], 0) for j in range(32)], axis=1)
    Hint = np.rint(cols.astype(np.float64) * np.sqrt(32.0)).astype(np.int64)
    assert np.array_equal(np.abs(Hint), np.ones((32, 32), np.int64))
    assert np.array_equal(Hint @ Hint, 32 * np.eye(32, dtype=np.int64))
    assert np.array_equal(Hint, _sylvester(32))
    Q = cols.astype(np.float64)
    assert np.abs(Q.T @ Q - np.eye(32)).max() < 1e-6
    # unit vector -> flat +-1/sqrt(32), exactly RN(1/sqrt(32)) in binary32
    assert np.all(np.abs(cols) == oracle.rsqrt32())
    assert np.float32(oracle.rsqrt32()).view(np.uint32) == np.float32(1 / np.sqrt(32.0)).view(np.uint32)


def test_rht_signs_and_values_vs_explicit_matrix():
    rng = np.random.default_rng(4)
    H = _sylvester(32).astype(np.float64) / np.sqrt(32.0)
    for seed in (0, 1, 12345):
        sigma = oracle.rht_sign_word(seed)
        assert sigma == oracle.philox4x32_10([0, 0, 5, 0], [seed & 0xFFFFFFFF, seed >> 32])[0]
        s = np.array([-1.0 if (sigma >> j) & 1 else 1.0 for j in range(32)])
        x = rng.standard_normal(32).astype(np.float32)
        z = oracle.rht32(x, sigma).astype(np.float64)
        want = H @ (s * x.astype(np.float64))
        assert np.abs(z - want).max() <= 8 * 2.0 ** -24 * np.abs(x).sum()


def test_s2f6_scale_rule_and_round_trip():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((64, 128)) * 10.0 ** rng.uniform(-3, 3, (64, 1))).astype(np.float32)
    x[3, :32] = 0
    seed = 0
    q, sc = oracle.rht_s2f6(x, seed)
    assert q.dtype == np.int8 and np.all(q >= -127)
    sigma = oracle.rht_sign_word(seed)
    for r in range(64):
        for b in range(4):
            z = oracle.rht32(x[r, b * 32:(b + 1) * 32], sigma).astype(np.float64)
            e = int(sc[r, b]) - 127
            amax = np.abs(z).max()
            assert e == _brute_exponent(amax, 127 / 64)
            k = np.rint(z * 2.0 ** (6 - e))
            assert np.array_equal(k.astype(np.int8), q[r, b * 32:(b + 1) * 32])
    xr = oracle.s2f6_dequant_inverse_rht(q, sc, seed)
    for r in range(64):
        for b in range(4):
            e = int(sc[r, b]) - 127
            err = np.linalg.norm(xr[r, b * 32:(b + 1) * 32] - x[r, b * 32:(b + 1) * 32])
            bound = np.sqrt(32) * 2.0 ** (e - 7) * 1.001 + 1e-6 * np.linalg.norm(x[r, b * 32:(b + 1) * 32])
            assert err <= bound
    assert np.all(q[3, :32] == 0) and sc[3, 0] == 0


def _receive_by_matrices(q, sc, seed, row_index, gates):
    """The receive side restated with explicit matrices: decoded block z =
    k / 64 * 2^(b - 127); back-transformed block = D_sigma (H / sqrt(32)) z
    with H the explicit Sylvester matrix; token rows = sum of gate * row."""
    rows, cols = q.shape
    sigma = oracle.rht_sign_word(seed)
    D = np.diag([-1.0 if (sigma >> j) & 1 else 1.0 for j in range(32)])
    M = D @ _sylvester(32).astype(np.float64) / np.sqrt(32.0)
    z = q.astype(np.float64).reshape(rows, cols // 32, 32) / 64.0 * np.exp2(sc.astype(np.float64) - 127.0)[:, :, None]
    back = np.einsum("ij,rbj->rbi", M, z).reshape(rows, cols)
    out = np.zeros((row_index.shape[0], cols))
    for t in range(row_index.shape[0]):
        for i in range(row_index.shape[1]):
            if row_index[t, i] >= 0:
                out[t] += float(gates[t, i]) * back[row_index[t, i]]
    return out


def test_combine_receive_vs_explicit_matrices():
    rng = np.random.default_rng(11)
    rows, cols, tokens, k = 12, 96, 7, 3
    q = rng.integers(-128, 128, (rows, cols)).astype(np.int8)
    q[0, :32] = -128
    q[1, 32:64] = 127
    sc = rng.integers(110, 141, (rows, cols // 32)).astype(np.uint8)
    idx = rng.integers(0, rows, (tokens, k))
    idx[2, 1] = -1          # a dropped choice
    idx[4, :] = -1          # a token with no choice left
    gates = rng.uniform(0.0, 1.0, (tokens, k)).astype(np.float32)
    for seed in (0, 7):
        got = oracle.combine_receive(q, sc, seed, idx, gates)
        want = _receive_by_matrices(q, sc, seed, idx, gates)
        scale = np.abs(want).max()
        assert np.abs(got - want).max() <= 1e-13 * scale
        assert np.all(got[4] == 0.0)
    # the sign word matters: another seed's signs give another result
    assert not np.allclose(oracle.combine_receive(q, sc, 0, idx, gates), oracle.combine_receive(q, sc, 7, idx, gates))
    # no token: empty result
    assert oracle.combine_receive(q, sc, 0, np.zeros((0, k), np.int64), np.zeros((0, k), np.float32)).shape == (0, cols)


def test_combine_receive_inverts_the_combine_quantisation():
    """Routed copies of each token row go through the forward combine
    quantisation and come back: with gates summing to 1 the token row is
    recovered to within the S2F6 rounding, half a step 2^(e-6) per
    transformed coordinate, i.e. sqrt(32) * 2^(e-7) in 2-norm per block
    (the transform is orthogonal), weighted by the gates."""
    rng = np.random.default_rng(12)
    tokens, experts, k, cols, seed = 40, 6, 3, 128, 5
    routing = W.route_topk(rng.standard_normal((tokens, experts)).astype(np.float32), k, pad=32)
    x = (rng.standard_normal((tokens, cols)) * 10.0 ** rng.uniform(-2, 2, (tokens, 1))).astype(np.float32)
    xr = np.zeros((routing.rows, cols), np.float32)
    real = routing.row_token >= 0
    xr[real] = x[routing.row_token[real]]
    q, sc = oracle.rht_s2f6(xr, seed)
    idx = routing.token_rows()
    np.testing.assert_allclose(routing.gates.sum(axis=1), 1.0, rtol=1e-6)
    got = oracle.combine_receive(q, sc, seed, idx, routing.gates)
    for t in range(tokens):
        for b in range(cols // 32):
            sl = slice(32 * b, 32 * b + 32)
            e = sc[idx[t], b].astype(np.float64) - 127.0
            bound = float(np.sum(routing.gates[t] * np.sqrt(32.0) * np.exp2(e - 7.0))) * 1.001
            bound += 1e-6 * np.linalg.norm(x[t, sl])   # binary32 butterflies of the forward side
            assert np.linalg.norm(got[t, sl] - x[t, sl] * routing.gates[t].astype(np.float64).sum()) <= bound


def test_routing_token_rows_inverts_row_token():
    r = W.route_topk(np.random.default_rng(13).standard_normal((50, 9)).astype(np.float32), 3, pad=32)
    idx = r.token_rows()
    assert idx.dtype == np.int32 and idx.shape == (50, 3)
    for t in range(50):
        for i in range(3):
            row = idx[t, i]
            assert r.row_token[row] == t
            assert r.offsets[r.topk[t, i]] <= row < r.offsets[r.topk[t, i] + 1]
    assert np.all(np.diff(r.gates, axis=1) <= 0) and np.all(r.gates > 0)


# ------------------------------------------------------------------ GEMMs
def _exact_nvfp4_matrix(codes, scales):
    rows, cols = codes.shape[0], codes.shape[1] * 2
    M = [[None] * cols for _ in range(rows)]
    for r in range(rows):
        for c in range(cols):
            byte = int(codes[r, c // 2])
            code = (byte >> 4) if c % 2 else (byte & 15)
            M[r][c] = Fraction(oracle.e2m1_value(code)) * Fraction(oracle.e4m3_value(int(scales[r, c // 16])))
    return M


def test_nvfp4_gemm_exact_rational():
    rng = np.random.default_rng(6)
    M, N, K = 5, 7, 64
    ac = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    asc = rng.integers(0x20, 0x60, (M, K // 16), dtype=np.uint8)
    bc = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    bsc = rng.integers(0x20, 0x60, (N, K // 16), dtype=np.uint8)
    ga = (2.0 ** rng.integers(-3, 3, M)).astype(np.float32)
    gb = np.float32(0.25)
    got = oracle.gemm_nvfp4(ac, asc, ga, bc, bsc, gb)
    A, B = _exact_nvfp4_matrix(ac, asc), _exact_nvfp4_matrix(bc, bsc)
    for m in range(M):
        for n in range(N):
            ex = sum(A[m][k] * B[n][k] for k in range(K)) * Fraction(float(ga[m])) * Fraction(float(gb))
            assert Fraction(got[m, n]) == ex


def test_grouped_gemm_groups_and_sampling():
    rng = np.random.default_rng(7)
    K, N, E = 32, 16, 4
    offs = [0, 5, 5, 12, 20]
    ac = rng.integers(0, 256, (20, K // 2), dtype=np.uint8)
    asc = rng.integers(0x20, 0x50, (20, K // 16), dtype=np.uint8)
    ga = rng.uniform(0.5, 2, 20).astype(np.float32)
    bc = rng.integers(0, 256, (E, N, K // 2), dtype=np.uint8)
    bsc = rng.integers(0x20, 0x50, (E, N, K // 16), dtype=np.uint8)
    gb = rng.uniform(0.5, 2, E).astype(np.float32)
    full = oracle.grouped_gemm_nvfp4(ac, asc, ga, bc, bsc, gb, offs)
    for e in range(E):
        for m in range(offs[e], offs[e + 1]):
            one = oracle.gemm_nvfp4(ac[m:m + 1], asc[m:m + 1], ga[m:m + 1], bc[e], bsc[e], gb[e])
            assert np.array_equal(full[m], one[0])
    rows = [0, 7, 19]
    assert np.array_equal(oracle.grouped_gemm_nvfp4(ac, asc, ga, bc, bsc, gb, offs, rows=rows), full[rows])


def _exact_mx(q, sc):
    rows, cols = q.shape
    return [[Fraction(oracle.e4m3_value(int(q[r, c]))) * Fraction(oracle.e8m0_value(int(sc[r, c // 32])))
             for c in range(cols)] for r in range(rows)]


def test_mxfp8_gemms_exact_rational():
    rng = np.random.default_rng(8)
    fin = np.array([b for b, _ in E4M3_FINITE], np.uint8)
    M, N, K = 6, 5, 64
    a = rng.choice(fin, (M, K)); a_sc = rng.integers(120, 134, (M, K // 32), dtype=np.uint8)
    b = rng.choice(fin, (2, N, K)); b_sc = rng.integers(120, 134, (2, N, K // 32), dtype=np.uint8)
    got = oracle.gemm_mxfp8_mgrouped(a, a_sc, b, b_sc, [0, 2, 6])
    A = _exact_mx(a, a_sc)
    for m in range(M):
        e = 0 if m < 2 else 1
        B = _exact_mx(b[e], b_sc[e])
        for n in range(N):
            assert Fraction(got[m, n]) == sum(A[m][k] * B[n][k] for k in range(K))
    # K-grouped: segments of the contraction axis
    Kt = 96
    a2 = rng.choice(fin, (M, Kt)); a2s = rng.integers(120, 134, (M, Kt // 32), dtype=np.uint8)
    b2 = rng.choice(fin, (N, Kt)); b2s = rng.integers(120, 134, (N, Kt // 32), dtype=np.uint8)
    offs = [0, 32, 32, 96]
    got2 = oracle.gemm_mxfp8_kgrouped(a2, a2s, b2, b2s, offs)
    A2, B2 = _exact_mx(a2, a2s), _exact_mx(b2, b2s)
    for e in range(3):
        for m in range(M):
            for n in range(N):
                ex = sum(A2[m][k] * B2[n][k] for k in range(offs[e], offs[e + 1]))
                assert Fraction(got2[e][m, n]) == ex


def test_swiglu_vs_torch_silu():
    rng = np.random.default_rng(9)
    y = W.normal_bf16_host(rng, (32, 64), 2.0)
    h = oracle.swiglu_bf16(y, 32)
    yf = torch.from_numpy(W.bf16_bits_to_f32(y).astype(np.float64))
    ref = torch.nn.functional.silu(yf[:, :32]) * yf[:, 32:]
    got = torch.from_numpy(W.bf16_bits_to_f32(h).astype(np.float64))
    ulp = torch.clamp(ref.abs(), min=1e-30) * 2.0 ** -8
    assert torch.all((got - ref).abs() <= ulp)


def test_swiglu_from_f64_vs_torch_and_bf16_inputs():
    """SwiGLU on binary64 GEMM outputs: against torch's silu in float64 (one
    bf16 rounding), and equal to the bf16-input form when the inputs are
    themselves bf16 values."""
    rng = np.random.default_rng(10)
    y = rng.standard_normal((16, 96)) * 3.0
    h = oracle.swiglu_bf16_from_f64(y, 48)
    yt = torch.from_numpy(y)
    ref = torch.nn.functional.silu(yt[:, :48]) * yt[:, 48:]
    got = torch.from_numpy(W.bf16_bits_to_f32(h).astype(np.float64))
    assert torch.all((got - ref).abs() <= ref.abs() * 2.0 ** -8 + 1e-30)
    yb = W.normal_bf16_host(rng, (16, 96), 2.0)
    assert np.array_equal(oracle.swiglu_bf16_from_f64(W.bf16_bits_to_f32(yb).astype(np.float64), 48),
                          oracle.swiglu_bf16(yb, 48))


def test_requant_window_equals_slice_of_full():
    """The windowed form (used for sampled checks at full size) equals the
    matching slice of the whole-tensor computation, random bits included."""
    rng = np.random.default_rng(31)
    batch, rows, cols = 3, 128, 64
    x = W.normal_bf16_host(rng, (batch * rows, cols))
    c, s, g = oracle.nvfp4_quantize(x, oracle.OUTER_PER_GROUP, group_offsets=np.arange(batch + 1) * rows)
    full, full_sc = oracle.requant_transpose_mxfp8(c, s, g, False, batch, rows, cols, 5, 3)
    b0, r0, nr = 1, 64, 32
    cw = c.reshape(batch, rows, -1)[b0:b0 + 1, r0:r0 + nr]
    sw = s.reshape(batch, rows, -1)[b0:b0 + 1, r0:r0 + nr]
    win, win_sc = oracle.requant_transpose_mxfp8(cw, sw, g[b0:b0 + 1], False, 1, nr, cols, 5, 3,
                                                 b_begin=b0, rows_total=rows, r_begin=r0)
    assert np.array_equal(win[0], full[b0][:, r0:r0 + nr])
    assert np.array_equal(win_sc[0], full_sc[b0][:, r0 // 32:(r0 + nr) // 32])
    # per-row outer scales (activations)
    c2, s2, g2 = oracle.nvfp4_quantize(x[:rows], oracle.OUTER_PER_ROW)
    f2, f2s = oracle.requant_transpose_mxfp8(c2, s2, g2, True, 1, rows, cols, 9, 1)
    w2, w2s = oracle.requant_transpose_mxfp8(c2[r0:r0 + nr], s2[r0:r0 + nr], g2[r0:r0 + nr], True, 1, nr, cols,
                                             9, 1, rows_total=rows, r_begin=r0)
    assert np.array_equal(w2[0], f2[0][:, r0:r0 + nr]) and np.array_equal(w2s[0], f2s[0][:, r0 // 32:(r0 + nr) // 32])
