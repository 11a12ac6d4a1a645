"""Oracle pins for the NVFP4 requantisation of the FP4 backward (dequantise ->
transpose -> NVFP4 with stochastic rounding), against the pages' worked
example and brute force over the E4M3 and E2M1 grids (no GPU)."""
import json
import os

import numpy as np

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def e4m3_grid():
    return np.array([oracle.e4m3_value(b) for b in range(0x7F)])  # 0 .. 448, ascending


def e2m1_value(code):
    v = E2M1[code & 7]
    return -v if code & 8 else v


def unpack(codes):
    lo, hi = codes & 15, codes >> 4
    return np.stack([lo, hi], axis=-1).reshape(*codes.shape[:-1], -1)


def decode_nvfp4(codes, scales, g):
    c = unpack(codes)
    v = np.vectorize(e2m1_value)(c)
    s = np.vectorize(oracle.e4m3_value)(scales)
    return v * np.repeat(s, 16, axis=-1) * g


def test_pages_transpose_example():
    """The pages' example: 5.4 stored as 0.5 in a scale-9 block (value 4.5);
    after the transpose its block has scale 2, 4.5 / 2 = 2.25, which rounds to
    2 (nearest) or to 2 / 3 with probabilities 3/4 / 1/4 (stochastic)."""
    ex = json.load(open(os.path.join(HERE, "golden", "pages_examples.json")))["transpose_sr_example"]
    rows, cols = 32, 64
    codes = np.zeros((rows, cols // 2), np.uint8)
    scales = np.zeros((rows, cols // 16), np.uint8)
    e4m3 = {oracle.e4m3_value(b): b for b in range(0x7F)}
    # row 0, column 0: code 0.5 in a block of scale 9 -> 4.5
    codes[0, 0] = 1
    scales[0, 0] = e4m3[ex["forward_scale"]]
    # row 1, column 0: 12 = 6 * 2, which sets the transposed block's scale to 12 / 6 = 2
    codes[1, 0] = 7
    scales[1, 0] = e4m3[2.0]
    # a block elsewhere with the largest scale fixes the outer scale at 1 (448 * 1 / 448)
    scales[20, 3] = e4m3[448.0]
    outer = np.ones(1, np.float32)
    assert ex["forward_code_value"] * ex["forward_scale"] == ex["forward_dequant"]
    c, s, g = oracle.requant_transpose_nvfp4(codes, scales, outer, False, 1, rows, cols, 0, 9, stochastic=False)
    assert g[0] == 1.0 and oracle.e4m3_value(s[0, 0, 0]) == ex["backward_scale"]
    assert e2m1_value(unpack(c)[0, 0, 0]) * 2.0 == ex["rn_value"] * 2.0   # 2.25 -> 2 by nearest
    assert e2m1_value(unpack(c)[0, 0, 1]) == 6.0                          # 12 / 2 = 6, exactly
    ups, n = 0, 4000
    vals = []
    for seed in range(n):
        c, s, g = oracle.requant_transpose_nvfp4(codes, scales, outer, False, 1, rows, cols, seed, 9)
        v = e2m1_value(unpack(c)[0, 0, 0])
        assert v in ex["sr_values"]
        ups += v == 3.0
        vals.append(v * oracle.e4m3_value(s[0, 0, 0]) * g[0])
    p = ups / n
    assert abs(p - ex["sr_probabilities"][1]) < 0.03, p
    assert abs(np.mean(vals) - ex["expected_dequant"]) < 0.07


def brute_force_rn(codes, scales, outer, per_row, batch, rows, cols):
    """Round-to-nearest requantisation written from the definition, with the
    block scale and the codes found by scanning the E4M3 and E2M1 grids."""
    grid = e4m3_grid()
    cds = codes.reshape(batch, rows, cols // 2)
    scs = scales.reshape(batch, rows, cols // 16)
    out_c = np.zeros((batch, cols, rows), np.uint8)
    out_s = np.zeros((batch, cols, rows // 16), np.uint8)
    out_g = np.zeros(batch, np.float32)
    for b in range(batch):
        g = (outer.reshape(batch, rows)[b] if per_row else np.full(rows, outer[b])).astype(np.float32)
        sd = np.vectorize(oracle.e4m3_value)(scs[b]).astype(np.float32) * g[:, None]
        m = np.float32(sd.max())
        gp = np.float32(1.0) if m == 0 else np.float32(m / np.float32(448.0))
        out_g[b] = gp
        cs = unpack(cds[b])
        dv = (np.vectorize(e2m1_value)(cs) * np.repeat(np.vectorize(oracle.e4m3_value)(scs[b]), 16, axis=1))
        d = (dv.astype(np.float32) * g[:, None]).astype(np.float32).T        # [cols, rows], binary32
        for c in range(cols):
            for rb in range(rows // 16):
                blk = d[c, rb * 16:(rb + 1) * 16]
                s = np.float32(np.abs(blk).max()) / np.float32(np.float32(6.0) * gp)
                idx = int(np.searchsorted(grid, float(s), side="left")) if s <= 448 else 0x7E
                S = min(idx, 0x7E)
                sdp = np.float32(np.float32(grid[S]) * gp)
                r = np.float32(0.0) if sdp == 0 else np.float32(np.float32(1.0) / sdp)
                out_s[b, c, rb] = S
                for j in range(16):
                    y = np.float32(blk[j] * r)
                    a = abs(float(y))
                    dist = np.abs(E2M1 - a)
                    best = np.flatnonzero(dist == dist.min())
                    k = best[0] if len(best) == 1 else best[best % 2 == 0][0]  # ties to the even code
                    out_c[b, c, rb * 16 + j] = k | (8 if np.signbit(y) else 0)
    packed = (out_c[..., 0::2] | (out_c[..., 1::2] << 4)).astype(np.uint8)
    return packed, out_s, out_g


def random_nvfp4(rng, rows, cols, per_row, batch=1):
    x = (rng.standard_normal((batch * rows, cols)) * np.exp(rng.uniform(-3, 3, (batch * rows, 1)))).astype(np.float32)
    x[3] = 0.0                                  # a zero row (outer scale 1 when per row)
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)
    if per_row:
        return oracle.nvfp4_quantize(bits, oracle.OUTER_PER_ROW, four_over_six=True)
    return oracle.nvfp4_quantize(bits, oracle.OUTER_PER_GROUP, group_offsets=np.arange(batch + 1) * rows)


def test_requant_nvfp4_rn_brute_force():
    rng = np.random.default_rng(21)
    for per_row, batch in ((True, 1), (False, 2)):
        rows, cols = 64, 64
        c, s, g = random_nvfp4(rng, rows, cols, per_row, batch)
        got = oracle.requant_transpose_nvfp4(c, s, g, per_row, batch, rows, cols, 0, 6, stochastic=False)
        want = brute_force_rn(c, s, g, per_row, batch, rows, cols)
        for a, b in zip(got, want):
            assert np.array_equal(np.asarray(a), np.asarray(b))


def test_requant_nvfp4_sr_neighbours_and_mean():
    """Each stochastic code is one of the two E2M1 neighbours of the scaled
    value; the scale never lets a value clip; the mean over seeds decodes to
    the dequantised input."""
    rng = np.random.default_rng(22)
    rows, cols = 32, 64
    c, s, g = random_nvfp4(rng, rows, cols, True)
    rn_c, rn_s, rn_g = oracle.requant_transpose_nvfp4(c, s, g, True, 1, rows, cols, 0, 6, stochastic=False)
    d = decode_nvfp4(c.reshape(rows, cols // 2), s.reshape(rows, cols // 16), g[:, None]).T   # [cols, rows]
    acc = np.zeros((cols, rows))
    n = 300
    for seed in range(n):
        sc_, ss_, sg_ = oracle.requant_transpose_nvfp4(c, s, g, True, 1, rows, cols, seed, 6)
        assert np.array_equal(ss_, rn_s) and np.array_equal(sg_, rn_g)   # scales do not depend on the bits
        v = decode_nvfp4(sc_[0], ss_[0], sg_[0])
        y_scaled = d / np.repeat(np.vectorize(oracle.e4m3_value)(ss_[0]) * sg_[0], 16, axis=1).clip(1e-300)
        assert np.all(np.abs(y_scaled) <= 6.0 * (1 + 2.0 ** -20))
        acc += v
    mean = acc / n
    step = np.repeat(np.vectorize(oracle.e4m3_value)(rn_s[0]) * rn_g[0], 16, axis=1) * 2.0  # <= one E2M1 step
    # the mean of n draws is within 5 standard deviations (a step / (2 sqrt(n))) of the value
    assert np.all(np.abs(mean - d) <= 5 * step / (2 * np.sqrt(n)) + 1e-12)
