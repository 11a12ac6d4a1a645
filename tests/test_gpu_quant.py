"""GPU parity of the quantisation kernels against the CPU oracle (bit-exact).

Inputs come from the seeded generators; the oracle sees the same bf16 bytes.
Codes, scales, outer scales and MXFP8 / S2F6 bytes must match exactly.
"""
import numpy as np
import pytest
import torch

import oracle
from precision_moe_numerics_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pmn():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from precision_moe_numerics_gb300 import build, pmn as P
    build.build()
    return P


def to_dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def host(t):
    if t.dtype == torch.bfloat16:
        t = t.view(torch.int16)
    return t.cpu().numpy()


def assert_same(gpu, ref, what):
    g = host(gpu) if isinstance(gpu, torch.Tensor) else gpu
    if g.dtype == np.float32:
        g, ref = g.view(np.uint32), np.asarray(ref, np.float32).view(np.uint32)
    bad = np.argwhere(g != ref)
    assert bad.size == 0, "%s: %d mismatches, first at %s: gpu %s oracle %s" % (
        what, len(bad), bad[0], g[tuple(bad[0])], ref[tuple(bad[0])])


@pytest.mark.parametrize("fos", [False, True])
@pytest.mark.parametrize("shape", [(1, 16), (37, 48), (256, 256), (100, 1536), (64, 4096), (9, 8192)])
def test_nvfp4_quantize_per_row(pmn, shape, fos):
    rng = np.random.default_rng(hash(shape) % 1000)
    x = W.normal_bf16_host(rng, shape, 1.0, 0.01, 30.0)
    x[0, :16] = 0  # a zero block
    if shape[0] > 2:
        x[2] = 0  # a zero row
    c, s, g = pmn.nvfp4_quantize(to_dev_bf16(x), four_over_six=fos)
    rc, rs, rg = oracle.nvfp4_quantize(x, oracle.OUTER_PER_ROW, four_over_six=fos)
    assert_same(g, rg, "outer")
    assert_same(s, rs, "scales")
    assert_same(c, rc, "codes")


def test_nvfp4_quantize_tiny_case_per_tensor(pmn):
    d = W.tiny(0)
    c, s, g = pmn.nvfp4_quantize(to_dev_bf16(d["x"]), outer_mode=pmn.OUTER_PER_GROUP, rows_per_group=256)
    rc, rs, rg = oracle.nvfp4_quantize(d["x"], oracle.OUTER_PER_GROUP, group_offsets=[0, 256])
    assert_same(g, rg, "outer")
    assert_same(s, rs, "scales")
    assert_same(c, rc, "codes")


def test_nvfp4_quantize_per_expert_weights(pmn):
    rng = np.random.default_rng(3)
    E, N, K = 5, 96, 512
    w = W.normal_bf16_host(rng, (E * N, K), 0.02)
    w[N:2 * N] = 0  # an all-zero expert
    c, s, g = pmn.nvfp4_quantize(to_dev_bf16(w), outer_mode=pmn.OUTER_PER_GROUP, rows_per_group=N)
    rc, rs, rg = oracle.nvfp4_quantize(w, oracle.OUTER_PER_GROUP, group_offsets=np.arange(E + 1) * N)
    assert_same(g, rg, "outer")
    assert_same(s, rs, "scales")
    assert_same(c, rc, "codes")


def test_nvfp4_quantize_per_expert_multichunk(pmn):
    """Groups spanning several work chunks of 4096 blocks with a ragged last
    chunk; each expert's amax sits in a different chunk (first, middle, the
    partial last one), so every chunk's amax must reach the group's scale."""
    rng = np.random.default_rng(11)
    E, N, K = 3, 520, 1024  # 33280 blocks per expert: 8 full chunks + 512 blocks
    w = W.normal_bf16_host(rng, (E * N, K), 0.02)
    for e, r in enumerate((3, 260, N - 1)):
        w[e * N + r, 17] = W.f32_to_bf16_bits(np.array([-7.5], np.float32))[0]
    c, s, g = pmn.nvfp4_quantize(to_dev_bf16(w), outer_mode=pmn.OUTER_PER_GROUP, rows_per_group=N)
    rc, rs, rg = oracle.nvfp4_quantize(w, oracle.OUTER_PER_GROUP, group_offsets=np.arange(E + 1) * N)
    assert_same(g, rg, "outer")
    assert_same(s, rs, "scales")
    assert_same(c, rc, "codes")
    assert pmn.get_device_error() == 0


def test_nvfp4_block_scale_rounding_boundaries(pmn):
    """Block amax values sweep every bf16 pattern from 2^-8 to 2^8, with outer
    scales chosen so that m * g is a power of two: amax / (m g) then lands
    exactly on E4M3 rounding midpoints (ties) and next to them, where the
    block scale's quotient must be the correctly rounded one."""
    rng = np.random.default_rng(17)
    v = np.arange(0x3B80, 0x4380, dtype=np.uint16)  # 2048 bf16 patterns
    amax = W.bf16_bits_to_f32(v)
    x = amax[:, None] * rng.uniform(-1.0, 1.0, (len(v), 16)).astype(np.float32)
    x[:, 0] = amax * np.where(rng.random(len(v)) < 0.5, -1.0, 1.0)
    x = W.f32_to_bf16_bits(x.reshape(16, 2048).astype(np.float32))
    x[:, 0] = W.f32_to_bf16_bits(np.array([448.0], np.float32))[0]  # group / row amax 448
    # per group: g = 448 / 2688, 6 g = 1
    c, s, g = pmn.nvfp4_quantize(to_dev_bf16(x), outer_mode=pmn.OUTER_PER_GROUP, rows_per_group=16)
    rc, rs, rg = oracle.nvfp4_quantize(x, oracle.OUTER_PER_GROUP, group_offsets=[0, 16])
    assert_same(g, rg, "outer")
    assert_same(s, rs, "scales")
    assert_same(c, rc, "codes")
    # per row with 4/6: g = 448 / 1792, 4 g = 1 and 6 g = 1.5
    c, s, g = pmn.nvfp4_quantize(to_dev_bf16(x), four_over_six=True)
    rc, rs, rg = oracle.nvfp4_quantize(x, oracle.OUTER_PER_ROW, four_over_six=True)
    assert_same(g, rg, "outer")
    assert_same(s, rs, "scales")
    assert_same(c, rc, "codes")


def test_nvfp4_quantize_expert_case_activations(pmn):
    d = W.expert(0, tokens=512)
    c, s, g = pmn.nvfp4_quantize(to_dev_bf16(d["x"]), four_over_six=True)
    rc, rs, rg = oracle.nvfp4_quantize(d["x"], oracle.OUTER_PER_ROW, four_over_six=True)
    assert_same(g, rg, "outer")
    assert_same(s, rs, "scales")
    assert_same(c, rc, "codes")


def test_nvfp4_quantize_swiglu(pmn):
    """h = silu(gate) * up (glue between w1 and w2), the SwiGLU input mode.
    The GPU forms h with expf in binary32: h must be within one bf16 step of
    the binary64 value on every element, and on every row the codes, scales
    and outer scale must equal, byte for byte, those of the plain per-row
    quantiser run on the kernel's own h (that quantiser is pinned to the
    oracle by test_nvfp4_quantize_per_row)."""
    rng = np.random.default_rng(5)
    rows, f = 64, 1536
    y = W.normal_bf16_host(rng, (rows, 2 * f), 0.5)
    c, s, g, h = pmn.nvfp4_quantize(to_dev_bf16(y), cols=f, swiglu=True, four_over_six=True, want_h=True)
    rh = oracle.swiglu_bf16(y, f)
    hg = host(h).view(np.uint16)
    hf, rf = W.bf16_bits_to_f32(hg).astype(np.float64), W.bf16_bits_to_f32(rh).astype(np.float64)
    assert np.all(np.abs(hf - rf) <= np.abs(rf) * 2.0 ** -7 + 1e-30)
    pc, ps, pg = pmn.nvfp4_quantize(h, four_over_six=True)
    assert_same(c, host(pc), "codes")
    assert_same(s, host(ps), "scales")
    assert_same(g, host(pg), "outer")
    c2, s2, g2 = pmn.nvfp4_quantize(to_dev_bf16(y), cols=f, swiglu=True, four_over_six=True)  # without h
    assert torch.equal(c, c2) and torch.equal(s, s2) and torch.equal(g, g2)


@pytest.mark.parametrize("shape", [(32, 32), (96, 256), (256, 4096), (4096, 64)])
def test_mxfp8_quantize_rowwise(pmn, shape):
    rng = np.random.default_rng(7)
    x = W.normal_bf16_host(rng, shape, 1e-3, 0.01, 50.0)
    x[0, :32] = 0
    q, sc = pmn.mxfp8_quantize(to_dev_bf16(x), transpose=False)
    rq, rsc = oracle.mxfp8_quantize(x, transpose=False)
    assert_same(sc, rsc, "scales")
    assert_same(q, rq, "values")


@pytest.mark.parametrize("shape", [(32, 32), (96, 256), (256, 4096), (4096, 72)])
def test_mxfp8_quantize_transposed(pmn, shape):
    rng = np.random.default_rng(8)
    x = W.normal_bf16_host(rng, shape, 1e-3, 0.01, 50.0)
    q, sc = pmn.mxfp8_quantize(to_dev_bf16(x), transpose=True)
    rq, rsc = oracle.mxfp8_quantize(x, transpose=True)
    assert_same(sc, rsc, "scales")
    assert_same(q, rq, "values")


@pytest.mark.parametrize("shape", [(32, 32), (256, 256), (160, 1536), (224, 96), (96, 4096), (384, 3072)])
def test_mxfp8_quantize_both(pmn, shape):
    """both orientations in one pass: the bytes of the oracle's rowwise and
    transposed MXFP8, and of the two separate library calls (partial tiles in
    both directions included)"""
    rng = np.random.default_rng(shape[0] + shape[1])
    x = W.normal_bf16_host(rng, shape, 1e-3, 0.01, 50.0)
    x[3, :] = 0  # an all-zero row and column block
    x[:, 5] = 0
    xd = to_dev_bf16(x)
    (q, sc), (qt, sct) = pmn.mxfp8_quantize_both(xd)
    rq, rsc = oracle.mxfp8_quantize(x, transpose=False)
    rqt, rsct = oracle.mxfp8_quantize(x, transpose=True)
    assert_same(sc, rsc, "row scales")
    assert_same(q, rq, "row values")
    assert_same(sct, rsct, "column scales")
    assert_same(qt, rqt, "column values")
    q2, sc2 = pmn.mxfp8_quantize(xd, transpose=False)
    qt2, sct2 = pmn.mxfp8_quantize(xd, transpose=True)
    for a, b in [(q, q2), (sc, sc2), (qt, qt2), (sct, sct2)]:
        assert torch.equal(a, b)


def test_mxfp8_extreme_blocks(pmn):
    """MXFP8 at the ends of the bf16 range, in both orientations and through
    the one-pass call: blocks of bf16 subnormals (the E8M0 exponent clamps at
    -127), blocks near the largest bf16, blocks whose amax is exactly
    448 * 2^k (scale 2^k) or one bf16 step above it (2^(k+1)), one huge value
    among tiny ones of both signs (negative values that round to zero keep
    their sign bit), and a column block of subnormals."""
    rng = np.random.default_rng(11)
    rows, cols = 96, 256
    x = W.normal_bf16_host(rng, (rows, cols), 1.0, 0.01, 20.0)
    sign = lambda n: (rng.integers(0, 2, n, dtype=np.uint16) << 15)
    x[0] = rng.integers(1, 0x80, cols, dtype=np.uint16) | sign(cols)          # subnormals
    x[1] = rng.integers(0x7F00, 0x7F80, cols, dtype=np.uint16) | sign(cols)   # near the largest bf16
    ks = []
    for b in range(cols // 32):                                               # amax at 448 * 2^k, or just above
        k = int(rng.integers(-20, 20))
        ks.append(k)
        top = np.float32(448.0 * 2.0 ** k).view(np.uint32) >> 16
        x[2, 32 * b:32 * b + 32] = (top - rng.integers(0x80, 0x800, 32)).astype(np.uint16) | sign(32)  # below top
        x[2, 32 * b + int(rng.integers(0, 32))] = np.uint16(top + (b & 1)) | np.uint16(0x8000 * (b >> 2 & 1))
    x[3] = rng.integers(0x0080, 0x0400, cols, dtype=np.uint16) | sign(cols)   # tiny normals ...
    x[3, ::32] = 0x7E00                                                       # ... under a huge value
    x[32:64, 64:96] = rng.integers(1, 0x80, (32, 32), dtype=np.uint16) | (
        rng.integers(0, 2, (32, 32), dtype=np.uint16) << 15)                  # a column block of subnormals
    xd = to_dev_bf16(x)
    rq, rsc = oracle.mxfp8_quantize(x, transpose=False)
    rqt, rsct = oracle.mxfp8_quantize(x, transpose=True)
    # the clamp, the planted block maxima and the negative zeros are exercised
    assert rsc[0].max() == 0 and (rq[3] == 0x80).any()
    assert np.array_equal(rsc[2].astype(int) - 127, [k + (b & 1) for b, k in enumerate(ks)])
    (q, sc), (qt, sct) = pmn.mxfp8_quantize_both(xd)
    q1, sc1 = pmn.mxfp8_quantize(xd, transpose=False)
    qt1, sct1 = pmn.mxfp8_quantize(xd, transpose=True)
    for got, want, what in [(q, rq, "row values"), (sc, rsc, "row scales"), (qt, rqt, "column values"),
                            (sct, rsct, "column scales"), (q1, rq, "rowwise call values"),
                            (sc1, rsc, "rowwise call scales"), (qt1, rqt, "transposed call values"),
                            (sct1, rsct, "transposed call scales")]:
        assert_same(got, want, what)


@pytest.mark.parametrize("stochastic", [True, False])
@pytest.mark.parametrize("batch,rows,cols,per_row", [(1, 32, 64, True), (1, 256, 256, True), (1, 160, 1536, True),
                                                     (3, 96, 128, False), (2, 512, 192, False)])
def test_requant_transpose(pmn, batch, rows, cols, per_row, stochastic):
    rng = np.random.default_rng(rows + cols)
    x = W.normal_bf16_host(rng, (batch * rows, cols), 1.0, 0.02, 30.0)
    x[:32] = 0  # a padding segment
    if per_row:
        c, s, g = oracle.nvfp4_quantize(x, oracle.OUTER_PER_ROW, four_over_six=True)
    else:
        c, s, g = oracle.nvfp4_quantize(x, oracle.OUTER_PER_GROUP, group_offsets=np.arange(batch + 1) * rows)
    seed, tag = 1234567, 2
    dc, ds, dg = (torch.from_numpy(a).cuda() for a in (c, s, g))
    q, qs = pmn.requant_transpose_sr_mxfp8(dc, ds, dg, per_row, batch, rows, cols, seed, tag, stochastic)
    rq, rqs = oracle.requant_transpose_mxfp8(c, s, g, per_row, batch, rows, cols, seed, tag, stochastic)
    assert_same(qs, rqs, "scales")
    assert_same(q, rq, "values")


def test_requant_gpu_chain_from_gpu_quantize(pmn):
    """GPU quantise then GPU requant equals the oracle chain on the same input."""
    d = W.tiny(0)
    c, s, g = pmn.nvfp4_quantize(to_dev_bf16(d["x"]), outer_mode=pmn.OUTER_PER_GROUP, rows_per_group=256)
    q, qs = pmn.requant_transpose_sr_mxfp8(c, s, g, False, 1, 256, 256, 0, 1)
    rc, rs, rg = oracle.nvfp4_quantize(d["x"], oracle.OUTER_PER_GROUP, group_offsets=[0, 256])
    rq, rqs = oracle.requant_transpose_mxfp8(rc, rs, rg, False, 1, 256, 256, 0, 1)
    assert_same(qs, rqs, "scales")
    assert_same(q, rq, "values")


@pytest.mark.parametrize("shape", [(1, 32), (64, 256), (300, 4096)])
def test_rht_s2f6_quantize(pmn, shape):
    rng = np.random.default_rng(11)
    x = (rng.standard_normal(shape) * 10.0 ** rng.uniform(-3, 2, (shape[0], 1))).astype(np.float32)
    x[0, :32] = 0
    for seed in (0, 99):
        q, sc = pmn.rht_s2f6_quantize(torch.from_numpy(x).cuda(), seed)
        rq, rsc = oracle.rht_s2f6(x, seed)
        assert_same(sc, rsc, "scales")
        assert_same(q, rq, "codes")


def test_rht_s2f6_extreme_blocks(pmn):
    """Blocks whose exponent needs the 2^64 pre-scale (amax below 2^-121, down
    into float32 subnormals) and blocks with an infinite value (the clamped
    exponent 127 and its general path; one infinity per block spreads through
    the butterflies without meeting another, so no NaN arises)."""
    rng = np.random.default_rng(13)
    rows = [rng.standard_normal(64) * 2.0 ** (-100 - r) for r in range(48)]
    inf_row = rng.standard_normal(64)
    inf_row[5], inf_row[40] = np.inf, -np.inf
    rows += [inf_row, rng.standard_normal(64)]
    x = np.stack(rows).astype(np.float32)
    for seed in (0, 7):
        q, sc = pmn.rht_s2f6_quantize(torch.from_numpy(x).cuda(), seed)
        rq, rsc = oracle.rht_s2f6(x, seed)
        assert_same(sc, rsc, "scales")
        assert_same(q, rq, "codes")
    assert (rsc[:48] < 127 - 121).any() and (rsc[48] == 254).all()  # both branches taken


def test_quantize_deterministic(pmn):
    rng = np.random.default_rng(12)
    x = to_dev_bf16(W.normal_bf16_host(rng, (512, 4096)))
    a = [pmn.nvfp4_quantize(x, four_over_six=True) for _ in range(3)]
    for t in a[1:]:
        for u, v in zip(a[0], t):
            assert torch.equal(u, v)


def test_invalid_arguments_rejected(pmn):
    x = torch.zeros((4, 24), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pmn.PmnError):
        pmn.nvfp4_quantize(x)  # cols % 16 != 0
    y = torch.zeros((40, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pmn.PmnError):
        pmn.mxfp8_quantize(y, transpose=True)  # rows % 32 != 0
    c = torch.zeros((32, 16), dtype=torch.uint8, device="cuda")
    s = torch.zeros((32, 2), dtype=torch.uint8, device="cuda")
    g = torch.ones(32, dtype=torch.float32, device="cuda")
    with pytest.raises(pmn.PmnError):
        pmn.requant_transpose_sr_mxfp8(c, s, g, True, 1, 32, 32, 0, 1)  # cols % 64 != 0
