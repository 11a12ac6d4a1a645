"""GPU parity of the block-scaled GEMMs against the binary64 oracle.

Tolerances (stated for the expert-layer path): float32 outputs within
relative Frobenius error 1e-5 and elementwise |err| <= 1e-3 * (|A| |B|)[m, n]
(outer scales included); bf16 outputs additionally within one bf16 step
(2^-8 relative) of the binary64 value.  The fused RHT + S2F6 epilogue is
checked two ways: its input (the scaled fp32 accumulator, read back through
the optional debug output) within the float32 tolerance of the binary64
product, and its bytes equal to those of the library's standalone combine
quantisation kernel run on that same input (which test_gpu_quant pins byte
for byte to the oracle on seeded inputs; the oracle itself never takes an
input from the CUDA path); also after decoding, against the oracle's combine
quantisation of the binary64 product (codes within one step, scales equal
except where the block maximum sits on a power-of-two boundary).
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


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def check_f32(got, ref, absab, what):
    got = np.asarray(got, np.float64)
    err = np.abs(got - ref)
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    assert rel <= 1e-5, "%s: relative Frobenius error %.3e" % (what, rel)
    bad = err > 1e-3 * absab + 1e-30
    assert not bad.any(), "%s: %d elements beyond 1e-3 |A||B|" % (what, bad.sum())


def check_bf16(got_bf16, ref, absab, what):
    g = W.bf16_bits_to_f32(got_bf16.view(np.uint16)).astype(np.float64)
    bad = np.abs(g - ref) > np.abs(ref) * 2.0 ** -8 + 1e-3 * absab + 1e-30
    assert not bad.any(), "%s: %d elements beyond one bf16 step" % (what, bad.sum())


def moe_case(seed=0, tokens=256, experts=8, k=2, d=512, f=256, pad=W.PAD):
    m = W.small_moe(seed, tokens=tokens, experts=experts, k=k, d=d, f=f, pad=pad)
    r = m["routing"]
    xa = oracle.nvfp4_quantize(m["x"], oracle.OUTER_PER_ROW, four_over_six=True)
    E = experts
    w1 = m["w1"].reshape(E * 2 * f, d)
    w1q = oracle.nvfp4_quantize(w1, oracle.OUTER_PER_GROUP, group_offsets=np.arange(E + 1) * 2 * f)
    w1q = (w1q[0].reshape(E, 2 * f, d // 2), w1q[1].reshape(E, 2 * f, d // 16), w1q[2])
    return m, r, xa, w1q


def abs_product(a_codes, a_scales, a_outer, b_codes, b_scales, b_outer, offsets):
    """(|A| |B|)[m, n] with the outer scales (binary64), per expert."""
    out = np.zeros((a_codes.shape[0], b_codes.shape[1]))
    for e in range(len(offsets) - 1):
        lo, hi = offsets[e], offsets[e + 1]
        if hi == lo:
            continue
        A = np.abs(oracle.nvfp4_dequant_f64(a_codes[lo:hi], a_scales[lo:hi]))
        B = np.abs(oracle.nvfp4_dequant_f64(b_codes[e], b_scales[e]))
        out[lo:hi] = (A @ B.T) * np.abs(a_outer[lo:hi, None].astype(np.float64)) * abs(float(b_outer[e]))
    return out


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_grouped_gemm_nvfp4_small_moe(pmn, out_dtype):
    m, r, (ac, asc, ag), (bc, bsc, bg) = moe_case()
    offs = r.offsets.astype(np.int32)
    out = pmn.grouped_gemm_nvfp4((dev(ac), dev(asc), dev(ag)), (dev(bc), dev(bsc), dev(bg)), dev(offs),
                                 out_dtype=out_dtype)
    ref = oracle.grouped_gemm_nvfp4(ac, asc, ag, bc, bsc, bg, r.offsets)
    absab = abs_product(ac, asc, ag, bc, bsc, bg, r.offsets)
    got = out.cpu()
    if out_dtype == torch.float32:
        check_f32(got.numpy(), ref, absab, "grouped nvfp4 f32")
    else:
        check_bf16(got.view(torch.int16).numpy(), ref, absab, "grouped nvfp4 bf16")


def test_nvfp4_gemm_tiny_case(pmn):
    """256 x 256 x 256 NVFP4 x NVFP4 with float32 accumulation (single group)."""
    d = W.tiny(0)
    a = oracle.nvfp4_quantize(d["x"], oracle.OUTER_PER_GROUP, group_offsets=[0, 256])
    b = oracle.nvfp4_quantize(d["b"], oracle.OUTER_PER_GROUP, group_offsets=[0, 256])
    ag = np.full(256, a[2][0], np.float32)
    offs = np.array([0, 256], np.int32)
    out = pmn.grouped_gemm_nvfp4((dev(a[0]), dev(a[1]), dev(ag)),
                                 (dev(b[0][None]), dev(b[1][None]), dev(b[2])), dev(offs), out_dtype=torch.float32)
    ref = oracle.gemm_nvfp4(a[0], a[1], ag, b[0], b[1], b[2][0])
    absab = abs_product(a[0], a[1], ag, b[0][None], b[1][None], b[2], [0, 256])
    check_f32(out.cpu().numpy(), ref, absab, "tiny gemm")


def test_grouped_gemm_nvfp4_edge_offsets(pmn):
    """empty experts, a 1-row expert, ragged tails, rows not a multiple of 32."""
    rng = np.random.default_rng(4)
    K, N, E = 512, 256, 6
    counts = [0, 1, 129, 0, 31, 300]
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    T = int(offs[-1])
    x = W.normal_bf16_host(rng, (T, K))
    w = W.normal_bf16_host(rng, (E * N, K), 0.02)
    ac, asc, ag = oracle.nvfp4_quantize(x, oracle.OUTER_PER_ROW)
    bq = oracle.nvfp4_quantize(w, oracle.OUTER_PER_GROUP, group_offsets=np.arange(E + 1) * N)
    bc, bsc, bg = bq[0].reshape(E, N, K // 2), bq[1].reshape(E, N, K // 16), bq[2]
    out = pmn.grouped_gemm_nvfp4((dev(ac), dev(asc), dev(ag)), (dev(bc), dev(bsc), dev(bg)), dev(offs),
                                 out_dtype=torch.float32)
    ref = oracle.grouped_gemm_nvfp4(ac, asc, ag, bc, bsc, bg, offs)
    absab = abs_product(ac, asc, ag, bc, bsc, bg, offs)
    check_f32(out.cpu().numpy(), ref, absab, "edge offsets")


def test_grouped_nvfp4_gemm_short_segments(pmn):
    """16 or fewer rows per expert on average (the library's 32-row tiles):
    empty experts, segments of 1..5 rows, and 33- and 70-row segments that
    span several 32-row tiles; fp32 and bf16 outputs"""
    rng = np.random.default_rng(44)
    n, k = 512, 256
    counts = np.array([1, 2, 0, 70, 3, 0, 5, 1, 0, 2, 33, 4])
    E = len(counts)
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    T = int(offs[-1])
    assert T <= 16 * E
    a = oracle.nvfp4_quantize(W.normal_bf16_host(rng, (T, k), 1.0, 0.01, 30.0), oracle.OUTER_PER_ROW,
                              four_over_six=True)
    bq = oracle.nvfp4_quantize(W.normal_bf16_host(rng, (E * n, k), 0.02), oracle.OUTER_PER_GROUP,
                               group_offsets=np.arange(E + 1) * n)
    bc, bsc, bg = bq[0].reshape(E, n, k // 2), bq[1].reshape(E, n, k // 16), bq[2]
    ref = oracle.grouped_gemm_nvfp4(*a, bc, bsc, bg, offs)
    absab = abs_product(*a, bc, bsc, bg, offs)
    A, B = tuple(dev(t) for t in a), (dev(bc), dev(bsc), dev(bg))
    out = pmn.grouped_gemm_nvfp4(A, B, dev(offs), out_dtype=torch.float32)
    check_f32(out.cpu().numpy(), ref, absab, "short segments, fp32")
    outb = pmn.grouped_gemm_nvfp4(A, B, dev(offs), out_dtype=torch.bfloat16)
    check_bf16(outb.view(torch.int16).cpu().numpy(), ref, absab, "short segments, bf16")


@pytest.mark.parametrize("tokens,pad", [(256, W.PAD), (16, 1)])
def test_w2_gemm_rht_s2f6(pmn, tokens, pad):
    """128-row expert segments (128-wide tiles), and a decode-like batch of
    unpadded segments of a few rows (the library then takes 256-wide tiles)."""
    m, r, (ac, asc, ag), _ = moe_case(tokens=tokens, pad=pad)
    E, d, f = 8, 512, 256
    w2 = m["w2"].reshape(E * d, f)
    hq = oracle.nvfp4_quantize(W.normal_bf16_host(np.random.default_rng(9), (r.rows, f)), oracle.OUTER_PER_ROW,
                               four_over_six=True)
    w2q = oracle.nvfp4_quantize(w2, oracle.OUTER_PER_GROUP, group_offsets=np.arange(E + 1) * d)
    bc, bsc, bg = w2q[0].reshape(E, d, f // 2), w2q[1].reshape(E, d, f // 16), w2q[2]
    offs = r.offsets.astype(np.int32)
    seed = 42
    acc = torch.zeros((r.rows, d), dtype=torch.float32, device="cuda")
    q, sc = pmn.w2_gemm_rht_s2f6((dev(hq[0]), dev(hq[1]), dev(hq[2])), (dev(bc), dev(bsc), dev(bg)), dev(offs),
                                 seed, debug_acc=acc)
    sq, ssc = pmn.rht_s2f6_quantize(acc, seed)  # the standalone epilogue kernel on the same input
    z = oracle.grouped_gemm_nvfp4(hq[0], hq[1], hq[2], bc, bsc, bg, r.offsets)
    q, sc, accn = q.cpu().numpy(), sc.cpu().numpy(), acc.cpu().numpy()
    # the epilogue's input is the GEMM result within the float32 tolerance ...
    check_f32(accn, z, abs_product(hq[0], hq[1], hq[2], bc, bsc, bg, r.offsets), "w2 accumulator")
    # ... and the fused epilogue's bytes are the standalone kernel's on exactly that input
    assert np.array_equal(sc, ssc.cpu().numpy()), "fused S2F6 scales differ from the standalone kernel's"
    assert np.array_equal(q, sq.cpu().numpy()), "fused S2F6 codes differ from the standalone kernel's"
    rq, rsc = oracle.rht_s2f6(z.astype(np.float32), seed)
    same_e = sc == rsc
    assert same_e.mean() > 0.99
    dq = np.abs(q.astype(np.int32) - rq.astype(np.int32)).reshape(q.shape[0], -1, 32)
    assert np.all(dq[same_e] <= 1)
    # decoded values agree everywhere within one code step of the coarser scale
    dec = oracle.s2f6_dequant_inverse_rht(q, sc, seed)
    rdec = oracle.s2f6_dequant_inverse_rht(rq, rsc, seed)
    step = np.repeat(np.maximum(2.0 ** (sc.astype(np.float64) - 127), 2.0 ** (rsc.astype(np.float64) - 127)) / 64,
                     32, axis=1)
    assert np.all(np.abs(dec - rdec) <= 32 * step)


def mx_case(rng, rows, cols, std=1e-3):
    x = W.normal_bf16_host(rng, (rows, cols), std, 0.01, 20.0)
    return oracle.mxfp8_quantize(x, transpose=False)


def check_mx(got, ref, absab, what):
    check_f32(got, ref, absab, what)


@pytest.mark.parametrize("K,N,out_dtype", [(1024, 256, torch.float32), (3072, 512, torch.bfloat16),
                                           (512, 256, torch.bfloat16), (1536, 128, torch.float32)])
def test_gemm_mxfp8_mgrouped(pmn, K, N, out_dtype):
    """M-grouped MXFP8 (the dX / dH form) against the oracle: ragged, empty
    and one-row segments; one to six groups of four 128-wide K steps (the
    256-wide tiles' scale rows cover four steps each); one or two 256-wide
    column tiles, or 128-wide tiles; fp32 and bf16 outputs."""
    rng = np.random.default_rng(21 + K + N)
    counts = [64, 0, 200, 32, 1]
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    G, M = len(counts), int(offs[-1])
    a, asc = mx_case(rng, M, K)
    b, bsc = mx_case(rng, G * N, K, 0.02)
    b, bsc = b.reshape(G, N, K), bsc.reshape(G, N, K // 32)
    out = pmn.gemm_mxfp8(dev(a), dev(asc), dev(b), dev(bsc), dev(offs), pmn.GROUP_M, out_dtype)
    ref = oracle.gemm_mxfp8_mgrouped(a, asc, b, bsc, offs)
    absab = np.zeros_like(ref)
    for g in range(G):
        lo, hi = offs[g], offs[g + 1]
        if hi > lo:
            absab[lo:hi] = np.abs(oracle.mxfp8_dequant_f64(a[lo:hi], asc[lo:hi])) @ np.abs(
                oracle.mxfp8_dequant_f64(b[g], bsc[g])).T
    if out_dtype == torch.float32:
        check_mx(out.cpu().numpy(), ref, absab, "mxfp8 M-grouped")
    else:
        check_bf16(out.view(torch.int16).cpu().numpy(), ref, absab, "mxfp8 M-grouped bf16")


def test_gemm_mxfp8_kgrouped(pmn):
    rng = np.random.default_rng(22)
    M, N, Kt = 256, 128, 1024
    offs = np.array([0, 128, 128, 512, 640, 1024], np.int32)  # an empty group, ragged (multiples of 128)
    G = len(offs) - 1
    a, asc = oracle.mxfp8_quantize(W.normal_bf16_host(rng, (Kt, M), 1e-3), transpose=True)
    b, bsc = oracle.mxfp8_quantize(W.normal_bf16_host(rng, (Kt, N), 1.0), transpose=True)
    out = pmn.gemm_mxfp8(dev(a), dev(asc), dev(b), dev(bsc), dev(offs), pmn.GROUP_K, torch.float32).cpu().numpy()
    ref = oracle.gemm_mxfp8_kgrouped(a, asc, b, bsc, offs)
    for g in range(G):
        lo, hi = offs[g], offs[g + 1]
        if hi == lo:
            assert np.all(out[g] == 0)
            continue
        absab = np.abs(oracle.mxfp8_dequant_f64(a[:, lo:hi], asc[:, lo // 32:hi // 32])) @ np.abs(
            oracle.mxfp8_dequant_f64(b[:, lo:hi], bsc[:, lo // 32:hi // 32])).T
        check_mx(out[g], ref[g], absab, "mxfp8 K-grouped g=%d" % g)


@pytest.mark.parametrize("M,N", [(256, 512), (128, 1536)])
def test_gemm_mxfp8_kgrouped_wide_tiles(pmn, M, N):
    """K-grouped with N a multiple of 256: the 256-wide tiles with eight
    epilogue warps (each holding half a row of the accumulator); an empty
    group, segments of one, four and six 128-row stages."""
    rng = np.random.default_rng(24 + N)
    offs = np.array([0, 128, 128, 640, 768, 1536], np.int32)
    G, Kt = len(offs) - 1, int(offs[-1])
    a, asc = oracle.mxfp8_quantize(W.normal_bf16_host(rng, (Kt, M), 1e-3, 0.01, 20.0), transpose=True)
    b, bsc = oracle.mxfp8_quantize(W.normal_bf16_host(rng, (Kt, N), 1.0), transpose=True)
    out = pmn.gemm_mxfp8(dev(a), dev(asc), dev(b), dev(bsc), dev(offs), pmn.GROUP_K, torch.float32).cpu().numpy()
    assert pmn.get_device_error() == 0
    ref = oracle.gemm_mxfp8_kgrouped(a, asc, b, bsc, offs)
    for g in range(G):
        lo, hi = offs[g], offs[g + 1]
        if hi == lo:
            assert np.all(out[g] == 0)
            continue
        absab = np.abs(oracle.mxfp8_dequant_f64(a[:, lo:hi], asc[:, lo // 32:hi // 32])) @ np.abs(
            oracle.mxfp8_dequant_f64(b[:, lo:hi], bsc[:, lo // 32:hi // 32])).T
        check_mx(out[g], ref[g], absab, "mxfp8 K-grouped wide g=%d" % g)


def test_gemm_mxfp8_kgrouped_rejects_unaligned_segments(pmn):
    """K segments must start on 128-row boundaries; a 32-aligned one runs no
    tile and latches the bad-offsets bit (checked on the device)."""
    rng = np.random.default_rng(23)
    M, N, Kt = 128, 128, 512
    offs = np.array([0, 96, 512], np.int32)
    a, asc = oracle.mxfp8_quantize(W.normal_bf16_host(rng, (Kt, M), 1e-3), transpose=True)
    b, bsc = oracle.mxfp8_quantize(W.normal_bf16_host(rng, (Kt, N), 1.0), transpose=True)
    pmn.gemm_mxfp8(dev(a), dev(asc), dev(b), dev(bsc), dev(offs), pmn.GROUP_K, torch.float32)
    torch.cuda.synchronize()
    assert pmn.get_device_error() == pmn.DEVERR_BAD_OFFSETS
    assert pmn.get_device_error() == 0  # read and cleared


def test_gemm_deterministic(pmn):
    m, r, (ac, asc, ag), (bc, bsc, bg) = moe_case(seed=3)
    offs = dev(r.offsets.astype(np.int32))
    A = (dev(ac), dev(asc), dev(ag))
    B = (dev(bc), dev(bsc), dev(bg))
    outs = [pmn.grouped_gemm_nvfp4(A, B, offs, out_dtype=torch.float32) for _ in range(3)]
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    assert pmn.get_device_error() == 0
