"""Failure handling and output bounds on the GPU, in forms that fault, trap or
hang nothing.

Bounded waits.  Every device wait of the library gives up after a wall-time
limit (pmn_set_wait_limit_ns), latches PMN_DEVERR_WAIT_TIMEOUT in the device
error word and lets its kernel return.  pmn_wait_selftest waits on an
mbarrier that nothing arrives on and on a counter that nothing increments,
with the primitives the GEMMs and the weight quantiser use: the latch must be
set, read once and cleared, and the context must stay usable.  The per-expert
weight quantiser is then run with a zero limit (a coding item gives up at
once when its group's amax is not yet complete): the call returns, the only
bit it may latch is the timeout, and the next call with the default limit is
byte-exact against the oracle.

Guard bytes.  Each output buffer of a representative call of every kernel
family sits between 256-byte guards; the guards must be untouched after the
call, and the output must come out the same whether the buffer was prefilled
with 0xAB or with 0x00, so every output byte was written.  (compute-sanitizer
is not available on this machine; these checks stand in for its memcheck on the
outputs.)
"""
import numpy as np
import pytest
import torch

import oracle
from precision_moe_numerics_gb300 import workloads as W

pytestmark = pytest.mark.gpu

GUARD = 256


@pytest.fixture(scope="module")
def P():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from precision_moe_numerics_gb300 import build, pmn
    build.build()
    return pmn


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def dev_bf16(bits):
    return dev(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def test_wait_selftest_latches_and_returns(P):
    assert P.get_device_error() == 0
    P.wait_selftest(2_000_000)  # 2 ms per wait
    torch.cuda.synchronize()
    assert P.get_device_error() == P.DEVERR_WAIT_TIMEOUT
    assert P.get_device_error() == 0  # read and cleared
    # the context is still usable: a quantisation afterwards is byte-exact
    x = W.normal_bf16_host(np.random.default_rng(1), (64, 256))
    c, s, g = P.nvfp4_quantize(dev_bf16(x), four_over_six=True)
    rc, rs, rg = oracle.nvfp4_quantize(x, oracle.OUTER_PER_ROW, four_over_six=True)
    assert np.array_equal(c.cpu().numpy(), rc) and np.array_equal(s.cpu().numpy(), rs)


def test_weight_quantiser_with_a_zero_wait_limit(P):
    rng = np.random.default_rng(2)
    E, N, K = 2, 2080, 1024  # 133120 blocks per expert: 65 work items each
    w = W.normal_bf16_host(rng, (E * N, K), 0.02)
    x = dev_bf16(w)
    prev = P.set_wait_limit_ns(0)
    try:
        P.nvfp4_quantize(x, outer_mode=P.OUTER_PER_GROUP, rows_per_group=N)
        torch.cuda.synchronize()
        err = P.get_device_error()
    finally:
        P.set_wait_limit_ns(prev)
    assert err in (0, P.DEVERR_WAIT_TIMEOUT), err
    c, s, g = P.nvfp4_quantize(x, outer_mode=P.OUTER_PER_GROUP, rows_per_group=N)
    torch.cuda.synchronize()
    assert P.get_device_error() == 0
    rc, rs, rg = oracle.nvfp4_quantize(w, oracle.OUTER_PER_GROUP, group_offsets=np.arange(E + 1) * N)
    assert np.array_equal(c.cpu().numpy(), rc) and np.array_equal(s.cpu().numpy(), rs)
    assert np.array_equal(g.cpu().numpy().view(np.uint32), rg.view(np.uint32))


def guarded(shape, dtype, fill):
    nbytes = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
    buf = torch.full((GUARD + nbytes + GUARD,), fill, dtype=torch.uint8, device="cuda")
    return buf, buf[GUARD:GUARD + nbytes].view(dtype).view(shape)


def check_guarded(P, call, specs, what):
    """call(*outs) with every output between guards, twice (0xAB and 0x00 prefill)"""
    results = []
    for fill in (0xAB, 0x00):
        bufs = [guarded(shape, dtype, fill) for shape, dtype in specs]
        call(*[v for _, v in bufs])
        torch.cuda.synchronize()
        for i, (buf, _) in enumerate(bufs):
            assert torch.all(buf[:GUARD] == fill) and torch.all(buf[-GUARD:] == fill), \
                "%s: output %d wrote outside its buffer" % (what, i)
        results.append([v.clone() for _, v in bufs])
    for i, (a, b) in enumerate(zip(*results)):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), "%s: output %d not fully written" % (what, i)
    assert P.get_device_error() == 0


def test_guard_bytes_quantisers(P):
    rng = np.random.default_rng(3)
    u8, f32 = torch.uint8, torch.float32
    x = dev_bf16(W.normal_bf16_host(rng, (96, 1536), 1.0, 0.01, 30.0))
    check_guarded(P, lambda c, s, g: P.nvfp4_quantize(x, four_over_six=True, out=(c, s, g)),
                  [((96, 768), u8), ((96, 96), u8), ((96,), f32)], "nvfp4 per row")
    y = dev_bf16(W.normal_bf16_host(rng, (32, 2 * 1536), 0.5))
    check_guarded(P, lambda c, s, g: P.nvfp4_quantize(y, cols=1536, swiglu=True, four_over_six=True,
                                                      out=(c, s, g)),
                  [((32, 768), u8), ((32, 96), u8), ((32,), f32)], "nvfp4 SwiGLU")
    w = dev_bf16(W.normal_bf16_host(rng, (3 * 520, 1024), 0.02))
    check_guarded(P, lambda c, s, g: P.nvfp4_quantize(w, outer_mode=P.OUTER_PER_GROUP, rows_per_group=520,
                                                      out=(c, s, g)),
                  [((1560, 512), u8), ((1560, 64), u8), ((3,), f32)], "nvfp4 per expert")
    d = dev_bf16(W.normal_bf16_host(rng, (256, 640), 1e-3))
    check_guarded(P, lambda q, s: P.mxfp8_quantize(d, False, out=(q, s)),
                  [((256, 640), u8), ((256, 20), u8)], "mxfp8 rows")
    check_guarded(P, lambda q, s: P.mxfp8_quantize(d, True, out=(q, s)),
                  [((640, 256), u8), ((640, 8), u8)], "mxfp8 transposed")
    check_guarded(P, lambda q, s: P.mxfp8_quantize_swiglu(y, out=(q, s)),
                  [((32, 1536), u8), ((32, 48), u8)], "mxfp8 SwiGLU")


def test_guard_bytes_requantisation_and_combine(P):
    rng = np.random.default_rng(4)
    u8, f32 = torch.uint8, torch.float32
    rows, cols = 160, 192
    c, s, g = (dev(a) for a in oracle.nvfp4_quantize(W.normal_bf16_host(rng, (rows, cols)), oracle.OUTER_PER_ROW,
                                                     four_over_six=True))
    check_guarded(P, lambda q, qs: P.requant_transpose_sr_mxfp8(c, s, g, True, 1, rows, cols, 5, 1, out=(q, qs)),
                  [((1, cols, rows), u8), ((1, cols, rows // 32), u8)], "requant MXFP8")
    check_guarded(P, lambda q, qs, go: P.requant_transpose_sr_nvfp4(c, s, g, True, 1, rows, cols, 5, 1,
                                                                    out=(q, qs, go)),
                  [((1, cols, rows // 2), u8), ((1, cols, rows // 16), u8), ((1,), f32)], "requant NVFP4")
    acc = dev(rng.standard_normal((64, 256)).astype(np.float32))
    check_guarded(P, lambda q, qs: P.rht_s2f6_quantize(acc, 9, out=(q, qs)),
                  [((64, 256), torch.int8), ((64, 8), u8)], "RHT + S2F6")
    q8, sc8 = W.combine_payload(64, 256, 3)
    idx = dev(np.array([[0, 5, -1], [63, 2, 7], [10, 11, 12], [-1, -1, -1]], np.int32))
    gates = dev(np.full((4, 3), 0.25, np.float32))
    check_guarded(P, lambda o: P.combine_receive_s2f6((dev(q8), dev(sc8)), 3, idx, gates, torch.bfloat16, out=o),
                  [((4, 256), torch.bfloat16)], "combine receive")


def test_guard_bytes_gemms(P):
    rng = np.random.default_rng(5)
    u8, f32, bf16 = torch.uint8, torch.float32, torch.bfloat16
    E, d, f = 3, 512, 256
    counts = [128, 129, 127]
    offs_h = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    T = int(offs_h[-1])
    offs = dev(offs_h)
    A = tuple(dev(a) for a in oracle.nvfp4_quantize(W.normal_bf16_host(rng, (T, d)), oracle.OUTER_PER_ROW,
                                                    four_over_six=True))
    wq = oracle.nvfp4_quantize(W.normal_bf16_host(rng, (E * 2 * f, d), 0.02), oracle.OUTER_PER_GROUP,
                               group_offsets=np.arange(E + 1) * 2 * f)
    B = (dev(wq[0].reshape(E, 2 * f, d // 2)), dev(wq[1].reshape(E, 2 * f, d // 16)), dev(wq[2]))
    check_guarded(P, lambda o: P.grouped_gemm_nvfp4(A, B, offs, out_dtype=bf16, out=o), [((T, 2 * f), bf16)],
                  "NVFP4 GEMM bf16")
    check_guarded(P, lambda o: P.grouped_gemm_nvfp4(A, B, offs, out_dtype=f32, out=o), [((T, 2 * f), f32)],
                  "NVFP4 GEMM f32")
    check_guarded(P, lambda h, c, s, g: P.w1_gemm_swiglu_nvfp4(A, B, offs, True, out=(c, s, g), h=h),
                  [((T, f), bf16), ((T, f // 2), u8), ((T, f // 16), u8), ((T,), f32)], "w1 GEMM + SwiGLU + NVFP4")
    H = tuple(dev(a) for a in oracle.nvfp4_quantize(W.normal_bf16_host(rng, (T, f)), oracle.OUTER_PER_ROW,
                                                    four_over_six=True))
    w2 = oracle.nvfp4_quantize(W.normal_bf16_host(rng, (E * d, f), 0.02), oracle.OUTER_PER_GROUP,
                               group_offsets=np.arange(E + 1) * d)
    B2 = (dev(w2[0].reshape(E, d, f // 2)), dev(w2[1].reshape(E, d, f // 16)), dev(w2[2]))
    check_guarded(P, lambda q, s: P.w2_gemm_rht_s2f6(H, B2, offs, 11, out=(q, s)),
                  [((T, d), torch.int8), ((T, d // 32), u8)], "w2 GEMM + RHT + S2F6")
    a8, a8s = (dev(v) for v in oracle.mxfp8_quantize(W.normal_bf16_host(rng, (T, d), 1e-3)))
    b8, b8s = oracle.mxfp8_quantize(W.normal_bf16_host(rng, (E * f, d), 0.02))
    b8, b8s = dev(b8.reshape(E, f, d)), dev(b8s.reshape(E, f, d // 32))
    check_guarded(P, lambda o: P.gemm_mxfp8(a8, a8s, b8, b8s, offs, P.GROUP_M, bf16, out=o), [((T, f), bf16)],
                  "MXFP8 M-grouped")
    Kt = 512
    koffs = dev(np.array([0, 128, 128, 512], np.int32))
    at, ats = (dev(v) for v in oracle.mxfp8_quantize(W.normal_bf16_host(rng, (Kt, 256), 1e-3), transpose=True))
    bt, bts = (dev(v) for v in oracle.mxfp8_quantize(W.normal_bf16_host(rng, (Kt, 128)), transpose=True))
    check_guarded(P, lambda o: P.gemm_mxfp8(at, ats, bt, bts, koffs, P.GROUP_K, f32, out=o), [((3, 256, 128), f32)],
                  "MXFP8 K-grouped")


def test_guard_bytes_short_segment_gemms(P):
    """The 32-row tiles that the NVFP4 GEMMs take for short segments (a
    decode-like batch, 16 rows per expert or fewer on average) store their
    rows directly: every output row written once, nothing past the last row."""
    rng = np.random.default_rng(6)
    u8, f32, bf16 = torch.uint8, torch.float32, torch.bfloat16
    E, d, f = 8, 512, 256
    counts = [1, 0, 40, 3, 2, 0, 5, 1]
    offs_h = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    T = int(offs_h[-1])
    assert T <= 16 * E
    offs = dev(offs_h)
    A = tuple(dev(a) for a in oracle.nvfp4_quantize(W.normal_bf16_host(rng, (T, d)), oracle.OUTER_PER_ROW,
                                                    four_over_six=True))
    wq = oracle.nvfp4_quantize(W.normal_bf16_host(rng, (E * 2 * f, d), 0.02), oracle.OUTER_PER_GROUP,
                               group_offsets=np.arange(E + 1) * 2 * f)
    B = (dev(wq[0].reshape(E, 2 * f, d // 2)), dev(wq[1].reshape(E, 2 * f, d // 16)), dev(wq[2]))
    check_guarded(P, lambda o: P.grouped_gemm_nvfp4(A, B, offs, out_dtype=bf16, out=o), [((T, 2 * f), bf16)],
                  "short NVFP4 GEMM bf16")
    check_guarded(P, lambda o: P.grouped_gemm_nvfp4(A, B, offs, out_dtype=f32, out=o), [((T, 2 * f), f32)],
                  "short NVFP4 GEMM f32")
    check_guarded(P, lambda h, c, s, g: P.w1_gemm_swiglu_nvfp4(A, B, offs, True, out=(c, s, g), h=h),
                  [((T, f), bf16), ((T, f // 2), u8), ((T, f // 16), u8), ((T,), f32)],
                  "short w1 GEMM + SwiGLU + NVFP4")
    H = tuple(dev(a) for a in oracle.nvfp4_quantize(W.normal_bf16_host(rng, (T, f)), oracle.OUTER_PER_ROW,
                                                    four_over_six=True))
    w2 = oracle.nvfp4_quantize(W.normal_bf16_host(rng, (E * d, f), 0.02), oracle.OUTER_PER_GROUP,
                               group_offsets=np.arange(E + 1) * d)
    B2 = (dev(w2[0].reshape(E, d, f // 2)), dev(w2[1].reshape(E, d, f // 16)), dev(w2[2]))
    check_guarded(P, lambda q, s: P.w2_gemm_rht_s2f6(H, B2, offs, 11, out=(q, s)),
                  [((T, d), torch.int8), ((T, d // 32), u8)], "short w2 GEMM + RHT + S2F6")
