"""GPU parity at the documented limits of the boundary: 1024 groups for every
grouped GEMM (most empty, some of one to three rows, one long segment), the
1025th rejected on the host, and the combine receive at its largest top-k
(64).  Tolerances and byte rules as in test_gpu_gemm.py,
test_gpu_swiglu_gemm.py and test_gpu_combine.py."""
import numpy as np
import pytest
import torch

import oracle
from precision_moe_numerics_gb300 import workloads as W
from swiglu_checks import check_h, check_h_coding, gemm_ref

pytestmark = pytest.mark.gpu

G = 1024


@pytest.fixture(scope="module")
def pmn():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from precision_moe_numerics_gb300 import build, pmn as P
    build.build()
    return P


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def sparse_counts(rng, groups, long_rows):
    counts = np.zeros(groups, np.int64)
    hit = rng.choice(groups, 60, replace=False)
    counts[hit] = rng.integers(1, 4, hit.size)
    counts[groups // 2] = long_rows
    counts[groups - 1] = 3  # the last group is not empty
    return counts


def nvfp4_operands(rng, counts, n, k):
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    T = int(offs[-1])
    E = len(counts)
    a = oracle.nvfp4_quantize(W.normal_bf16_host(rng, (T, k), 1.0, 0.01, 30.0), oracle.OUTER_PER_ROW,
                              four_over_six=True)
    bq = oracle.nvfp4_quantize(W.normal_bf16_host(rng, (E * n, k), 0.02), oracle.OUTER_PER_GROUP,
                               group_offsets=np.arange(E + 1) * n)
    b = (bq[0].reshape(E, n, k // 2), bq[1].reshape(E, n, k // 16), bq[2])
    return offs, a, b


def test_grouped_nvfp4_gemm_at_1024_experts(pmn):
    rng = np.random.default_rng(61)
    n, k = 128, 256
    offs, a, b = nvfp4_operands(rng, sparse_counts(rng, G, 200), n, k)
    out = pmn.grouped_gemm_nvfp4(tuple(dev(x) for x in a), tuple(dev(x) for x in b), dev(offs),
                                 out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert pmn.get_device_error() == 0
    ref, absab = gemm_ref(*a, *b, offs)
    got = out.cpu().numpy().astype(np.float64)
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert rel <= 1e-5, rel
    assert np.all(np.abs(got - ref) <= 1e-3 * absab + 1e-30)
    # one group more than the scheduler's table holds: rejected on the host (contents never read)
    T2 = G + 1
    u8 = lambda *shape: torch.zeros(shape, dtype=torch.uint8, device="cuda")
    a2 = (u8(T2, k // 2), u8(T2, k // 16), torch.ones(T2, device="cuda"))
    b2 = (u8(G + 1, n, k // 2), u8(G + 1, n, k // 16), torch.ones(G + 1, device="cuda"))
    offs2 = torch.arange(G + 2, dtype=torch.int32, device="cuda")
    with pytest.raises(pmn.PmnError):
        pmn.grouped_gemm_nvfp4(a2, b2, offs2)


def test_swiglu_gemm_at_1024_experts(pmn):
    rng = np.random.default_rng(62)
    f, k = 128, 256
    offs, a, b = nvfp4_operands(rng, sparse_counts(rng, G, 150), 2 * f, k)
    A = tuple(dev(x) for x in a)
    h = torch.empty((int(offs[-1]), f), dtype=torch.bfloat16, device="cuda")
    codes, scales, outer = pmn.w1_gemm_swiglu_nvfp4(A, tuple(dev(x) for x in b), dev(offs), True, h=h)
    torch.cuda.synchronize()
    assert pmn.get_device_error() == 0
    y_ref, absab = gemm_ref(*a, *b, offs)
    check_h(h.view(torch.int16).cpu().numpy().view(np.uint16), y_ref, absab, f, "1024 experts")
    check_h_coding(pmn, h, codes, scales, outer, int(offs[-1]), "1024 experts")


def test_mxfp8_gemms_at_1024_groups(pmn):
    rng = np.random.default_rng(63)
    # M-grouped: dX-shaped, K = 512
    counts = sparse_counts(rng, G, 130)
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    M, N, K = int(offs[-1]), 128, 512
    a, asc = oracle.mxfp8_quantize(W.normal_bf16_host(rng, (M, K), 1e-3, 0.01, 20.0))
    b, bsc = oracle.mxfp8_quantize(W.normal_bf16_host(rng, (G * N, K), 0.02))
    b, bsc = b.reshape(G, N, K), bsc.reshape(G, N, K // 32)
    out = pmn.gemm_mxfp8(dev(a), dev(asc), dev(b), dev(bsc), dev(offs), pmn.GROUP_M, torch.float32)
    ref = oracle.gemm_mxfp8_mgrouped(a, asc, b, bsc, offs)
    got = out.cpu().numpy().astype(np.float64)
    for g in np.nonzero(counts)[0]:
        lo, hi = offs[g], offs[g + 1]
        absab = np.abs(oracle.mxfp8_dequant_f64(a[lo:hi], asc[lo:hi])) @ np.abs(
            oracle.mxfp8_dequant_f64(b[g], bsc[g])).T
        assert np.all(np.abs(got[lo:hi] - ref[lo:hi]) <= 1e-3 * absab + 1e-30), "M-grouped group %d" % g
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert rel <= 1e-5, rel
    # K-grouped: dW-shaped, segments of 0 or 128 rows over 1024 groups
    kc = np.zeros(G, np.int64)
    kc[rng.choice(G, 8, replace=False)] = 128
    koffs = np.concatenate([[0], np.cumsum(kc)]).astype(np.int32)
    Kt, Mw, Nw = int(koffs[-1]), 128, 128
    at, ats = oracle.mxfp8_quantize(W.normal_bf16_host(rng, (Kt, Mw), 1e-3), transpose=True)
    bt, bts = oracle.mxfp8_quantize(W.normal_bf16_host(rng, (Kt, Nw)), transpose=True)
    outk = pmn.gemm_mxfp8(dev(at), dev(ats), dev(bt), dev(bts), dev(koffs), pmn.GROUP_K, torch.float32)
    torch.cuda.synchronize()
    assert pmn.get_device_error() == 0
    outk = outk.cpu().numpy()
    for g in range(G):
        lo, hi = koffs[g], koffs[g + 1]
        if hi == lo:
            assert np.all(outk[g] == 0), "empty K group %d" % g
            continue
        A = oracle.mxfp8_dequant_f64(at[:, lo:hi], ats[:, lo // 32:hi // 32])
        B = oracle.mxfp8_dequant_f64(bt[:, lo:hi], bts[:, lo // 32:hi // 32])
        assert np.all(np.abs(outk[g] - A @ B.T) <= 1e-3 * (np.abs(A) @ np.abs(B).T) + 1e-30), "K group %d" % g


def test_combine_receive_at_top64(pmn):
    from test_gpu_combine import check, tolerance
    rng = np.random.default_rng(64)
    rows, cols, tokens, k = 512, 256, 16, 64
    q, sc = W.combine_payload(rows, cols, 5)
    idx = rng.integers(0, rows, (tokens, k)).astype(np.int32)
    idx[0, 5] = -1  # a dropped choice
    gates = rng.random((tokens, k)).astype(np.float32)
    gates /= gates.sum(axis=1, keepdims=True)
    out = pmn.combine_receive_s2f6((dev(q), dev(sc)), 5, dev(idx), dev(gates), out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert pmn.get_device_error() == 0
    ref = oracle.combine_receive(q, sc, 5, idx, gates)
    check(out, ref, tolerance(q, sc, idx, gates), "top-64 combine")
