"""GPU parity of the combine's receive side (S2F6 decode, inverse RHT-32,
gate-weighted sum back to token order) against the binary64 oracle.

Tolerance, from the kernel's float32 arithmetic: the kernel sums the k
choices before the transform (u = sum_i s_i k_i by fma, s_i = gate_i
2^(e_i - 6)), runs five butterfly stages and one multiply by RN(1/sqrt(32)).
Each of those k + 7 roundings is at most 2^-24 of a partial sum bounded by
A = sum_i |gate_i| sum_{m in block} |k_im| 2^(e_i - 6) / sqrt(32)
(times sqrt(32) for the butterflies, which the final scale takes back), so
|float32 result - binary64| <= (k + 8) 2^-24 A; the test allows twice that.
Where a row scale gate * 2^(e - 6) falls below the float32 normal range it
rounds on the 2^-149 grid instead (2^-150 |k|_1 / sqrt(32), doubled), and
partial sums in that range add (k + 8) 32 2^-149 at most.  A
bf16 result must be the nearest-even rounding of some value within that
band: RN(ref - tol) <= got <= RN(ref + tol).
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


def tolerance(q, sc, idx, gates):
    rows, cols = q.shape
    nb, k = cols // 32, idx.shape[1]
    l1 = np.abs(q.astype(np.float64)).reshape(rows, nb, 32).sum(axis=2)
    pw = np.exp2(sc.astype(np.float64) - 133.0)
    A = np.zeros((idx.shape[0], nb))
    S = np.zeros((idx.shape[0], nb))
    for i in range(k):
        ok = idx[:, i] >= 0
        g = np.abs(gates[ok, i].astype(np.float64))[:, None]
        A[ok] += g * l1[idx[ok, i]] * pw[idx[ok, i]]
        # a row scale below the float32 normal range rounds on the 2^-149 grid
        S[ok] += np.where(g * pw[idx[ok, i]] < 2.0 ** -126, 2.0 ** -150, 0.0) * l1[idx[ok, i]]
    tol = (2.0 * (k + 8) * 2.0 ** -24 * A + 2.0 * S) / np.sqrt(32.0) + (k + 8) * 32 * 2.0 ** -149
    return np.repeat(tol, 32, axis=1)


def check(got, ref, tol, what):
    if got.dtype == torch.float32:
        err = np.abs(got.cpu().numpy().astype(np.float64) - ref)
        assert np.all(err <= tol), "%s: %d elements beyond the float32 bound (max excess %.3e)" % (
            what, int((err > tol).sum()), float((err - tol).max()))
    else:
        g = W.bf16_bits_to_f32(got.cpu().view(torch.int16).numpy().view(np.uint16)).astype(np.float64)
        lo = W.bf16_bits_to_f32(oracle.bf16_rne_array(ref - tol)).astype(np.float64)
        hi = W.bf16_bits_to_f32(oracle.bf16_rne_array(ref + tol)).astype(np.float64)
        bad = (g < lo) | (g > hi)
        assert not bad.any(), "%s: %d bf16 elements outside the rounded band" % (what, int(bad.sum()))


def random_payload(rng, rows, cols):
    q = rng.integers(-128, 128, (rows, cols)).astype(np.int8)
    sc = rng.integers(112, 136, (rows, cols // 32)).astype(np.uint8)
    if rows > 2:
        q[1, :] = 127
        q[2, :] = -128
        sc[0, :] = 0                # the smallest E8M0 scale: subnormal row scales
    return q, sc


@pytest.mark.parametrize("k", [8, 3, 1])
@pytest.mark.parametrize("cols", [96, 4096])
def test_combine_receive_random(pmn, k, cols):
    rng = np.random.default_rng(100 + k + cols)
    rows, tokens, seed = 301, 53, 77
    q, sc = random_payload(rng, rows, cols)
    idx = rng.integers(0, rows, (tokens, k)).astype(np.int32)
    idx[5, 0] = -1                  # a dropped choice
    idx[9, :] = -1                  # a token with none left
    idx[11, :] = np.arange(k) % 3   # rows 0..2: extremes and the smallest scale
    gates = rng.uniform(0.0, 1.0, (tokens, k)).astype(np.float32)
    ref = oracle.combine_receive(q, sc, seed, idx, gates)
    tol = tolerance(q, sc, idx, gates)
    for dt in (torch.float32, torch.bfloat16):
        got = pmn.combine_receive_s2f6((dev(q), dev(sc)), seed, dev(idx), dev(gates), out_dtype=dt)
        torch.cuda.synchronize()
        check(got, ref, tol, "combine receive k=%d cols=%d %s" % (k, cols, dt))
        assert np.all(got[9].float().cpu().numpy() == 0.0)
    assert pmn.get_device_error() == 0


def test_combine_receive_round_trip_through_the_w2_epilogue_format(pmn):
    """Routed copies of token rows go through the library's combine
    quantisation and come back through the receive call; the result is
    checked against the oracle on the same payload and, through the oracle's
    own round-trip bound, against the token rows."""
    rng = np.random.default_rng(7)
    routing = W.route_topk(rng.standard_normal((200, 16)).astype(np.float32), 8, pad=32)
    cols, seed = 1024, 3
    x = (rng.standard_normal((200, cols)) * 10.0 ** rng.uniform(-2, 2, (200, 1))).astype(np.float32)
    xr = np.zeros((routing.rows, cols), np.float32)
    real = routing.row_token >= 0
    xr[real] = x[routing.row_token[real]]
    qd, scd = pmn.rht_s2f6_quantize(dev(xr), seed)
    idx, gates = routing.token_rows(), routing.gates
    got = pmn.combine_receive_s2f6((qd, scd), seed, dev(idx), dev(gates), out_dtype=torch.float32)
    q, sc = qd.cpu().numpy(), scd.cpu().numpy()
    rq, rsc = oracle.rht_s2f6(xr, seed)   # the payload is the oracle's, byte for byte
    assert np.array_equal(q, rq) and np.array_equal(sc, rsc)
    ref = oracle.combine_receive(rq, rsc, seed, idx, gates)
    check(got, ref, tolerance(rq, rsc, idx, gates), "round trip")
    err = np.linalg.norm((got.cpu().numpy().astype(np.float64) - x).reshape(200, -1, 32), axis=2)
    e = rsc[idx].astype(np.float64) - 127.0                   # [tokens, k, blocks]
    bound = (gates[:, :, None] * np.sqrt(32.0) * np.exp2(e - 7.0)).sum(axis=1) * 1.001 + 1e-5 * np.linalg.norm(
        x.reshape(200, -1, 32), axis=2)
    assert np.all(err <= bound)


def test_combine_receive_bad_index_latches_and_adds_nothing(pmn):
    rng = np.random.default_rng(8)
    rows, cols, tokens, k, seed = 64, 128, 10, 8, 5
    q, sc = random_payload(rng, rows, cols)
    idx = rng.integers(0, rows, (tokens, k)).astype(np.int32)
    gates = rng.uniform(0.0, 1.0, (tokens, k)).astype(np.float32)
    bad = idx.copy()
    bad[3, 2] = rows + 5            # out of range: the kernel skips the access
    assert pmn.get_device_error() == 0
    got = pmn.combine_receive_s2f6((dev(q), dev(sc)), seed, dev(bad), dev(gates), out_dtype=torch.float32)
    assert pmn.get_device_error() & pmn.DEVERR_BAD_OFFSETS
    assert pmn.get_device_error() == 0
    dropped = idx.copy()
    dropped[3, 2] = -1
    ref = oracle.combine_receive(q, sc, seed, dropped, gates)
    check(got, ref, tolerance(q, sc, dropped, gates), "bad index dropped")


def test_combine_receive_edge_cases(pmn):
    q = torch.zeros((32, 64), dtype=torch.int8, device="cuda")
    sc = torch.full((32, 2), 127, dtype=torch.uint8, device="cuda")
    empty = pmn.combine_receive_s2f6((q, sc), 0, torch.zeros((0, 8), dtype=torch.int32, device="cuda"),
                                     torch.zeros((0, 8), dtype=torch.float32, device="cuda"))
    assert empty.shape == (0, 64)
    with pytest.raises(pmn.PmnError):   # k > 64
        pmn.combine_receive_s2f6((q, sc), 0, torch.zeros((2, 65), dtype=torch.int32, device="cuda"),
                                 torch.zeros((2, 65), dtype=torch.float32, device="cuda"))
    q2 = torch.zeros((32, 48), dtype=torch.int8, device="cuda")     # cols % 32 != 0
    with pytest.raises(pmn.PmnError):
        pmn.combine_receive_s2f6((q2, torch.zeros((32, 1), dtype=torch.uint8, device="cuda")), 0,
                                 torch.zeros((2, 8), dtype=torch.int32, device="cuda"),
                                 torch.zeros((2, 8), dtype=torch.float32, device="cuda"))
    # deterministic run to run
    rng = np.random.default_rng(9)
    qq, ss = random_payload(rng, 128, 256)
    idx = dev(rng.integers(0, 128, (40, 8)).astype(np.int32))
    g = dev(rng.uniform(0, 1, (40, 8)).astype(np.float32))
    a = pmn.combine_receive_s2f6((dev(qq), dev(ss)), 1, idx, g)
    b = pmn.combine_receive_s2f6((dev(qq), dev(ss)), 1, idx, g)
    assert torch.equal(a, b)


def test_combine_receive_fullsize_sampled(pmn):
    """The bench's launch configuration: 16384 tokens, top-8 over 384
    experts, d_model 4096, bf16 out, the routed rows padded and allocated as
    the layer step allocates them; sampled tokens against the oracle."""
    r = W.moe_routing(0)
    rows = ((r.rows + 511) // 512) * 512
    q, sc = W.combine_payload(rows, W.D_MODEL, 0)
    idx, gates = r.token_rows(), r.gates
    got = pmn.combine_receive_s2f6((dev(q), dev(sc)), 0, dev(idx), dev(gates), out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert pmn.get_device_error() == 0
    tokens = idx.shape[0]
    pick = np.unique(np.concatenate([[0, 1, tokens - 1], np.random.default_rng(2).choice(tokens, 61, replace=False)]))
    ref = oracle.combine_receive(q, sc, 0, idx[pick], gates[pick])
    check(got[torch.from_numpy(pick).cuda()], ref, tolerance(q, sc, idx[pick], gates[pick]), "full size")
