"""GPU parity of the NVFP4 requantisation of the FP4 backward (dequantise ->
transpose -> NVFP4 with stochastic or nearest rounding) against the oracle:
codes, E4M3 scales and the outer scale byte for byte, on oracle-quantised
inputs with per-token (4/6) and per-expert outer scales, ragged tiles, zero
padding rows and an all-zero entry."""
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


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def case(rng, batch, rows, cols, per_row):
    x = W.normal_bf16_host(rng, (batch * rows, cols), 1.0, 0.002, 40.0)
    x[rows - 32:rows] = 0                      # zero padding rows at the end of the first entry
    if per_row:
        return oracle.nvfp4_quantize(x, oracle.OUTER_PER_ROW, four_over_six=True)
    return oracle.nvfp4_quantize(x, oracle.OUTER_PER_GROUP, group_offsets=np.arange(batch + 1) * rows)


@pytest.mark.parametrize("per_row,batch,rows,cols", [(True, 1, 256, 512), (True, 1, 160, 192),
                                                     (False, 3, 128, 256), (False, 2, 96, 1536)])
@pytest.mark.parametrize("stochastic", [True, False])
def test_requant_nvfp4_matches_oracle(P, per_row, batch, rows, cols, stochastic):
    rng = np.random.default_rng(rows + cols + batch)
    c, s, g = case(rng, batch, rows, cols, per_row)
    if not per_row and batch > 2:
        c[rows:2 * rows] = 0                   # an all-zero entry: outer scale 1, zero scales
        s[rows:2 * rows] = 0
    seed, tag = 1234, 3
    got = P.requant_transpose_sr_nvfp4(dev(c), dev(s), dev(g), per_row, batch, rows, cols, seed, tag,
                                       stochastic=stochastic)
    torch.cuda.synchronize()
    want = oracle.requant_transpose_nvfp4(c, s, g, per_row, batch, rows, cols, seed, tag, stochastic=stochastic)
    for a, b, what in zip(got, want, ("codes", "scales", "outer")):
        a = a.cpu().numpy()
        if what == "outer":
            a, b = a.view(np.uint32), b.view(np.uint32)
        bad = np.argwhere(a.reshape(b.shape) != b)
        assert bad.size == 0, "%s: %d mismatches, first at %s" % (what, len(bad), bad[0])


def test_requant_nvfp4_deterministic_and_arguments(P):
    rng = np.random.default_rng(5)
    c, s, g = case(rng, 1, 128, 128, True)
    a = P.requant_transpose_sr_nvfp4(dev(c), dev(s), dev(g), True, 1, 128, 128, 9, 1)
    b = P.requant_transpose_sr_nvfp4(dev(c), dev(s), dev(g), True, 1, 128, 128, 9, 1)
    for u, v in zip(a, b):
        assert torch.equal(u, v)
    with pytest.raises(P.PmnError):            # rows % 32 != 0
        P.requant_transpose_sr_nvfp4(dev(c[:112]), dev(s[:112]), dev(g[:112]), True, 1, 112, 128, 9, 1)


@pytest.mark.parametrize("hot_row", [0, 37, 63])
def test_requant_nvfp4_outer_from_planted_row(P, hot_row):
    """The new outer scale is the largest dec(S) * g of the entry: one row
    carries a value far above the rest, so the maximum sits in that row and
    pairing a scale with its neighbour row's outer scale would change it.
    Five scale words per row, so 16-byte pieces of the scales cross rows."""
    rows, cols = 96, 320
    rng = np.random.default_rng(hot_row)
    x = W.normal_bf16_host(rng, (rows, cols), 1.0, 0.002, 40.0)
    x[rows - 32:] = 0
    x[hot_row, (7 * hot_row) % cols] = 0x4461   # bf16 bits of 900.0
    c, s, g = oracle.nvfp4_quantize(x, oracle.OUTER_PER_ROW, four_over_six=True)
    got = P.requant_transpose_sr_nvfp4(dev(c), dev(s), dev(g), True, 1, rows, cols, 77, 2)
    torch.cuda.synchronize()
    want = oracle.requant_transpose_nvfp4(c, s, g, True, 1, rows, cols, 77, 2, stochastic=True)
    assert got[2].cpu().numpy().view(np.uint32)[0] == want[2].view(np.uint32)[0]
    for a, b in zip(got[:2], want[:2]):
        assert np.array_equal(a.cpu().numpy().reshape(b.shape), b)
