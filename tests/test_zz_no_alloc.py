"""The per-group NVFP4 quantisation entry point whose scratch is a fixed device
array (pmn_nvfp4_quantize_per_group_noalloc) produces the same bytes as the
workspace entry point, call after call.  It serves callers that cannot
allocate device memory while they run (all memory reserved at start-up, or a
host framework that owns every allocation).  Collected last, so it also runs
after every other GPU test has used the library; it passes alone as well."""
import numpy as np
import pytest
import torch

from precision_moe_numerics_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pmn():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from precision_moe_numerics_gb300 import build, pmn as p
    build.build()
    return p


def dev_bf16(host_bits):
    return torch.from_numpy(host_bits.view(np.int16)).cuda().view(torch.bfloat16)


def test_noalloc_matches_allocating_entry_point_on_two_calls(pmn):
    rng = np.random.default_rng(5)
    E, N, K = 4, 520, 1024  # several work chunks per expert, ragged last chunk
    w = W.normal_bf16_host(rng, (E * N, K), 0.02)
    w[2 * N:3 * N] = 0  # an all-zero expert
    x = dev_bf16(w)
    ref = pmn.nvfp4_quantize(x, outer_mode=pmn.OUTER_PER_GROUP, rows_per_group=N)
    for call in range(2):
        got = pmn.nvfp4_quantize_per_group_noalloc(x, N)
        torch.cuda.synchronize()
        for a, b, what in zip(got, ref, ("codes", "scales", "outer")):
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), "call %d: %s differ" % (call, what)
    assert pmn.get_device_error() == 0


def test_noalloc_group_limit(pmn):
    rng = np.random.default_rng(6)
    x = dev_bf16(W.normal_bf16_host(rng, (1024 * 16, 64), 1.0))
    ref = pmn.nvfp4_quantize(x, outer_mode=pmn.OUTER_PER_GROUP, rows_per_group=16)
    got = pmn.nvfp4_quantize_per_group_noalloc(x, 16)  # exactly the maximum, 1024 groups
    for a, b in zip(got, ref):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    y = dev_bf16(W.normal_bf16_host(rng, (1025 * 16, 64), 1.0))
    with pytest.raises(pmn.PmnError):
        pmn.nvfp4_quantize_per_group_noalloc(y, 16)  # 1025 groups: rejected on the host
    assert pmn.get_device_error() == 0


def test_noalloc_on_a_side_stream_with_four_over_six(pmn):
    """The stream argument and the 4/6 flag are forwarded: two calls in a row on
    a non-default stream, byte for byte against the workspace entry point
    (four_over_six=1) on the same stream."""
    rng = np.random.default_rng(7)
    E, N, K = 3, 600, 2048
    x = dev_bf16(W.normal_bf16_host(rng, (E * N, K), 0.02, 0.001, 30.0))
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        ref = pmn.nvfp4_quantize(x, outer_mode=pmn.OUTER_PER_GROUP, rows_per_group=N, four_over_six=True,
                                 stream=side)
        for call in range(2):
            got = pmn.nvfp4_quantize_per_group_noalloc(x, N, four_over_six=True, stream=side)
            side.synchronize()
            for a, b, what in zip(got, ref, ("codes", "scales", "outer")):
                assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), "call %d: %s differ" % (call, what)
    # the 4/6 flag reached the kernel: its outer scale is amax / (4 * 448), not amax / (6 * 448)
    amax = x.float().abs().view(E, -1).amax(dim=1)
    assert torch.allclose(got[2], amax / 1792.0, rtol=1e-6, atol=0.0)
    assert pmn.get_device_error(side) == 0
