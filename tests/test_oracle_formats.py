"""Pins for the oracle's element and scale formats (no GPU).

Each check compares the oracle with something other than itself: the value
set printed on the pages, PyTorch's float8 dtypes, the host conversions in
CUDA's cuda_fp4.h / cuda_fp8.h headers, or a brute-force nearest search.
"""
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest
import torch

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_fp4_value_set_matches_pages(golden):
    vals = sorted({oracle.e2m1_value(c) for c in range(16)})
    want = sorted(set(golden["fp4_value_set"]["values"]))
    assert vals == want
    assert max(abs(v) for v in vals) == golden["fp4_value_set"]["max_magnitude"]
    assert np.signbit(oracle.e2m1_value(8)) and oracle.e2m1_value(8) == 0.0


def test_e4m3_decode_all_bytes_vs_torch():
    b = torch.arange(256, dtype=torch.uint8)
    ref = b.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_value(i) for i in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])
    assert np.nanmax(got) == 448.0


def test_e8m0_decode_all_bytes_vs_torch():
    b = torch.arange(256, dtype=torch.uint8)
    ref = b.view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    got = np.array([oracle.e8m0_value(i) for i in range(256)])
    assert np.isnan(got[255]) and np.isnan(ref[255])
    assert np.array_equal(ref[:255], got[:255])


def test_s2f6_range_and_decode(golden):
    vals = np.array([oracle.s2f6_value(k) for k in range(-128, 128)])
    assert np.array_equal(vals, np.arange(-128, 128) / 64.0)
    assert vals.min() == golden["s2f6"]["min"] and vals.max() == golden["s2f6"]["max"]


def _all_finite_bf16_as_f32():
    bits = np.arange(65536, dtype=np.uint32)
    f = (bits << 16).view(np.float32)
    return f[np.isfinite(f)]


def _brute_e2m1(v):
    """Nearest of the 8 magnitudes by exhaustive search; ties to the even code;
    saturate at 6; sign kept."""
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    a = min(abs(float(v)), 6.0)
    best, bestd = None, None
    for c, m in enumerate(mags):
        d = abs(a - m)
        if bestd is None or d < bestd or (d == bestd and c % 2 == 0 and best % 2 == 1):
            best, bestd = c, d
    return best | (8 if np.signbit(v) else 0)


def test_e2m1_rne_brute_force_all_bf16():
    vals = _all_finite_bf16_as_f32()
    # restrict to the interesting range; everything above 6 saturates
    sel = vals[np.abs(vals) < 16.0]
    for v in sel[::7]:
        assert oracle.e2m1_rne(v) == _brute_e2m1(v), v
    for v in [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, 100.0, -1e30, 1e-30]:
        assert oracle.e2m1_rne(v) == _brute_e2m1(np.float32(v)), v


def test_three_point_two_rounds_to_three(golden):
    ex = golden["rounding_error_example"]
    c = oracle.e2m1_rne(ex["x"])
    assert oracle.e2m1_value(c) == ex["q"]
    assert abs((oracle.e2m1_value(c) - ex["x"]) - ex["error"]) < 1e-6


def test_e4m3_rne_vs_torch_in_range():
    vals = _all_finite_bf16_as_f32()
    vals = vals[np.abs(vals) < 464.0]
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_rne(v) for v in vals], np.uint8)
    assert np.array_equal(ref, got)
    rng = np.random.default_rng(5)
    r = (rng.standard_normal(20000) * 60).astype(np.float32)
    r = r[np.abs(r) < 464]
    ref = torch.from_numpy(r).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ref, np.array([oracle.e4m3_rne(v) for v in r], np.uint8))


def test_e4m3_saturates():
    for v in [464.0, 480.0, 1e6, 3e38]:
        assert oracle.e4m3_rne(v) == 0x7E
        assert oracle.e4m3_rne(-v) == 0xFE


@pytest.fixture(scope="module")
def cuda_host_codecs():
    gxx = shutil.which("g++")
    inc = "/usr/local/cuda/include"
    if gxx is None or not os.path.exists(os.path.join(inc, "cuda_fp4.h")):
        pytest.skip("no g++ or CUDA headers")
    d = tempfile.mkdtemp()
    exe = os.path.join(d, "codecs")
    subprocess.run([gxx, "-O1", "-I", inc, os.path.join(ROOT, "tests", "cuda_host_codecs.cpp"), "-o", exe],
                   check=True)
    yield exe
    shutil.rmtree(d, ignore_errors=True)


def test_codecs_vs_cuda_header_conversions(cuda_host_codecs):
    vals = _all_finite_bf16_as_f32()
    rng = np.random.default_rng(11)
    extra = np.concatenate([(rng.standard_normal(50000) * s).astype(np.float32) for s in (0.3, 3.0, 100.0)])
    vals = np.concatenate([vals, extra]).astype(np.float32)
    p = subprocess.run([cuda_host_codecs], input=vals.tobytes(), capture_output=True, check=True)
    out = np.frombuffer(p.stdout, np.uint8)
    fp4, fp8 = out[:len(vals)], out[len(vals):]
    got4 = np.array([oracle.e2m1_rne(v) for v in vals], np.uint8)
    got8 = np.array([oracle.e4m3_rne(v) for v in vals], np.uint8)
    assert np.array_equal(got4, fp4)
    assert np.array_equal(got8, fp8)


def test_bf16_rne_vs_torch():
    rng = np.random.default_rng(3)
    v = rng.standard_normal(20000) * 10.0 ** rng.integers(-8, 8, 20000)
    # torch rounds binary32 -> bf16; use values exact in binary32 to compare
    v32 = v.astype(np.float32)
    ref = torch.from_numpy(v32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.bf16_rne_array(v32.astype(np.float64))
    assert np.array_equal(ref, got)


def test_storage_bits_per_value(golden):
    """The pages' bits per value (NVFP4 4.5, MXFP8 and the S2F6 combine 8.25)
    measured on the buffers the oracle returns: the bytes of every code and
    scale tensor (outer scales are per row or per tensor, not per value)."""
    import precision_moe_numerics_gb300.workloads as W
    bpv = golden["bits_per_value"]
    rng = np.random.default_rng(4)
    rows, cols = 64, 4096
    x = W.normal_bf16_host(rng, (rows, cols))
    c, s, g = oracle.nvfp4_quantize(x, oracle.OUTER_PER_ROW, four_over_six=True)
    assert (c.nbytes + s.nbytes) * 8 / x.size == bpv["nvfp4"]
    assert g.shape == (rows,)
    q, qs = oracle.mxfp8_quantize(x)
    assert (q.nbytes + qs.nbytes) * 8 / x.size == bpv["mxfp8"]
    qt, qts = oracle.mxfp8_quantize(x, transpose=True)
    assert (qt.nbytes + qts.nbytes) * 8 / x.size == bpv["mxfp8"]
    rq, rqs = oracle.requant_transpose_mxfp8(c, s, g, True, 1, rows, cols, 0, oracle.TAG_X)
    assert (rq.nbytes + rqs.nbytes) * 8 / x.size == bpv["mxfp8"]
    z, zs = oracle.rht_s2f6(W.bf16_bits_to_f32(x), 0)
    assert (z.nbytes + zs.nbytes) * 8 / x.size == bpv["combine_s2f6"]
    fc, fs, fg = oracle.requant_transpose_nvfp4(c, s, g, True, 1, rows, cols, 0, oracle.TAG_X)
    assert (fc.nbytes + fs.nbytes) * 8 / x.size == bpv["nvfp4"]
