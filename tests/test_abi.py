"""The C-ABI library builds, loads and exports every entry point that
include/pmn.h declares (no GPU needed: nothing is launched)."""
import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    with open(os.path.join(ROOT, "include", "pmn.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"^PMN_API\s+[\w\s\*]*?\b(pmn_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def libpath():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    from precision_moe_numerics_gb300 import build
    return build.build()


def test_header_declares_the_path():
    syms = declared_symbols()
    for name in ["pmn_nvfp4_quantize", "pmn_requant_transpose_sr_mxfp8", "pmn_grouped_gemm_nvfp4",
                 "pmn_gemm_mxfp8", "pmn_w2_gemm_rht_s2f6", "pmn_mxfp8_quantize", "pmn_rht_s2f6_quantize",
                 "pmn_get_device_error", "pmn_status_string", "pmn_version", "pmn_combine_receive_s2f6",
                 "pmn_mxfp8_quantize_swiglu", "pmn_requant_transpose_sr_nvfp4"]:
        assert name in syms


def test_library_exports_every_declared_symbol(libpath):
    L = ctypes.CDLL(libpath)
    for name in declared_symbols():
        assert hasattr(L, name), name
    from precision_moe_numerics_gb300 import pmn
    assert set(pmn.SIGNATURES) == set(declared_symbols())
    L.pmn_status_string.restype = ctypes.c_char_p
    L.pmn_status_string.argtypes = [ctypes.c_int]
    assert L.pmn_status_string(0) == b"ok"
    assert L.pmn_version() >= 100


def test_host_argument_checks_need_no_gpu(libpath):
    """Invalid arguments are rejected on the host before any CUDA call."""
    from precision_moe_numerics_gb300 import pmn
    L = pmn.lib()
    null = None
    assert L.pmn_nvfp4_quantize(null, 4, 24, 24, 0, 0, 0, 0, null, null, null, null, null, 0,
                                null) == pmn.ERR_INVALID_ARG
    assert L.pmn_mxfp8_quantize(null, 40, 64, 1, null, null, null) == pmn.ERR_INVALID_ARG
    assert L.pmn_mxfp8_quantize_both(null, 64, 64, null, null, null, null, null) == pmn.ERR_INVALID_ARG
    assert L.pmn_mxfp8_quantize_both(1 << 20, 48, 64, 1 << 20, 1 << 20, 1 << 20, 1 << 20, null) == pmn.ERR_INVALID_ARG
    # more than 65535 rows of 128-row CTAs: refused before anything is enqueued
    big = 65536 * 128
    assert L.pmn_mxfp8_quantize_both(1 << 20, big, 32, 1 << 20, 1 << 20, 1 << 20, 1 << 20, null) == pmn.ERR_UNSUPPORTED
    assert L.pmn_mxfp8_quantize(1 << 20, big, 32, 1, 1 << 20, 1 << 20, null) == pmn.ERR_UNSUPPORTED
    assert L.pmn_requant_transpose_sr_mxfp8(null, null, null, 0, 1, 32, 32, 0, 1, 0, null, null,
                                            null) == pmn.ERR_INVALID_ARG
    assert L.pmn_grouped_gemm_nvfp4(null, null, null, null, null, null, null, 0, 0, 128, 256, 0, null,
                                    null) == pmn.ERR_INVALID_ARG
    assert L.pmn_gemm_mxfp8(null, null, null, null, null, 1, 5, 128, 128, 512, 0, null, null) == pmn.ERR_INVALID_ARG
    assert L.pmn_rht_s2f6_quantize(null, 1, 31, 0, null, null, null) == pmn.ERR_INVALID_ARG
    fake = 1 << 20
    # combine receive: cols % 32, k out of 1 .. 64, unknown output kind, misaligned output
    assert L.pmn_combine_receive_s2f6(fake, fake, 64, 48, 0, fake, fake, 4, 8, pmn.OUT_BF16, fake,
                                      null) == pmn.ERR_INVALID_ARG
    assert L.pmn_combine_receive_s2f6(fake, fake, 64, 64, 0, fake, fake, 4, 65, pmn.OUT_BF16, fake,
                                      null) == pmn.ERR_INVALID_ARG
    assert L.pmn_combine_receive_s2f6(fake, fake, 64, 64, 0, fake, fake, 4, 0, pmn.OUT_BF16, fake,
                                      null) == pmn.ERR_INVALID_ARG
    assert L.pmn_combine_receive_s2f6(fake, fake, 64, 64, 0, fake, fake, 4, 8, 7, fake, null) == pmn.ERR_INVALID_ARG
    assert L.pmn_combine_receive_s2f6(fake, fake, 64, 64, 0, fake, fake, 4, 8, pmn.OUT_F32, fake + 4,
                                      null) == pmn.ERR_INVALID_ARG
    assert L.pmn_combine_receive_s2f6(null, null, 64, 64, 0, null, null, 4, 8, pmn.OUT_F32, null,
                                      null) == pmn.ERR_INVALID_ARG
    # no token: nothing to do, NULL buffers allowed
    assert L.pmn_combine_receive_s2f6(null, null, 64, 64, 0, null, null, 0, 8, pmn.OUT_F32, null, null) == pmn.OK
    # SwiGLU + MXFP8: f % 32, misaligned input
    assert L.pmn_mxfp8_quantize_swiglu(fake, 4, 48, fake, fake, null, null) == pmn.ERR_INVALID_ARG
    assert L.pmn_mxfp8_quantize_swiglu(fake + 2, 4, 64, fake, fake, null, null) == pmn.ERR_INVALID_ARG
    assert L.pmn_mxfp8_quantize_swiglu(null, 0, 64, null, null, null, null) == pmn.OK
    # FP4 backward requantisation: rows % 32, cols % 64, unknown rounding, misaligned outer output
    assert L.pmn_requant_transpose_sr_nvfp4(fake, fake, fake, 0, 1, 48, 64, 0, 1, 0, fake, fake, fake,
                                            null) == pmn.ERR_INVALID_ARG
    assert L.pmn_requant_transpose_sr_nvfp4(fake, fake, fake, 0, 1, 64, 96, 0, 1, 0, fake, fake, fake,
                                            null) == pmn.ERR_INVALID_ARG
    assert L.pmn_requant_transpose_sr_nvfp4(fake, fake, fake, 0, 1, 64, 64, 0, 1, 5, fake, fake, fake,
                                            null) == pmn.ERR_INVALID_ARG
    assert L.pmn_requant_transpose_sr_nvfp4(fake, fake, fake, 0, 1, 64, 64, 0, 1, 0, fake, fake, fake + 2,
                                            null) == pmn.ERR_INVALID_ARG
    assert L.pmn_requant_transpose_sr_nvfp4(null, null, null, 0, 0, 64, 64, 0, 1, 0, null, null, null,
                                            null) == pmn.OK          # no entry: nothing to do
    # per-group quantisation: a missing, short or misaligned workspace is rejected on the host
    need = L.pmn_nvfp4_quantize_workspace_bytes(pmn.OUTER_PER_GROUP, 4 * 256, 256)
    assert need == (64 + 2 * 4) * 4
    args = (fake, 4 * 256, 64, 64, pmn.IN_BF16, pmn.OUTER_PER_GROUP, 256, 0, fake, fake, fake, null)
    assert L.pmn_nvfp4_quantize(*args, null, need, null) == pmn.ERR_INVALID_ARG
    assert L.pmn_nvfp4_quantize(*args, fake, need - 4, null) == pmn.ERR_INVALID_ARG
    assert L.pmn_nvfp4_quantize(*args, fake + 8, need, null) == pmn.ERR_INVALID_ARG
    # no rows: nothing to do (the workspace is checked first, and it is valid here)
    assert L.pmn_nvfp4_quantize(fake, 0, 64, 64, pmn.IN_BF16, pmn.OUTER_PER_GROUP, 256, 0, fake, fake, fake, null,
                                fake, need, null) == pmn.OK
    assert L.pmn_nvfp4_quantize_workspace_bytes(pmn.OUTER_PER_ROW, 4, 0) == 0
    assert L.pmn_nvfp4_quantize_workspace_bytes(pmn.OUTER_PER_GROUP, 100, 16) == -1  # rows % rows_per_group
    assert L.pmn_nvfp4_quantize_workspace_bytes(7, 4, 1) == -1
    # bounded-wait self-test: limits above 2 s are refused before anything is enqueued
    assert L.pmn_wait_selftest(2000000001, null) == pmn.ERR_INVALID_ARG
    # the wait limit is process-wide and returns the previous value
    prev = L.pmn_set_wait_limit_ns(123)
    assert L.pmn_set_wait_limit_ns(prev) == 123
    # more groups than the fixed scratch holds: rejected before any pointer is used
    assert L.pmn_nvfp4_quantize_per_group_noalloc(fake, 1025 * 16, 64, 16, 0, fake, fake, fake,
                                                  null) == pmn.ERR_INVALID_ARG


def test_product_path_does_not_import_oracle():
    """The library and its binding never reach the CPU oracle."""
    pkg = os.path.join(ROOT, "precision_moe_numerics_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                with open(os.path.join(dirpath, fn)) as f:
                    src = f.read()
                assert "import oracle" not in src and "from oracle" not in src, fn
                assert "pmn_oracle" not in src, fn
