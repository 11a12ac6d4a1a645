"""Host-side logic of bench.py (no GPU): the clock sampler keeps only the
samples taken inside the timed region and reports throttle reasons; the DRAM
traffic table counts an entry only while the kernel source is unchanged; the
decode forward's algorithmic bytes are the hit experts' weights plus the
activations; the oracle's CPU baseline reports all threads and one."""
import datetime
import importlib.util
import os
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def load_bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def smi_line(t, mhz, power_cap="Not Active", thermal="Not Active"):
    ts = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return "%s, 0, %d, 2070, 450.00, 0x0, Not Active, Not Active, %s, %s" % (ts, mhz, thermal, power_cap)


def test_clock_sampler_keeps_the_timed_region():
    b = load_bench()
    c = b.ClockSampler(0)
    now = time.time()
    c.out = "\n".join([smi_line(now - 2.0, 900, thermal="Active"),   # warm-up, before the region
                       smi_line(now + 0.10, 2070),
                       smi_line(now + 0.15, 2040, power_cap="Active"),
                       smi_line(now + 0.20, 2070),
                       smi_line(now + 3.00, 600)])                       # after the region
    c.t0, c.t1 = now, now + 0.25
    s = c.summary()
    assert s["samples"] == 3
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]


def test_clock_sampler_without_samples():
    b = load_bench()
    c = b.ClockSampler(0)
    c.out = ""
    assert c.summary()["reasons"] == ["unsampled"]


def test_traffic_table_parses_and_hashes_sources():
    b = load_bench()
    table = b.traffic_table()
    assert "gemm_dw1_mxfp8" in table
    nbytes, sha = table["gemm_dw1_mxfp8"]
    assert nbytes > 1e10 and len(sha) == 12
    # the hash covers the kernel's sources: GEMM and quantiser calls hash different files
    assert b.source_sha("gemm_dw1_mxfp8") != b.source_sha("quant_w1")
    assert b.source_sha("gemm_dw1_mxfp8") == b.source_sha("gemm1_swiglu_nvfp4")


def test_decode_accounting():
    from precision_moe_numerics_gb300 import layer
    from precision_moe_numerics_gb300 import workloads as W
    r = W.decode_routing(0)
    assert r.real_rows == W.DECODE_TOKENS * W.TOP_K and r.rows == r.real_rows  # segments not padded
    hit = int((r.counts > 0).sum())
    fl, by, wb = layer.decode_algorithmic(r.counts, W.D_MODEL, W.D_FF)
    nv = 0.5 + 1 / 16
    assert wb == hit * ((2 * W.D_FF * W.D_MODEL + W.D_MODEL * W.D_FF) * nv + 8)
    assert by > wb
    assert fl == 2.0 * r.real_rows * 2 * W.D_FF * W.D_MODEL + 2.0 * r.real_rows * W.D_MODEL * W.D_FF
    x = W.decode_x(r, 0)
    assert x.shape == (r.rows, W.D_MODEL) and x.dtype == np.uint16


def test_combine_accounting():
    b = load_bench()
    # 16384 tokens x top-8 rows of 4096 S2F6 bytes + 128 scale bytes, index + gate each, bf16 out
    assert b.combine_algorithmic(16384, 8, 4096) == 16384 * 8 * (4096 + 128 + 8) + 16384 * 4096 * 2
    from precision_moe_numerics_gb300 import workloads as W
    q, sc = W.combine_payload(64, 256, 0)
    assert q.dtype == np.int8 and q.shape == (64, 256) and np.abs(q.astype(int)).max() <= 127
    assert sc.dtype == np.uint8 and sc.shape == (64, 8) and 118 <= sc.min() and sc.max() < 130


def test_mxfp8_forward_accounting():
    from precision_moe_numerics_gb300 import layer
    fl, by = layer.mxfp8_forward_algorithmic(131072, 384, 4096, 1536)
    assert fl == 2.0 * 131072 * 3072 * 4096 + 2.0 * 131072 * 4096 * 1536
    w = 384 * (3072 * 4096 + 4096 * 1536)        # weight elements: bf16 read, MXFP8 written and read
    assert by > w * (2 + 2 * 1.03125) and by < w * (2 + 2 * 1.03125) * 1.25


def test_result_line_carries_the_contract_keys():
    import json
    b = load_bench()
    roof = {"bound": "hbm", "achieved": 5300.0, "peak": 6680.8, "unit": "GB/s", "frac": 0.79, "traffic": 1.9e10}
    cpu = {"value": 0.09, "unit": "TFLOP/s", "cores": 16, "kind": "oracle", "sample": "34 experts"}
    e2e = {"value": 650.0, "unit": "TFLOP/s", "h2d_bytes_per_step": 1, "d2h_bytes_per_step": 2}
    clocks = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}
    line = b.result_line(747.2, 1, 30, 3, 19.87, {"workload": "w"}, roof, cpu, e2e, 540, clocks,
                         {"decode": None, "components": {}})
    json.dumps(line)
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e",
                "gpu_launches", "clocks"):
        assert key in line, key
    assert line["value"] == 747.2 and line["higher_is_better"] is True and line["scaling"] == "weak"
    assert line["data"] == "synthetic" and line["gpu_launches"] == 540 and "workload" in line["config"]
    assert set(roof) <= set(line["roofline"]) and line["cpu_baseline"]["kind"] == "oracle"
    assert "decode" in line and "components" in line


def test_cpu_baseline_reports_all_threads_and_one():
    """The oracle's CPU baseline on a small layer: the all-threads figure with
    the thread count OpenMP really uses, a one-thread figure beside it, and the
    thread count restored afterwards."""
    import types
    import oracle
    from precision_moe_numerics_gb300 import workloads as W
    inp = W.moe_device(0, device="cpu", experts=4, tokens=64, d=256, f=128)
    before = oracle.max_threads()
    res = load_bench().cpu_baseline(inp, types.SimpleNamespace(seed=0), budget_s=0.0)
    assert res["kind"] == "oracle" and res["cores"] == before and res["value"] > 0
    assert res["single_thread"]["cores"] == 1 and res["single_thread"]["value"] > 0
    assert "of 4 experts" in res["sample"]
    assert oracle.max_threads() == before
