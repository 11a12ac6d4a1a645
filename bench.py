"""Benchmark of the MoE expert layer's block-scaled numerics path on GB300.

One step = one pass of the whole path over one batch: NVFP4 quantisation of
the bf16 master weights (per expert) and of the routed activations (per token,
4/6), the grouped NVFP4 w1 GEMM with SwiGLU in its epilogue and the NVFP4
quantisation of h, the grouped NVFP4 w2 GEMM with the fused RHT-32 + S2F6
combine quantisation, the
dequantise -> transpose -> SR -> MXFP8 requantisation of X, H, W1 and W2, the
MXFP8 quantisation of dY and dY1 (both orientations) and the four grouped
MXFP8 gradient GEMMs (dX, dW1, dH, dW2).  Workload: 384 experts, top-8 routing
of 16384 tokens (131072 routed rows), d_model 4096, expert d_ff 1536, seeded
synthetic data drawn on the device.

value = expert-GEMM FLOPs of the step (forward NVFP4 + backward MXFP8, on the
real routed rows) / step time.  Per-kernel throughput and roofline fractions
are reported in `components`; the dominant kernel's in `roofline`.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun (N > 1) every rank runs its own replica of the layer (no data
path collective; weak scaling); rank 0 prints one JSON line.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "NVFP4 expert-GEMM TFLOPS (% FP4 peak); quant/requant GB/s (% HBM peak)"
WORKLOAD = ("moe_expert_layer_step: 384 experts, top-8 of 16384 tokens (131072 routed rows, expert segments "
            "padded to 128), d_model 4096, d_ff 1536; NVFP4 fwd + RHT/S2F6 combine + SR-MXFP8 bwd")
NOMINAL_TC_RATIO = {"fp4": 13.5 / 2.25, "fp8": 4.5 / 2.25}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 50 ms from before the
    warm-up; summary() keeps the samples taken between mark_start() and
    mark_end() (host wall clock, the timed region)."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        import datetime
        rows = []
        for line in (self.out or "").strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
            except ValueError:
                continue
        if self.t0 is not None and self.t1 is not None:
            inside = [r for r in rows if self.t0 - 0.05 <= r[0] <= self.t1 + 0.05]
            if inside:
                rows = inside
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, _, r in rows for i, v in enumerate(r) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in rows), "sm_max_mhz": max(r[2] for r in rows),
                "reasons": reasons, "samples": len(rows)}


def traffic_table():
    """DRAM bytes per launch from committed ncu summaries: lines
    `<call-name> <bytes-per-launch> <sha256-prefix-of-source>`; an entry counts
    only while the kernel source is unchanged."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    out = {}
    if not os.path.exists(path):
        return out
    with open(path) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            name, nbytes, sha = line.split()[:3]
            out[name] = (float(nbytes), sha)
    return out


def source_sha(name):
    src = "gemm.cu" if ("gemm" in name) else "quantize.cu"
    h = hashlib.sha256()
    for fn in (src, "numerics.cuh", "sm100.cuh"):
        with open(os.path.join(ROOT, "precision_moe_numerics_gb300", "csrc", fn), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:12]


# ---------------------------------------------------------------------- oracle sample
def oracle_sample(inputs, experts, seed=0):
    """Runs the CPU oracle over the step restricted to `experts` (host copies of
    the same device inputs).  Returns (flops, seconds, threads)."""
    import numpy as np
    import oracle
    import torch

    r = inputs["routing"]
    D, F = inputs["x"].shape[1], inputs["w2"].shape[2]
    F2 = 2 * F
    flops = 0.0
    host = {}
    for e in experts:
        lo, hi = int(r.offsets[e]), int(r.offsets[e + 1])
        n = hi - lo
        if n == 0:
            continue
        hb = lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16)
        host[e] = (hb(inputs["x"][lo:hi]), hb(inputs["w1"][e]), hb(inputs["w2"][e]), hb(inputs["dy"][lo:hi]),
                   hb(inputs["dy1"][lo:hi]), int(r.counts[e]))
    t0 = time.perf_counter()
    for e, (x, w1, w2, dy, dy1, real) in host.items():
        n = x.shape[0]
        w1q = oracle.nvfp4_quantize(w1, oracle.OUTER_PER_GROUP, group_offsets=[0, F2])
        w2q = oracle.nvfp4_quantize(w2, oracle.OUTER_PER_GROUP, group_offsets=[0, D])
        xq = oracle.nvfp4_quantize(x, oracle.OUTER_PER_ROW, four_over_six=True)
        y = oracle.grouped_gemm_nvfp4(xq[0], xq[1], xq[2], w1q[0][None], w1q[1][None], w1q[2], [0, n])
        h = oracle.swiglu_bf16(oracle.bf16_rne_array(y), F)
        hq = oracle.nvfp4_quantize(h, oracle.OUTER_PER_ROW, four_over_six=True)
        z = oracle.grouped_gemm_nvfp4(hq[0], hq[1], hq[2], w2q[0][None], w2q[1][None], w2q[2], [0, n])
        oracle.rht_s2f6(z.astype(np.float32), seed)
        xt = oracle.requant_transpose_mxfp8(xq[0], xq[1], xq[2], True, 1, n, D, seed, oracle.TAG_X)
        ht = oracle.requant_transpose_mxfp8(hq[0], hq[1], hq[2], True, 1, n, F, seed, oracle.TAG_H)
        w1t = oracle.requant_transpose_mxfp8(w1q[0], w1q[1], w1q[2], False, 1, F2, D, seed, oracle.TAG_W1)
        w2t = oracle.requant_transpose_mxfp8(w2q[0], w2q[1], w2q[2], False, 1, D, F, seed, oracle.TAG_W2)
        dyr, dyt = oracle.mxfp8_quantize(dy), oracle.mxfp8_quantize(dy, transpose=True)
        dy1r, dy1t = oracle.mxfp8_quantize(dy1), oracle.mxfp8_quantize(dy1, transpose=True)
        oracle.gemm_mxfp8_mgrouped(dyr[0], dyr[1], w2t[0], w2t[1], [0, n])
        oracle.gemm_mxfp8_kgrouped(dyt[0], dyt[1], ht[0][0], ht[1][0], [0, n])
        oracle.gemm_mxfp8_mgrouped(dy1r[0], dy1r[1], w1t[0], w1t[1], [0, n])
        oracle.gemm_mxfp8_kgrouped(dy1t[0], dy1t[1], xt[0][0], xt[1][0], [0, n])
        flops += 3 * (2.0 * real * D * F2 + 2.0 * real * F * D)
    dt = time.perf_counter() - t0
    return flops, dt, oracle.max_threads()


def pick_sample_experts(r, k):
    """k experts spread over the index range (deterministic)."""
    import numpy as np
    nz = [e for e in range(len(r.counts)) if r.counts[e] > 0]
    idx = np.linspace(0, len(nz) - 1, k).round().astype(int)
    return [nz[i] for i in sorted(set(idx.tolist()))]


# ---------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--experts", type=int, default=None, help="smaller layer for profiling (default 384)")
    ap.add_argument("--tokens", type=int, default=None, help="tokens routed (default 16384)")
    ap.add_argument("--only", default=None, help="time only this call of the step (profiling)")
    ap.add_argument("--combine-only", action="store_true",
                    help="profiling: time only the combine receive, on a seeded payload (--steps calls)")
    ap.add_argument("--no-decode", action="store_true", help="skip the decode, combine-receive, MXFP8-forward, "
                    "FP4-requant and single-expert measurements")
    ap.add_argument("--single-expert-only", action="store_true",
                    help="profiling: only the single-expert forward (T = 4096), printed as one JSON object")
    ap.add_argument("--fp4-requant-only", action="store_true",
                    help="profiling: the step once, then only the FP4-backward requantisations (--steps passes), "
                    "printed as one JSON object")
    args = ap.parse_args()
    rank, world, local = dist_env()

    import torch
    import torch.distributed as dist

    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    if args.impl == "reference":
        if rank == 0:
            run_reference(args)
        if world > 1:
            dist.destroy_process_group()
        return
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from precision_moe_numerics_gb300 import build, layer, pmn
    from precision_moe_numerics_gb300 import workloads as W
    build.build()

    if args.single_expert_only:  # profiling: the single-expert forward alone (< 1 GB on the device)
        res = run_single_expert(args, dev, W, pmn, reps=args.steps)
        if rank == 0:
            print(json.dumps({"single_expert": res}))
        return

    if args.combine_only:  # profiling: the combine receive alone on a seeded payload (< 1 GB on the device)
        r = W.moe_routing(args.seed)
        rows = ((r.rows + 511) // 512) * 512
        q, sc = W.combine_payload(rows, W.D_MODEL, args.seed)
        z = (torch.from_numpy(q).to(dev), torch.from_numpy(sc).to(dev))
        res = run_combine(z, r, args, dev, pmn, reps=args.steps)
        if rank == 0:
            print(json.dumps({"combine_receive": res}))
        return

    kw = {}
    if args.experts:
        kw["experts"] = args.experts
    if args.tokens:
        kw["tokens"] = args.tokens
    inp = W.moe_device(args.seed + rank, device=dev, **kw)
    r = inp["routing"]
    offsets = torch.from_numpy(r.offsets.astype("int32")).to(dev)
    L = layer.ExpertLayerStep(inp["x"], inp["w1"], inp["w2"], inp["dy"], inp["dy1"], offsets, r.real_rows,
                              seed=args.seed)
    calls = L.kernel_calls()
    alg = layer.algorithmic(L.shape)
    if args.fp4_requant_only:  # profiling: the step once (the saved NVFP4 tensors), then the FP4 requantisations
        for _, f in calls:
            f()
        res = run_fp4_requant(L, args, pmn, reps=args.steps)
        if rank == 0:
            print(json.dumps({"fp4_backward_requant": res}))
        return
    if args.only:
        for name, f in calls:  # the step once, so every operand of the chosen call exists
            f()
        only = args.only.split(",")
        calls = [(n, f) for n, f in calls if n in only]
        if len(calls) != len(only):
            raise SystemExit("unknown call in " + args.only)
        alg = {n: alg[n] for n in only}
    flops_step = sum(v[0] for v in alg.values())

    with ClockSampler(local) as clk:  # sampling from before the warm-up; the timed region is marked
        for _ in range(args.warmup):
            for _, f in calls:
                f()
        torch.cuda.synchronize()
        if pmn.get_device_error() != 0:
            raise RuntimeError("device error during warm-up")

        stream = torch.cuda.current_stream()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)] for _ in range(args.steps)]
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        clk.mark_start()
        t_start.record(stream)
        for s in range(args.steps):
            ev[s][0].record(stream)
            for i, (_, f) in enumerate(calls):
                f()
                ev[s][i + 1].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
        clk.mark_end()
    if world > 1:
        dist.barrier()
    ms_total = t_start.elapsed_time(t_end)
    if pmn.get_device_error() != 0:
        raise RuntimeError("device error during the timed region")
    per_call_ms = {name: sum(ev[s][i].elapsed_time(ev[s][i + 1]) for s in range(args.steps)) / args.steps
                   for i, (name, _) in enumerate(calls)}
    ms_step = max_over_ranks(ms_total, world, dist, dev) / args.steps
    value = whole_job_value(flops_step, world, ms_step)

    # ------------------------------------------------------------ end to end
    e2e = None
    if not args.no_e2e and not args.only:
        e2e = run_e2e(L, inp, args, dev, flops_step, world)

    # ------------------------------------------------------------ decode shape
    dec = None
    if not args.no_decode and not args.only:
        dec = run_decode(L, args, dev, W, layer, pmn)

    comb = mxf = fp4b = single = None
    if not args.no_decode and not args.only:
        comb = run_combine(L.z, r, args, dev, pmn)
        mxf = run_mxfp8_forward(inp, r, offsets, args, layer, pmn)
        fp4b = run_fp4_requant(L, args, pmn)
        single = run_single_expert(args, dev, W, pmn)

    pk = peaks()
    comps = {}
    for name, (fl, by) in alg.items():
        ms = per_call_ms[name]
        c = {"ms": round(ms, 4), "GB/s": round(by / (ms * 1e-3) / 1e9, 1),
             "hbm_frac": round(by / (ms * 1e-3) / 1e9 / pk["hbm_gbs"], 3)}
        if fl:
            kind = "fp4" if "nvfp4" in name else "fp8"
            tc_peak = pk["bf16_tflops_sustained"] * NOMINAL_TC_RATIO[kind]
            c["TFLOP/s"] = round(fl / (ms * 1e-3) / 1e12, 1)
            c["tc_frac"] = round(fl / (ms * 1e-3) / 1e12 / tc_peak, 3)
        comps[name] = c
    dom = max(per_call_ms, key=per_call_ms.get)
    fl, by = alg[dom]
    tr = traffic_table().get(dom)
    traffic = tr[0] if tr and tr[1] == source_sha(dom) else None
    if fl:
        kind = "fp4" if "nvfp4" in dom else "fp8"
        tc_peak = pk["bf16_tflops_sustained"] * NOMINAL_TC_RATIO[kind]
        t_c, t_m = fl / tc_peak / 1e12, by / pk["hbm_gbs"] / 1e9
    else:
        t_c, t_m = 0.0, 1.0
    ms = per_call_ms[dom]
    if t_c > t_m:
        roof = {"bound": "tensor", "achieved": round(fl / (ms * 1e-3) / 1e12, 1), "peak": round(tc_peak, 1),
                "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": round(by / (ms * 1e-3) / 1e9, 1), "peak": pk["hbm_gbs"], "unit": "GB/s"}
    roof.update({"frac": round(roof["achieved"] / roof["peak"], 3), "traffic": traffic, "kernel": dom,
                 "algorithmic_bytes": by, "flops": fl, "ms": round(ms, 4), "peak_source": pk["source"],
                 "share_of_step": round(ms / ms_step, 3)})

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.only:
        cpu = cpu_baseline(inp, args)

    clocks = clk.summary()
    if rank == 0:
        launches = (layer.launches_per_step() if not args.only else
                    sum(layer.LAUNCHES.get(n, 1) for n in args.only.split(","))) * args.steps
        config = {"workload": WORKLOAD, "routed_rows": r.real_rows, "padded_rows": r.rows,
                  "experts": L.shape.experts, "d_model": L.shape.d_model, "d_ff": L.shape.d_ff,
                  "flops_per_step": flops_step, "l2": "inputs larger than L2 (no flush needed)",
                  "parallelism": "replicas" if world > 1 else "single-gpu"}
        extra = {"decode": dec, "combine_receive": comb, "mxfp8_forward": mxf, "fp4_backward_requant": fp4b,
                 "single_expert": single, "components": comps}
        print(json.dumps(result_line(value, world, args.steps, args.warmup, ms_step, config, roof, cpu, e2e,
                                     launches, clocks, extra)))
    if world > 1:
        dist.destroy_process_group()


def run_decode(L, args, dev, W, layer, pmn, reps=20):
    """The decode-shaped forward: 64 tokens routed top-8 over the layer's
    experts (segments of a few rows, not padded), quantised and run through
    both NVFP4 GEMMs (RHT + S2F6 epilogue on w2) against the step's resident
    NVFP4 weights of every expert.  CUDA events around `reps` forwards on the
    launching stream; the hit experts' weights (about 3.1 GB) exceed L2, so
    every forward streams them from HBM."""
    import numpy as np
    import torch
    r = W.decode_routing(args.seed)
    xb = W.decode_x(r, args.seed, L.shape.d_model)
    x = torch.from_numpy(np.ascontiguousarray(xb).view(np.int16)).view(torch.bfloat16).to(dev)
    offs = torch.from_numpy(r.offsets.astype(np.int32)).to(dev)
    fwd = layer.DecodeForward(x, L.w1q3(), L.w2q3(), offs, seed=args.seed, device=dev)
    for _ in range(max(args.warmup, 3)):
        fwd.forward()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        fwd.forward()
    b.record(stream)
    torch.cuda.synchronize()
    if pmn.get_device_error() != 0:
        raise RuntimeError("device error in the decode forward")
    ms = a.elapsed_time(b) / reps
    fl, by, wb = layer.decode_algorithmic(r.counts, L.shape.d_model, L.shape.d_ff)
    pk = peaks()
    gbs = by / (ms * 1e-3) / 1e9
    return {"workload": "decode forward: %d tokens, top-%d of %d experts (%d rows, %d experts hit, unpadded), "
                        "NVFP4 weights resident" % (W.DECODE_TOKENS, W.TOP_K, L.shape.experts, r.real_rows,
                                                    int((r.counts > 0).sum())),
            "ms": round(ms, 4), "TFLOP/s": round(fl / (ms * 1e-3) / 1e12, 2), "weight_bytes": wb,
            "algorithmic_bytes": by, "GB/s": round(gbs, 1), "hbm_frac": round(gbs / pk["hbm_gbs"], 3),
            "bound": "hbm", "reps": reps,
            "gpu_launches": sum(layer.LAUNCHES.get(n, 1) for n, _ in fwd.kernel_calls()) * reps}


def run_single_expert(args, dev, W, pmn, reps=20):
    """The single-expert forward: T = 4096 tokens (N(0,1), 0.1 % of entries
    x30) through one expert (w1 [3072, 4096], w2 [4096, 1536], N(0, 0.02)).
    Each call of the forward is timed alone with CUDA events on the launching
    stream, `reps` times, with L2 flushed (a 256 MB write) before every timed
    call, since the operands (17 MB of NVFP4) fit in L2.  The w1 GEMM at this
    shape is tensor-bound (arithmetic intensity ~2500 FLOP/B): its TFLOP/s
    against the FP4 tensor peak is the measure of the block-scaled MMA
    pipeline."""
    import numpy as np
    import torch
    d = W.expert(args.seed)
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
    x, w1, w2 = bf(d["x"]), bf(d["w1"]), bf(d["w2"])
    T, D = x.shape
    F = w2.shape[1]
    u8, f32 = torch.uint8, torch.float32
    e = lambda *shape, dtype=u8: torch.empty(shape, dtype=dtype, device=dev)
    xq = (e(T, D // 2), e(T, D // 16), e(T, dtype=f32))
    w1q = (e(2 * F, D // 2), e(2 * F, D // 16), e(1, dtype=f32))
    w2q = (e(D, F // 2), e(D, F // 16), e(1, dtype=f32))
    hq = (e(T, F // 2), e(T, F // 16), e(T, dtype=f32))
    h = e(T, F, dtype=torch.bfloat16)
    y = e(T, 2 * F, dtype=torch.bfloat16)
    z = e(T, D, dtype=torch.bfloat16)
    ws = e(pmn.nvfp4_quantize_workspace_bytes(pmn.OUTER_PER_GROUP, D, D))
    offs = torch.tensor([0, T], dtype=torch.int32, device=dev)
    w1q3 = lambda: (w1q[0].view(1, 2 * F, D // 2), w1q[1].view(1, 2 * F, D // 16), w1q[2])
    w2q3 = lambda: (w2q[0].view(1, D, F // 2), w2q[1].view(1, D, F // 16), w2q[2])
    g1, g2 = 2.0 * T * 2 * F * D, 2.0 * T * D * F
    nv = 0.5 + 1 / 16
    calls = [
        ("quant_x", lambda: pmn.nvfp4_quantize(x, four_over_six=True, out=xq), 0, T * D * (2 + nv)),
        ("quant_w1", lambda: pmn.nvfp4_quantize(w1, outer_mode=pmn.OUTER_PER_GROUP, rows_per_group=2 * F, out=w1q,
                                                workspace=ws), 0, 2 * F * D * (2 + nv)),
        ("quant_w2", lambda: pmn.nvfp4_quantize(w2, outer_mode=pmn.OUTER_PER_GROUP, rows_per_group=D, out=w2q,
                                                workspace=ws), 0, D * F * (2 + nv)),
        ("gemm1_swiglu_only", lambda: pmn.grouped_gemm_nvfp4(xq, w1q3(), offs, swiglu=True, out=h), g1,
         (T * D + 2 * F * D) * nv + T * F * 2),
        ("gemm1_swiglu_nvfp4", lambda: pmn.w1_gemm_swiglu_nvfp4(xq, w1q3(), offs, True, out=hq, h=h), g1,
         (T * D + 2 * F * D) * nv + T * F * 2 * 2 + T * F * nv),
        ("gemm1_bf16", lambda: pmn.grouped_gemm_nvfp4(xq, w1q3(), offs, out=y), g1,
         (T * D + 2 * F * D) * nv + T * 2 * F * 2),
        ("gemm2_bf16", lambda: pmn.grouped_gemm_nvfp4(hq, w2q3(), offs, out=z), g2, (T * F + D * F) * nv + T * D * 2),
    ]
    flush = torch.empty(256 << 20, dtype=u8, device=dev)
    stream = torch.cuda.current_stream()
    pk = peaks()
    fp4_peak = pk["bf16_tflops_sustained"] * NOMINAL_TC_RATIO["fp4"]
    out = {}
    for name, f, fl, by in calls:
        for _ in range(3):
            f()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for a, b in ev:
            flush.zero_()
            a.record(stream)
            f()
            b.record(stream)
        torch.cuda.synchronize()
        ms = sum(a.elapsed_time(b) for a, b in ev) / reps
        c = {"ms": round(ms, 4), "GB/s": round(by / (ms * 1e-3) / 1e9, 1),
             "hbm_frac": round(by / (ms * 1e-3) / 1e9 / pk["hbm_gbs"], 3)}
        if fl:
            c["TFLOP/s"] = round(fl / (ms * 1e-3) / 1e12, 1)
            c["tc_frac"] = round(fl / (ms * 1e-3) / 1e12 / fp4_peak, 3)
        out[name] = c
    if pmn.get_device_error() != 0:
        raise RuntimeError("device error in the single-expert forward")
    fwd_ms = out["quant_x"]["ms"] + out["gemm1_swiglu_nvfp4"]["ms"] + out["gemm2_bf16"]["ms"]
    return {"workload": "single expert forward: T=%d tokens, d_model %d, d_ff %d (w1 [%d, %d], w2 [%d, %d]); "
                        "X NVFP4 4/6 per token, weights NVFP4 per expert (quantised once, resident)"
                        % (T, D, F, 2 * F, D, D, F),
            "l2": "flushed (256 MB write) before every timed call",
            "forward_ms": round(fwd_ms, 4), "forward_TFLOP/s": round((g1 + g2) / (fwd_ms * 1e-3) / 1e12, 1),
            "fp4_peak_tflops": round(fp4_peak, 1), "reps": reps, "calls": out}


def result_line(value, world, steps, warmup, ms_step, config, roofline, cpu, e2e, launches, clocks, extra):
    """The one JSON line of the default run: the contract's keys, then the
    measurements made beside the step."""
    line = {"metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
            "steps": steps, "warmup": warmup, "ms_per_step": round(ms_step, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "nvfp4+mxfp8",
            "data": "synthetic", "config": config, "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": launches, "clocks": clocks}
    line.update(extra)
    return line


def max_over_ranks(ms_total, world, dist, device):
    """The timed region's length (ms), the maximum over the ranks: each rank
    times its own replica, and the job takes as long as the slowest."""
    import torch
    t = torch.tensor([float(ms_total)], device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.item()


def whole_job_value(flops_per_rank_step, world, ms_step):
    """Whole-job TFLOP/s: every rank's FLOPs over the slowest rank's step time."""
    return flops_per_rank_step * world / (ms_step * 1e-3) / 1e12


def run_combine(payload, r, args, dev, pmn, reps=20):
    """The combine's receive side at the step's size: the layer's S2F6
    payload (all routed rows) decoded, transformed back and summed with the
    gates into 16384 bf16 token rows.  CUDA events around `reps` calls on the
    launching stream; the payload (~0.6 GB) exceeds L2."""
    import numpy as np
    import torch
    idx = torch.from_numpy(r.token_rows()).to(dev)
    gates = torch.from_numpy(r.gates).to(dev)
    tokens, k = idx.shape
    d = payload[0].shape[1]
    out = torch.empty((tokens, d), dtype=torch.bfloat16, device=dev)
    for _ in range(max(args.warmup, 3)):
        pmn.combine_receive_s2f6(payload, args.seed, idx, gates, out=out)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        pmn.combine_receive_s2f6(payload, args.seed, idx, gates, out=out)
    b.record(stream)
    torch.cuda.synchronize()
    if pmn.get_device_error() != 0:
        raise RuntimeError("device error in the combine receive")
    ms = a.elapsed_time(b) / reps
    by = combine_algorithmic(tokens, k, d)
    gbs = by / (ms * 1e-3) / 1e9
    return {"workload": "combine receive: %d tokens x top-%d S2F6 rows of %d (+ E8M0 per 32) -> bf16 token rows"
                        % (tokens, k, d),
            "ms": round(ms, 4), "algorithmic_bytes": by, "GB/s": round(gbs, 1),
            "hbm_frac": round(gbs / peaks()["hbm_gbs"], 3), "bound": "hbm", "reps": reps, "gpu_launches": reps}


def run_mxfp8_forward(inp, r, offsets, args, layer, pmn, reps=10):
    """The layer's forward in MXFP8 (the precision of the last 16.6 % of
    layers): MXFP8 quantisation of W1, W2 (every call, as in a training step)
    and X, the grouped FP8 GEMMs, SwiGLU + MXFP8 of h.  CUDA events around
    `reps` forwards on the launching stream; weights (14.5 GB bf16) and
    activations exceed L2."""
    import torch
    fw = layer.MXFP8Forward(inp["x"], inp["w1"], inp["w2"], offsets, device=inp["x"].device)
    calls = fw.kernel_calls()
    for _ in range(max(args.warmup, 3)):
        fw.forward()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)] for _ in range(reps)]
    for i in range(reps):
        for j, (_, f) in enumerate(calls):
            ev[i][j].record(stream)
            f()
        ev[i][-1].record(stream)
    torch.cuda.synchronize()
    if pmn.get_device_error() != 0:
        raise RuntimeError("device error in the MXFP8 forward")
    ms = sum(ev[i][0].elapsed_time(ev[i][-1]) for i in range(reps)) / reps
    per = {name: round(sum(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(reps)) / reps, 4)
           for j, (name, _) in enumerate(calls)}
    E, F2, D = inp["w1"].shape
    fl, by = layer.mxfp8_forward_algorithmic(r.real_rows, E, D, F2 // 2)
    pk = peaks()
    fp8_peak = pk["bf16_tflops_sustained"] * NOMINAL_TC_RATIO["fp8"]
    gemm_ms = per["mx_gemm1"] + per["mx_gemm2"]
    del fw
    return {"workload": "MXFP8 forward of the layer (last 16.6 %% of layers): %d experts, %d routed rows, "
                        "d_model %d, d_ff %d; weights quantised every call" % (E, r.real_rows, D, F2 // 2),
            "ms": round(ms, 4), "TFLOP/s": round(fl / (ms * 1e-3) / 1e12, 1), "flops": fl, "algorithmic_bytes": by,
            "GB/s": round(by / (ms * 1e-3) / 1e9, 1), "hbm_frac": round(by / (ms * 1e-3) / 1e9 / pk["hbm_gbs"], 3),
            "gemm_TFLOP/s": round(fl / (gemm_ms * 1e-3) / 1e12, 1),
            "gemm_tc_frac": round(fl / (gemm_ms * 1e-3) / 1e12 / fp8_peak, 3),
            "calls_ms": per, "reps": reps, "gpu_launches": len(calls) * reps}


def run_fp4_requant(L, args, pmn, reps=10):
    """The FP4 backward's requantisations at the step's size: the step's saved
    NVFP4 X, H (per token) and W1, W2 (per expert) dequantised, transposed and
    requantised to NVFP4 with stochastic rounding, as the step's MXFP8
    requantisations do.  CUDA events per call over `reps` passes on the
    launching stream; every tensor exceeds L2 or streams past it."""
    import torch
    E, F2, D = L.w1.shape
    F, T = F2 // 2, L.shape.rows
    outs = {}

    def buf(batch, rows, cols):
        return (torch.empty((batch, cols, rows // 2), dtype=torch.uint8, device=L.x.device),
                torch.empty((batch, cols, rows // 16), dtype=torch.uint8, device=L.x.device),
                torch.empty((batch,), dtype=torch.float32, device=L.x.device))

    calls = [("fp4_requant_x", (L.xq, True, 1, T, D, pmn.TAG_X)), ("fp4_requant_h", (L.hq, True, 1, T, F, pmn.TAG_H)),
             ("fp4_requant_w1", (L.w1q, False, E, F2, D, pmn.TAG_W1)),
             ("fp4_requant_w2", (L.w2q, False, E, D, F, pmn.TAG_W2))]
    for name, (src, per_row, batch, rows, cols, tag) in calls:
        outs[name] = buf(batch, rows, cols)

    def run(name, src, per_row, batch, rows, cols, tag):
        pmn.requant_transpose_sr_nvfp4(src[0], src[1], src[2], per_row, batch, rows, cols, args.seed, tag,
                                       out=outs[name])

    for _ in range(max(args.warmup, 3)):
        for name, a in calls:
            run(name, *a)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)] for _ in range(reps)]
    for i in range(reps):
        for j, (name, a) in enumerate(calls):
            ev[i][j].record(stream)
            run(name, *a)
        ev[i][-1].record(stream)
    torch.cuda.synchronize()
    if pmn.get_device_error() != 0:
        raise RuntimeError("device error in the FP4 requantisation")
    nv = 0.5 + 1 / 16
    R = L.shape.real_rows
    elems = {"fp4_requant_x": R * D, "fp4_requant_h": R * F, "fp4_requant_w1": E * F2 * D,
             "fp4_requant_w2": E * D * F}
    pk = peaks()
    res = {}
    for j, (name, _) in enumerate(calls):
        ms = sum(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(reps)) / reps
        by = elems[name] * 2 * nv
        res[name] = {"ms": round(ms, 4), "GB/s": round(by / (ms * 1e-3) / 1e9, 1),
                     "hbm_frac": round(by / (ms * 1e-3) / 1e9 / pk["hbm_gbs"], 3)}
    del outs
    return {"workload": "NVFP4 -> transposed NVFP4 with stochastic rounding (FP4 backward) of the step's "
                        "saved X, H, W1, W2", "calls": res, "reps": reps, "gpu_launches": 3 * len(calls) * reps}


def combine_algorithmic(tokens, k, d):
    """Bytes the combine receive must move: each routed row's S2F6 bytes and
    scales read once, the index and gate of every choice, the bf16 token rows
    written."""
    return tokens * k * (d + d // 32 + 8) + tokens * d * 2


def run_e2e(L, inp, args, dev, flops_step, world):
    """Same step through the binding with host buffers: every step copies the
    batch inputs (routed X, dY, dY1) from pinned host memory and reads back the
    forward result (S2F6 combine payload + scales) and dX.  Steps are
    pipelined over two sets of device input/output buffers: the host->device
    copies of step i+1 (one copy stream) and the device->host copies of step
    i-1 (another) run while step i computes.  The timed region opens before
    the first step's input copies and closes after the last step's results
    have landed in host memory."""
    import torch
    keys = ("x", "dy", "dy1")
    pins = {k: torch.empty_like(inp[k], device="cpu").pin_memory() for k in keys}
    for k in pins:
        pins[k].copy_(inp[k])
    # two device buffer sets (set 0 is the layer's own)
    dev_in = [{k: getattr(L, k) for k in keys}, {k: torch.empty_like(getattr(L, k)) for k in keys}]
    dev_out = [(L.z, L.dx), ((torch.empty_like(L.z[0]), torch.empty_like(L.z[1])), torch.empty_like(L.dx))]
    outs = [[torch.empty_like(L.z[0], device="cpu").pin_memory(), torch.empty_like(L.z[1], device="cpu").pin_memory(),
             torch.empty_like(L.dx, device="cpu").pin_memory()] for _ in range(2)]
    bi = sum(p.numel() * p.element_size() for p in pins.values())
    bo = sum(o.numel() * o.element_size() for o in outs[0])
    comp = torch.cuda.current_stream()
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()

    def run(nsteps, start=None):
        in_free = [None, None]   # compute finished reading set b
        out_free = [None, None]  # host copies of set b's results finished
        in_ready = [None, None]
        last = []
        for i in range(nsteps + 1):
            # issue the input copies of step i, then compute step i - 1
            if i < nsteps:
                b = i % 2
                with torch.cuda.stream(h2d):
                    if start is not None and i == 0:
                        h2d.wait_event(start)
                    if in_free[b] is not None:
                        h2d.wait_event(in_free[b])
                    for k in keys:
                        dev_in[b][k].copy_(pins[k], non_blocking=True)
                    in_ready[b] = ev()
                    in_ready[b].record(h2d)
            if i >= 1:
                j = i - 1
                b = j % 2
                comp.wait_event(in_ready[b])
                if out_free[b] is not None:
                    comp.wait_event(out_free[b])
                for k in keys:
                    setattr(L, k, dev_in[b][k])
                L.z, L.dx = dev_out[b]
                L.step()
                in_free[b] = ev()
                in_free[b].record(comp)
                with torch.cuda.stream(d2h):
                    d2h.wait_event(in_free[b])
                    o = outs[b]
                    o[0].copy_(L.z[0], non_blocking=True)
                    o[1].copy_(L.z[1], non_blocking=True)
                    o[2].copy_(L.dx, non_blocking=True)
                    out_free[b] = ev()
                    out_free[b].record(d2h)
                last.append(out_free[b])
        for e in last[-2:]:
            comp.wait_event(e)

    run(2)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(comp)
    run(args.steps, start=a)
    b.record(comp)
    torch.cuda.synchronize()
    for k in keys:  # leave the layer on its own buffers
        setattr(L, k, dev_in[0][k])
    L.z, L.dx = dev_out[0]
    ms = a.elapsed_time(b) / args.steps
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = t.item()
    return {"value": round(flops_step * world / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s", "ms_per_step": round(ms, 3),
            "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "pipelined": "copies of step i+1 / i-1 overlap step i"}


def cpu_baseline(inp, args, budget_s=12.0):
    r = inp["routing"]
    k = 1
    flops, dt, threads = oracle_sample(inp, pick_sample_experts(r, 1), args.seed)
    # grow the sample to about `budget_s` of CPU work
    per = dt
    k = max(1, min(48, int(budget_s / max(per, 1e-3))))
    experts = pick_sample_experts(r, k)
    flops, dt, threads = oracle_sample(inp, experts, args.seed)
    # the same step on one thread, over one expert
    import oracle
    one = pick_sample_experts(r, 1)
    oracle.set_num_threads(1)
    try:
        f1, t1, _ = oracle_sample(inp, one, args.seed)
    finally:
        oracle.set_num_threads(threads)
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": "the full step (quantise, GEMMs in binary64, SwiGLU, RHT+S2F6, SR requant, dY quant, "
                      "gradient GEMMs) for %d of %d experts (%d routed rows), %.1f s" % (
                          len(experts), len(r.counts), int(sum(r.counts[e] for e in experts)), dt),
            "single_thread": {"value": round(f1 / t1 / 1e12, 6), "cores": 1,
                              "sample": "the same step for 1 expert (%d routed rows), %.1f s" % (
                                  int(r.counts[one[0]]), t1)}}


def run_reference(args):
    """The oracle timed as the reference arm: each step is the oracle's pass
    over a bounded sample of experts of the same workload (host inputs drawn
    with the same seeded generator on the host)."""
    import numpy as np
    import torch
    from precision_moe_numerics_gb300 import workloads as W
    r = W.moe_routing(args.seed)
    k = 2
    experts = pick_sample_experts(r, k)
    rng_dev = "cpu"
    gen = torch.Generator(device=rng_dev)
    gen.manual_seed(args.seed + 100)
    D, F = W.D_MODEL, W.D_FF
    inputs = {"routing": r}
    rows = r.rows
    x = torch.zeros((rows, D), dtype=torch.bfloat16)
    dy = torch.zeros((rows, D), dtype=torch.bfloat16)
    dy1 = torch.zeros((rows, 2 * F), dtype=torch.bfloat16)
    w1 = torch.zeros((r.counts.size, 2 * F, D), dtype=torch.bfloat16)
    w2 = torch.zeros((r.counts.size, D, F), dtype=torch.bfloat16)
    for e in experts:
        lo, hi = int(r.offsets[e]), int(r.offsets[e + 1])
        real = int(r.counts[e])
        x[lo:lo + real] = W.normal_bf16_device(gen, (real, D), 1.0, 0.001, 30.0, device=rng_dev)
        dy[lo:lo + real] = W.normal_bf16_device(gen, (real, D), 1e-3, device=rng_dev)
        dy1[lo:lo + real] = W.normal_bf16_device(gen, (real, 2 * F), 1e-3, device=rng_dev)
        w1[e] = W.normal_bf16_device(gen, (2 * F, D), 0.02, device=rng_dev)
        w2[e] = W.normal_bf16_device(gen, (D, F), 0.02, device=rng_dev)
    inputs.update({"x": x, "dy": dy, "dy1": dy1, "w1": w1, "w2": w2})
    for _ in range(args.warmup):
        oracle_sample(inputs, experts, args.seed)
    tot_f, tot_t, threads = 0.0, 0.0, 1
    for _ in range(args.steps):
        f, t, threads = oracle_sample(inputs, experts, args.seed)
        tot_f += f
        tot_t += t
    value = tot_f / tot_t / 1e12
    sample = "the full step for %d of 384 experts (%d routed rows) per step" % (
        len(experts), int(sum(r.counts[e] for e in experts)))
    line = {"metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(tot_t / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 GEMMs, f32 quantisers",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": WORKLOAD, "sample_experts": experts},
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


if __name__ == "__main__":
    main()
