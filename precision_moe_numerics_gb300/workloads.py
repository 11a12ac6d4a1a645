"""Seeded synthetic inputs for the expert-layer workloads.

This module only draws random numbers and lays them out; it holds none of the
quantisation arithmetic, so both the CUDA path and the CPU oracle can be fed
from it.  All draws are seeded.  Small cases are drawn on the host with numpy's
PCG64; full-size cases are drawn on the device with torch's seeded CUDA
generator, and the oracle reads sampled rows of them.

Workloads (shapes of the pages' MoE layer: 384 experts, top-8, d_model 4096,
expert d_ff 1536):
  tiny      X 256x256 ~ N(0,1), 4 rows x50; B 256x256 ~ N(0,1) for a 256^3 GEMM
  expert    T=4096 tokens ~ N(0,1) with 0.1 % entries x30; w1 [3072,4096] and
            w2 [4096,1536] ~ N(0, 0.02^2)
  moe       16384 tokens, logits [16384,384] ~ N(0,1), top-8 (ties to the lower
            expert), routed rows sorted by expert then token, every expert
            segment padded with zero rows to a multiple of 128; 384 experts of
            w1/w2 as above
  backward  the moe layout plus dY [rows,4096] and dY1 [rows,3072] ~ N(0,1e-3^2)
  decode    64 tokens, top-8 -> 512 rows over the distinct experts hit
"""
from dataclasses import dataclass

import numpy as np
import torch

D_MODEL = 4096
D_FF = 1536
N_EXPERTS = 384
TOP_K = 8
MOE_TOKENS = 16384
DECODE_TOKENS = 64
PAD = 128  # expert segments: whole 128-deep K stages for the weight-gradient GEMMs


def f32_to_bf16_bits(a):
    """Cast binary32 -> bfloat16 (round to nearest even) and return uint16 bits."""
    t = torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_bf16_host(rng, shape, std=1.0, outlier_p=0.0, outlier_mult=1.0):
    x = rng.standard_normal(shape, dtype=np.float32) * np.float32(std)
    if outlier_p > 0:
        mask = rng.random(shape, dtype=np.float32) < outlier_p
        x = np.where(mask, x * np.float32(outlier_mult), x)
    return f32_to_bf16_bits(x)


def normal_bf16_device(gen, shape, std=1.0, outlier_p=0.0, outlier_mult=1.0, device="cuda", out=None):
    """Seeded draw straight into a device bf16 tensor (generator `gen` on `device`)."""
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    if outlier_p > 0:
        m = torch.rand(shape, generator=gen, device=device, dtype=torch.float32) < outlier_p
        x = torch.where(m, x * outlier_mult, x)
    if out is None:
        return x.to(torch.bfloat16)
    out.copy_(x)
    return out


# ------------------------------------------------------------------ routing
@dataclass
class Routing:
    """Routed-row layout: rows of expert e are offsets[e]..offsets[e+1]
    (padded to a multiple of `pad`); counts[e] real rows; row_token[i] is the
    token of routed row i, -1 for a padding row."""
    offsets: np.ndarray      # int64 [E+1]
    counts: np.ndarray       # int64 [E]
    row_token: np.ndarray    # int64 [rows]
    topk: np.ndarray         # int64 [tokens, k]
    gates: np.ndarray = None  # float32 [tokens, k]: softmax over the k chosen logits

    @property
    def rows(self):
        return int(self.offsets[-1])

    @property
    def real_rows(self):
        return int(self.counts.sum())

    def token_rows(self):
        """int32 [tokens, k]: the routed row that holds token t's i-th choice
        (the inverse of row_token, in the order of topk)."""
        tokens, k = self.topk.shape
        r = np.nonzero(self.row_token >= 0)[0]
        t = self.row_token[r]
        e = np.searchsorted(self.offsets, r, side="right") - 1
        slot = (self.topk[t] == e[:, None]).argmax(axis=1)
        out = np.full((tokens, k), -1, np.int64)
        out[t, slot] = r
        return out.astype(np.int32)


def route_topk(logits, k=TOP_K, pad=PAD):
    """top-k experts per token (ties to the lower index; the softmax is
    monotone so the top-k of the logits is the top-k of the probabilities)."""
    tokens, E = logits.shape
    order = np.argsort(-logits, axis=1, kind="stable")[:, :k]
    counts = np.bincount(order.reshape(-1), minlength=E).astype(np.int64)
    padded = ((counts + pad - 1) // pad) * pad if pad > 1 else counts
    offsets = np.zeros(E + 1, np.int64)
    offsets[1:] = np.cumsum(padded)
    row_token = np.full(offsets[-1], -1, np.int64)
    # rows sorted by expert, then token
    flat_e = order.reshape(-1)
    flat_t = np.repeat(np.arange(tokens), k)
    srt = np.lexsort((flat_t, flat_e))
    fill = offsets[:-1].copy()
    for e, t in zip(flat_e[srt], flat_t[srt]):
        row_token[fill[e]] = t
        fill[e] += 1
    sel = np.take_along_axis(logits, order, axis=1).astype(np.float64)
    ex = np.exp(sel - sel[:, :1])
    gates = (ex / ex.sum(axis=1, keepdims=True)).astype(np.float32)
    return Routing(offsets, counts, row_token, order.astype(np.int64), gates)


def moe_routing(seed=0, tokens=MOE_TOKENS, experts=N_EXPERTS, k=TOP_K, pad=PAD):
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((tokens, experts), dtype=np.float32)
    return route_topk(logits, k, pad)


def decode_routing(seed=0):
    rng = np.random.default_rng(seed + 4)
    logits = rng.standard_normal((DECODE_TOKENS, N_EXPERTS), dtype=np.float32)
    return route_topk(logits, TOP_K, pad=1)


def decode_x(routing, seed=0, d=D_MODEL):
    """bf16 bits of the decode batch's routed rows [rows, d]: the tokens ~
    N(0,1) with 0.1 % entries x30, row i a copy of token row_token[i]."""
    rng = np.random.default_rng(seed + 5)
    xt = normal_bf16_host(rng, (DECODE_TOKENS, d), 1.0, 0.001, 30.0)
    return xt[routing.row_token]


def combine_payload(rows, d=D_MODEL, seed=0):
    """A seeded combine payload in the shape the w2 epilogue emits: int8
    S2F6 bytes [rows, d] (k ~ round(N(0, 42^2)) clipped to +-127, so a block's
    largest |k| is near the top of the range, as the epilogue's scale rule
    makes it) and E8M0 bytes [rows, d/32] between 2^-9 and 2^2."""
    rng = np.random.default_rng(seed + 6)
    q = np.clip(np.rint(rng.standard_normal((rows, d), dtype=np.float32) * 42.0), -127, 127).astype(np.int8)
    sc = rng.integers(118, 130, (rows, d // 32)).astype(np.uint8)
    return q, sc


# ------------------------------------------------------------------ host cases
def tiny(seed=0, n=256, outlier_rows=4, outlier_mult=50.0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n, n), dtype=np.float32)
    rows = rng.choice(n, size=outlier_rows, replace=False)
    x[rows] *= np.float32(outlier_mult)
    b = rng.standard_normal((n, n), dtype=np.float32)
    return {"x": f32_to_bf16_bits(x), "b": f32_to_bf16_bits(b), "outlier_rows": np.sort(rows)}


def expert(seed=0, tokens=4096, d=D_MODEL, f=D_FF):
    rng = np.random.default_rng(seed + 1)
    x = normal_bf16_host(rng, (tokens, d), 1.0, 0.001, 30.0)
    w1 = normal_bf16_host(rng, (2 * f, d), 0.02)
    w2 = normal_bf16_host(rng, (d, f), 0.02)
    return {"x": x, "w1": w1, "w2": w2}


def small_moe(seed=0, tokens=256, experts=8, k=2, d=256, f=128, pad=PAD):
    """A scaled-down MoE layout (ragged expert segments, some possibly empty)
    used for parity tests the oracle finishes in seconds."""
    rng = np.random.default_rng(seed + 7)
    logits = rng.standard_normal((tokens, experts), dtype=np.float32)
    logits[:, 0] -= 4.0  # make expert 0 rare (ragged, possibly empty)
    r = route_topk(logits, k, pad)
    xt = normal_bf16_host(rng, (tokens, d), 1.0, 0.001, 30.0)
    x = np.zeros((r.rows, d), np.uint16)
    m = r.row_token >= 0
    x[m] = xt[r.row_token[m]]
    w1 = normal_bf16_host(rng, (experts, 2 * f, d), 0.02)
    w2 = normal_bf16_host(rng, (experts, d, f), 0.02)
    dy = normal_bf16_host(rng, (r.rows, d), 1e-3)
    dy[~m] = 0
    dy1 = normal_bf16_host(rng, (r.rows, 2 * f), 1e-3)
    dy1[~m] = 0
    return {"routing": r, "x": x, "w1": w1, "w2": w2, "dy": dy, "dy1": dy1}


# ------------------------------------------------------------------ device cases
def moe_device(seed=0, device="cuda", with_backward=True, experts=N_EXPERTS, tokens=MOE_TOKENS,
               d=D_MODEL, f=D_FF, align_rows=512):
    """Full-size MoE layer inputs drawn on the device (bf16 tensors).  Row
    buffers hold `rows_alloc` rows (the routed rows rounded up to
    `align_rows`); rows past the last expert segment are zero."""
    r = moe_routing(seed, tokens, experts, k=min(TOP_K, experts))
    rows_alloc = ((r.rows + align_rows - 1) // align_rows) * align_rows
    gen = torch.Generator(device=device)
    gen.manual_seed(seed + 100)
    xt = normal_bf16_device(gen, (tokens, d), 1.0, 0.001, 30.0, device)
    rt = torch.full((rows_alloc,), -1, dtype=torch.int64, device=device)
    rt[:r.rows] = torch.from_numpy(r.row_token).to(device)
    x = torch.zeros((rows_alloc, d), dtype=torch.bfloat16, device=device)
    m = rt >= 0
    x[m] = xt[rt[m]]
    del xt
    w1 = torch.empty((experts, 2 * f, d), dtype=torch.bfloat16, device=device)
    w2 = torch.empty((experts, d, f), dtype=torch.bfloat16, device=device)
    for e in range(experts):
        normal_bf16_device(gen, (2 * f, d), 0.02, device=device, out=w1[e])
        normal_bf16_device(gen, (d, f), 0.02, device=device, out=w2[e])
    out = {"routing": r, "x": x, "w1": w1, "w2": w2, "rows_alloc": rows_alloc}
    if with_backward:
        dy = normal_bf16_device(gen, (rows_alloc, d), 1e-3, device=device)
        dy[~m] = 0
        dy1 = normal_bf16_device(gen, (rows_alloc, 2 * f), 1e-3, device=device)
        dy1[~m] = 0
        out["dy"] = dy
        out["dy1"] = dy1
    return out
