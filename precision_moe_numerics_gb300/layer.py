"""One pass of the MoE expert layer's block-scaled numerics path on one GPU.

Forward (page "Thinking Machines ... Inkling 2 Small", sections [Layers],
[Cost], [NVLink]):
  W1, W2 (bf16 master weights)  -> NVFP4, outer scale per expert
  X (routed rows, bf16)         -> NVFP4, outer scale per token, 4/6
  H  = silu(Y_gate) * Y_up,     grouped NVFP4 GEMM with SwiGLU in its
       Y = X . W1^T             epilogue (bf16 h), then NVFP4 of h per token,
                                4/6 (one call, two kernels)
  Z  = H . W2^T                 grouped NVFP4 GEMM with the RHT-32 + S2F6
                                combine quantisation in its epilogue
Backward (section [SR]):
  saved X, H, W1, W2 (NVFP4)    -> dequantise, transpose, SR -> MXFP8
  dY, dY1 (bf16)                -> MXFP8 (RN), rowwise and transposed
  dH  = dY  . W2                M-grouped MXFP8 GEMM -> bf16
  dW2 = dY^T . H  per expert    K-grouped MXFP8 GEMM -> fp32
  dX  = dY1 . W1                M-grouped MXFP8 GEMM -> bf16
  dW1 = dY1^T . X per expert    K-grouped MXFP8 GEMM -> fp32

All buffers are allocated once (torch, device memory); step() only enqueues
the library's kernels on the current stream.
"""
from dataclasses import dataclass

import torch

from . import pmn

ALIGN_ROWS = 512  # routed-row buffers are padded so MXFP8 scale rows are 16-byte pitched


@dataclass
class LayerShape:
    experts: int
    d_model: int
    d_ff: int
    rows: int        # allocated routed rows (multiple of ALIGN_ROWS)
    real_rows: int   # routed (token, expert) pairs


def flops_forward(s: LayerShape):
    return 2.0 * s.real_rows * s.d_model * (2 * s.d_ff) + 2.0 * s.real_rows * s.d_ff * s.d_model


def flops_backward(s: LayerShape):
    # dX, dW1 (w1 layer) and dH, dW2 (w2 layer): two GEMMs of each forward shape
    return 2.0 * flops_forward(s)


class ExpertLayerStep:
    def __init__(self, x, w1, w2, dy, dy1, offsets, real_rows, seed=0, device="cuda"):
        E, F2, D = w1.shape
        F = F2 // 2
        T = x.shape[0]
        assert T % ALIGN_ROWS == 0 and w2.shape == (E, D, F)
        self.shape = LayerShape(E, D, F, T, real_rows)
        self.x, self.w1, self.w2, self.dy, self.dy1 = x, w1, w2, dy, dy1
        self.offsets = offsets
        self.seed = seed
        u8, f32, bf16 = torch.uint8, torch.float32, torch.bfloat16

        def e(*shape, dtype=u8):
            return torch.empty(shape, dtype=dtype, device=device)

        # scratch of the per-expert weight quantiser (caller-owned workspace)
        self.ws = e(max(pmn.nvfp4_quantize_workspace_bytes(pmn.OUTER_PER_GROUP, E * F2, F2),
                        pmn.nvfp4_quantize_workspace_bytes(pmn.OUTER_PER_GROUP, E * D, D)))
        # forward operands
        self.w1q = (e(E * F2, D // 2), e(E * F2, D // 16), e(E, dtype=f32))
        self.w2q = (e(E * D, F // 2), e(E * D, F // 16), e(E, dtype=f32))
        self.xq = (e(T, D // 2), e(T, D // 16), e(T, dtype=f32))
        self.h = e(T, F, dtype=bf16)
        self.hq = (e(T, F // 2), e(T, F // 16), e(T, dtype=f32))
        self.z = (e(T, D, dtype=torch.int8), e(T, D // 32))
        # backward operands
        self.xt = (e(1, D, T), e(1, D, T // 32))
        self.ht = (e(1, F, T), e(1, F, T // 32))
        self.w1t = (e(E, D, F2), e(E, D, F2 // 32))
        self.w2t = (e(E, F, D), e(E, F, D // 32))
        self.dy_r = (e(T, D), e(T, D // 32))
        self.dy_t = (e(D, T), e(D, T // 32))
        self.dy1_r = (e(T, F2), e(T, F2 // 32))
        self.dy1_t = (e(F2, T), e(F2, T // 32))
        self.dh = e(T, F, dtype=bf16)
        self.dx = e(T, D, dtype=bf16)
        self.dw1 = e(E, F2, D, dtype=f32)
        self.dw2 = e(E, D, F, dtype=f32)

    def w1q3(self):
        E, F2, D = self.w1.shape
        c, s, g = self.w1q
        return c.view(E, F2, D // 2), s.view(E, F2, D // 16), g

    def w2q3(self):
        E, D, F = self.w2.shape
        c, s, g = self.w2q
        return c.view(E, D, F // 2), s.view(E, D, F // 16), g

    def kernel_calls(self):
        """(name, callable) pairs in step order; each call enqueues library kernels."""
        s = self.shape
        E, D, F, T = s.experts, s.d_model, s.d_ff, s.rows
        F2 = 2 * F
        P = pmn
        return [
            ("quant_w1", lambda: P.nvfp4_quantize(self.w1.view(E * F2, D), outer_mode=P.OUTER_PER_GROUP,
                                                  rows_per_group=F2, out=self.w1q, workspace=self.ws)),
            ("quant_w2", lambda: P.nvfp4_quantize(self.w2.view(E * D, F), outer_mode=P.OUTER_PER_GROUP,
                                                  rows_per_group=D, out=self.w2q, workspace=self.ws)),
            ("quant_x", lambda: P.nvfp4_quantize(self.x, four_over_six=True, out=self.xq)),
            ("gemm1_swiglu_nvfp4", lambda: P.w1_gemm_swiglu_nvfp4(self.xq, self.w1q3(), self.offsets, True,
                                                                  out=self.hq, h=self.h)),
            ("gemm2_nvfp4_rht_s2f6", lambda: P.w2_gemm_rht_s2f6(self.hq, self.w2q3(), self.offsets, self.seed,
                                                                out=self.z)),
            ("requant_x", lambda: P.requant_transpose_sr_mxfp8(*self.xq, True, 1, T, D, self.seed, P.TAG_X,
                                                               out=self.xt)),
            ("requant_h", lambda: P.requant_transpose_sr_mxfp8(*self.hq, True, 1, T, F, self.seed, P.TAG_H,
                                                               out=self.ht)),
            ("requant_w1", lambda: P.requant_transpose_sr_mxfp8(*self.w1q, False, E, F2, D, self.seed, P.TAG_W1,
                                                                out=self.w1t)),
            ("requant_w2", lambda: P.requant_transpose_sr_mxfp8(*self.w2q, False, E, D, F, self.seed, P.TAG_W2,
                                                                out=self.w2t)),
            # both orientations of each gradient in one pass (rowwise for dH / dX,
            # transposed for the weight gradients)
            ("quant_dy", lambda: P.mxfp8_quantize_both(self.dy, out=self.dy_r, out_t=self.dy_t)),
            ("quant_dy1", lambda: P.mxfp8_quantize_both(self.dy1, out=self.dy1_r, out_t=self.dy1_t)),
            ("gemm_dh_mxfp8", lambda: P.gemm_mxfp8(self.dy_r[0], self.dy_r[1], self.w2t[0], self.w2t[1],
                                                   self.offsets, P.GROUP_M, torch.bfloat16, out=self.dh)),
            ("gemm_dw2_mxfp8", lambda: P.gemm_mxfp8(self.dy_t[0], self.dy_t[1], self.ht[0][0], self.ht[1][0],
                                                    self.offsets, P.GROUP_K, torch.float32, out=self.dw2)),
            ("gemm_dx_mxfp8", lambda: P.gemm_mxfp8(self.dy1_r[0], self.dy1_r[1], self.w1t[0], self.w1t[1],
                                                   self.offsets, P.GROUP_M, torch.bfloat16, out=self.dx)),
            ("gemm_dw1_mxfp8", lambda: P.gemm_mxfp8(self.dy1_t[0], self.dy1_t[1], self.xt[0][0], self.xt[1][0],
                                                    self.offsets, P.GROUP_K, torch.float32, out=self.dw1)),
        ]

    def step(self):
        for _, f in self.kernel_calls():
            f()


class DecodeForward:
    """The forward pass of a decode batch: a few tokens routed top-k over the
    experts (segments of a few rows, not padded), against NVFP4 weights of
    every expert already resident in HBM (e.g. an ExpertLayerStep's w1q3() and
    w2q3()).  Its time is set by streaming the hit experts' weights."""

    def __init__(self, x, w1q3, w2q3, offsets, seed=0, device="cuda"):
        T, D = x.shape
        E, F2 = w1q3[0].shape[0], w1q3[0].shape[1]
        F = F2 // 2
        self.x, self.w1q3, self.w2q3, self.offsets, self.seed = x, w1q3, w2q3, offsets, seed
        u8, f32 = torch.uint8, torch.float32

        def e(*shape, dtype=u8):
            return torch.empty(shape, dtype=dtype, device=device)

        self.xq = (e(T, D // 2), e(T, D // 16), e(T, dtype=f32))
        self.h = e(T, F, dtype=torch.bfloat16)
        self.hq = (e(T, F // 2), e(T, F // 16), e(T, dtype=f32))
        self.z = (e(T, D, dtype=torch.int8), e(T, D // 32))
        self.F = F

    def kernel_calls(self):
        P = pmn
        return [
            ("quant_x", lambda: P.nvfp4_quantize(self.x, four_over_six=True, out=self.xq)),
            ("gemm1_swiglu_nvfp4", lambda: P.w1_gemm_swiglu_nvfp4(self.xq, self.w1q3, self.offsets, True,
                                                                  out=self.hq, h=self.h)),
            ("gemm2_nvfp4_rht_s2f6", lambda: P.w2_gemm_rht_s2f6(self.hq, self.w2q3, self.offsets, self.seed,
                                                                out=self.z)),
        ]

    def forward(self):
        for _, f in self.kernel_calls():
            f()


class MXFP8Forward:
    """The expert layer's forward in MXFP8, the precision the pages keep for
    the last 16.6 % of layers [Cost]: X, W1 and W2 quantised to MXFP8 with
    round to nearest (E8M0 per 32 along the contraction), both grouped GEMMs
    on the block-scaled FP8 tensor cores with bf16 outputs, and SwiGLU +
    MXFP8 of h between them.  The weights are quantised on every call, as in
    a training step.  x: bf16 [rows, D] routed rows; w1 bf16 [E, 2F, D];
    w2 bf16 [E, D, F]; offsets: device int32 [E+1]."""

    def __init__(self, x, w1, w2, offsets, device="cuda"):
        T, D = x.shape
        E, F2, _ = w1.shape
        F = F2 // 2
        self.x, self.w1, self.w2, self.offsets = x, w1, w2, offsets
        self.E, self.D, self.F = E, D, F
        u8, bf16 = torch.uint8, torch.bfloat16

        def e(*shape, dtype=u8):
            return torch.empty(shape, dtype=dtype, device=device)

        self.w1q = (e(E * F2, D), e(E * F2, D // 32))
        self.w2q = (e(E * D, F), e(E * D, F // 32))
        self.xq = (e(T, D), e(T, D // 32))
        self.y = e(T, F2, dtype=bf16)
        self.hq = (e(T, F), e(T, F // 32))
        self.z = e(T, D, dtype=bf16)

    def kernel_calls(self):
        P = pmn
        E, D, F = self.E, self.D, self.F
        return [
            ("mx_quant_w1", lambda: P.mxfp8_quantize(self.w1.view(E * 2 * F, D), out=self.w1q)),
            ("mx_quant_w2", lambda: P.mxfp8_quantize(self.w2.view(E * D, F), out=self.w2q)),
            ("mx_quant_x", lambda: P.mxfp8_quantize(self.x, out=self.xq)),
            ("mx_gemm1", lambda: P.gemm_mxfp8(self.xq[0], self.xq[1], self.w1q[0].view(E, 2 * F, D),
                                              self.w1q[1].view(E, 2 * F, D // 32), self.offsets, P.GROUP_M,
                                              torch.bfloat16, out=self.y)),
            ("mx_swiglu_quant_h", lambda: P.mxfp8_quantize_swiglu(self.y, out=self.hq)),
            ("mx_gemm2", lambda: P.gemm_mxfp8(self.hq[0], self.hq[1], self.w2q[0].view(E, D, F),
                                              self.w2q[1].view(E, D, F // 32), self.offsets, P.GROUP_M,
                                              torch.bfloat16, out=self.z)),
        ]

    def forward(self):
        for _, f in self.kernel_calls():
            f()


def mxfp8_forward_algorithmic(real_rows, experts, d_model, d_ff):
    """(flops, algorithmic HBM bytes) of MXFP8Forward on the real routed rows:
    bf16 weights and X read once, their MXFP8 copies written and read once,
    Y and h round trips, the bf16 output written."""
    mx = 1 + 1 / 32
    R, E, D, F2 = real_rows, experts, d_model, 2 * d_ff
    w = E * (F2 * D + D * d_ff)
    by = w * (2 + 2 * mx) + R * D * (2 + 2 * mx) + R * F2 * 2 * 2 + R * d_ff * 2 * mx + R * D * 2
    flops = 2.0 * R * F2 * D + 2.0 * R * D * d_ff
    return flops, by


def decode_algorithmic(counts, d_model, d_ff):
    """(flops, algorithmic HBM bytes) of DecodeForward: the hit experts'
    NVFP4 weights (codes, scales, outer scale) dominate the bytes."""
    nv = 0.5 + 1 / 16
    R = int(counts.sum())
    hit = int((counts > 0).sum())
    F2 = 2 * d_ff
    wbytes = hit * ((F2 * d_model + d_model * d_ff) * nv + 8)
    # X in and its NVFP4 out; h (bf16) written and read; h NVFP4 written and read; the payload written
    act = R * d_model * (2 + nv) + R * d_ff * 2 * 2 + R * d_ff * nv * 2 + R * d_model * (1 + 1 / 32)
    flops = 2.0 * R * F2 * d_model + 2.0 * R * d_model * d_ff
    return flops, wbytes + act, wbytes


# launches of library kernels per call name (for the launch count); a call
# not listed launches one kernel (the scratch clear of the per-group weight
# quantiser is a memset, not a kernel of the library)
LAUNCHES = {"gemm1_swiglu_nvfp4": 2}  # the GEMM with the SwiGLU epilogue, then the NVFP4 coding of h
STEP_CALLS = ["quant_w1", "quant_w2", "quant_x", "gemm1_swiglu_nvfp4", "gemm2_nvfp4_rht_s2f6",
              "requant_x", "requant_h", "requant_w1", "requant_w2", "quant_dy", "quant_dy1",
              "gemm_dh_mxfp8", "gemm_dw2_mxfp8", "gemm_dx_mxfp8",
              "gemm_dw1_mxfp8"]


def launches_per_step():
    return sum(LAUNCHES.get(n, 1) for n in STEP_CALLS)


def algorithmic(shape: LayerShape):
    """Per call: (flops, algorithmic HBM bytes) on real rows (padding excluded)."""
    E, D, F, R = shape.experts, shape.d_model, shape.d_ff, shape.real_rows
    F2 = 2 * F
    nv = 0.5 + 1 / 16      # NVFP4 bytes per element (codes + E4M3 scales)
    mx = 1 + 1 / 32        # MXFP8 / S2F6 bytes per element (values + E8M0 scales)
    w1n, w2n = E * F2 * D, E * D * F
    out = {
        "quant_w1": (0, w1n * (2 + nv)),
        "quant_w2": (0, w2n * (2 + nv)),
        "quant_x": (0, R * D * (2 + nv)),
        # X and W1 (NVFP4) read; bf16 h written by the GEMM and read by the coding kernel; NVFP4 h written
        "gemm1_swiglu_nvfp4": (2.0 * R * F2 * D, (R * D + w1n) * nv + R * F * 2 * 2 + R * F * nv),
        "gemm2_nvfp4_rht_s2f6": (2.0 * R * D * F, (R * F + w2n) * nv + R * D * mx),
        "requant_x": (0, R * D * (nv + mx)),
        "requant_h": (0, R * F * (nv + mx)),
        "requant_w1": (0, w1n * (nv + mx)),
        "requant_w2": (0, w2n * (nv + mx)),
        "quant_dy": (0, R * D * (2 + 2 * mx)),      # bf16 read once, both MXFP8 orientations written
        "quant_dy1": (0, R * F2 * (2 + 2 * mx)),
        "gemm_dh_mxfp8": (2.0 * R * D * F, (R * D + w2n) * mx + R * F * 2),
        "gemm_dw2_mxfp8": (2.0 * R * D * F, (R * D + R * F) * mx + w2n * 4),
        "gemm_dx_mxfp8": (2.0 * R * F2 * D, (R * F2 + w1n) * mx + R * D * 2),
        "gemm_dw1_mxfp8": (2.0 * R * F2 * D, (R * F2 + R * D) * mx + w1n * 4),
    }
    return out
