/*
 * pmn.h -- C ABI of the block-scaled MoE expert-layer numerics library
 * (GB300, sm_103a).
 *
 * The operations follow the page "Thinking Machines ... Inkling 2 Small ...
 * native 4-bit forward passes" (arex-research.com, 2026-11-14), cited by
 * section:
 *   [Bits]   "fewer bits, faster arithmetic" (更少的比特换更快的算术)
 *   [Layers] "only the expert forward in 4-bit" (只把专家层的前向传播降到 4-bit)
 *   [SR]     "transpose regroups, stochastic rounding keeps the expectation"
 *            (转置打散分组,随机舍入保住期望值)
 *   [NVLink] "NVLink becomes the bottleneck" (计算提速后,NVLink 通信成了新瓶颈)
 *   [Cost]   "the recipe's costs" (配方的代价)
 *
 * Conventions for every call
 *  - All tensor arguments are DEVICE pointers owned by the caller; the library
 *    never synchronises the device inside a call and allocates nothing: where
 *    a kernel needs scratch, the caller passes a workspace whose size a
 *    query returns.  Work is enqueued on `stream` (a cudaStream_t passed as
 *    void*; NULL = legacy default stream) and returns immediately.
 *  - Layouts are row-major and dense unless a leading dimension is given.
 *    NVFP4 tensor [R, C]: codes uint8 [R, C/2] (element 2i in the low nibble,
 *    2i+1 in the high nibble), scales uint8 [R, C/16] (E4M3), outer float32.
 *    MXFP8 tensor [R, C]: values uint8 [R, C] (E4M3), scales uint8 [R, C/32]
 *    (E8M0, value 2^(b-127)).  S2F6 tensor [R, C]: int8 [R, C] (k/64), scales
 *    uint8 [R, C/32] (E8M0).  bf16 tensors are uint16 bit patterns.
 *  - Pointers must be 16-byte aligned; sizes must satisfy the per-call rules
 *    below.  Arguments are checked on the host before anything is enqueued;
 *    a violation returns PMN_ERR_INVALID_ARG and enqueues nothing.
 *  - A failed launch returns PMN_ERR_CUDA.  Kernels never trap: a bounded
 *    device-side wait that runs out latches a bit in a device error word and
 *    the kernel returns; pmn_get_device_error() reads and clears it.
 *  - Every result is bit-reproducible run to run (no atomics in reductions
 *    whose order could change a value).
 */
#ifndef PMN_H
#define PMN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define PMN_API __attribute__((visibility("default")))
#else
#define PMN_API
#endif

typedef int pmn_status;
#define PMN_OK 0
#define PMN_ERR_INVALID_ARG 1
#define PMN_ERR_UNSUPPORTED 2
#define PMN_ERR_CUDA 3
#define PMN_ERR_TIMEOUT 4

/* input modes of pmn_nvfp4_quantize */
#define PMN_IN_BF16 0
#define PMN_IN_BF16_SWIGLU 1
/* outer-scale modes */
#define PMN_OUTER_PER_ROW 0
#define PMN_OUTER_PER_GROUP 1
/* rounding of pmn_requant_transpose_sr_mxfp8 */
#define PMN_ROUND_SR 0
#define PMN_ROUND_RN 1
/* GEMM outputs / epilogues */
#define PMN_OUT_BF16 0
#define PMN_OUT_F32 1
#define PMN_OUT_RHT_S2F6 2
#define PMN_OUT_SWIGLU_BF16 3
/* grouping of pmn_gemm_mxfp8 */
#define PMN_GROUP_M 0
#define PMN_GROUP_K 1

/* device error bits (pmn_get_device_error) */
#define PMN_DEVERR_WAIT_TIMEOUT 1
#define PMN_DEVERR_BAD_OFFSETS 2

/* Library version (major * 10000 + minor * 100 + patch). */
PMN_API int pmn_version(void);

/* Human-readable name of a status code (static string). */
PMN_API const char *pmn_status_string(pmn_status s);

/* Reads and clears the device error word; synchronises `stream` only.
 * *err receives the PMN_DEVERR_* bits latched since the last call. */
PMN_API pmn_status pmn_get_device_error(void *stream, int32_t *err);

/* Wall-time limit, in nanoseconds, of every bounded device wait of the
 * library's kernels (GEMM pipeline barriers, the weight quantiser's wait for
 * a group's amax): a wait that runs out latches PMN_DEVERR_WAIT_TIMEOUT and
 * its kernel winds down and returns.  Default 4 s.  Process-wide, read when
 * a kernel is enqueued; returns the previous limit.  The pages have no
 * counterpart: it exists so that failure handling can be exercised. */
PMN_API uint64_t pmn_set_wait_limit_ns(uint64_t ns);

/* Self-test of the bounded waits: enqueues one CTA whose thread waits on an
 * mbarrier that nothing arrives on, then on a device counter that nothing
 * increments, each for `limit_ns` (<= 2e9, else PMN_ERR_INVALID_ARG), with
 * the wait primitives of the GEMMs and the weight quantiser.  Both waits run
 * out: PMN_DEVERR_WAIT_TIMEOUT is latched and the kernel returns, leaving
 * the context usable.  The pages have no counterpart. */
PMN_API pmn_status pmn_wait_selftest(uint64_t limit_ns, void *stream);

/*
 * NVFP4 quantisation [SR] (16-value blocks, E4M3 block scale set from the
 * block absmax, E2M1 codes by round-to-nearest-even) with a float32 outer
 * scale per row or per group of rows [Cost] and the optional 4/6 choice
 * between two candidate block scales [Cost].
 *
 *  x        bf16 [rows, ldx] (PMN_IN_BF16: the row's first `cols` values are
 *           quantised) or bf16 [rows, ldx] holding gate | up halves of width
 *           `cols` each (PMN_IN_BF16_SWIGLU: h = silu(gate) * up is formed in
 *           float32 -- gate * up / (1 + e^-gate) with the hardware's
 *           approximate exponential and division, within a few dozen float32
 *           ulps -- rounded to bf16, then quantised).
 *  rows, cols  cols % 16 == 0, cols <= 8192 (one row lives in one CTA).
 *  ldx      leading dimension of x in elements (>= cols, or >= 2*cols).
 *  outer_mode  PMN_OUTER_PER_ROW: outer[rows], g = amax(row) / M.
 *           PMN_OUTER_PER_GROUP: outer[rows / rows_per_group], g over each
 *           block of rows_per_group consecutive rows (one expert's weight
 *           matrix, or the whole tensor).  M = 6 * 448, or 4 * 448 with
 *           four_over_six; g = 1 for an all-zero row/group.
 *  rows_per_group  PER_GROUP only: rows % rows_per_group == 0.
 *  four_over_six   0 or 1: keep, per block, the candidate scale amax/6 or
 *           amax/4 with the smaller squared dequantisation error (ties: 6).
 *  codes    out uint8 [rows, cols/2];  scales  out uint8 [rows, cols/16];
 *  outer    out float32 (see outer_mode).
 *  h_out    optional out bf16 [rows, cols]: the SwiGLU value that was
 *           quantised (PMN_IN_BF16_SWIGLU only; NULL to skip).
 *  workspace, workspace_bytes  PER_GROUP only (ignored for PER_ROW): caller-
 *           owned device scratch, 16-byte aligned, at least
 *           pmn_nvfp4_quantize_workspace_bytes(...) bytes (else
 *           PMN_ERR_INVALID_ARG); its contents on entry do not matter (the
 *           call clears it on `stream`).  Calls that share one workspace must
 *           not overlap on the GPU (calls on one stream are ordered).
 * PER_GROUP runs one persistent kernel that reads each group for its amax and
 * codes it while it is still in L2; the workspace holds its ticket counter,
 * per-group counts and amax.  A group whose amax pass never completes
 * (bounded wait, pmn_set_wait_limit_ns) latches PMN_DEVERR_WAIT_TIMEOUT.
 */
PMN_API pmn_status pmn_nvfp4_quantize(const void *x, int64_t rows, int64_t cols, int64_t ldx, int in_mode,
                              int outer_mode, int64_t rows_per_group, int four_over_six,
                              uint8_t *codes, uint8_t *scales, float *outer, void *h_out,
                              void *workspace, int64_t workspace_bytes, void *stream);

/* Workspace bytes pmn_nvfp4_quantize needs: (64 + 2 * groups) * 4 for
 * PMN_OUTER_PER_GROUP (groups = rows / rows_per_group), 0 for
 * PMN_OUTER_PER_ROW, -1 for invalid arguments.  Host only; no CUDA call. */
PMN_API int64_t pmn_nvfp4_quantize_workspace_bytes(int outer_mode, int64_t rows, int64_t rows_per_group);

/*
 * pmn_nvfp4_quantize with PMN_OUTER_PER_GROUP (ldx = cols), computing the
 * same bytes, but with its scratch in a fixed device array of the library
 * (a file-scope __device__ array of (64 + 2 * 1024) 32-bit words, which every
 * GPU that loads the library holds until the process exits) instead of a
 * workspace: the caller neither allocates nor passes scratch.  The pages
 * have no counterpart to this entry point.  It is for callers that cannot
 * call cudaMalloc or any allocator while they run: a serving loop whose
 * device memory is all reserved at start-up, or a host framework that owns
 * every device allocation and hands this library only its input and output
 * buffers.
 *  rows / rows_per_group <= 1024 groups, else PMN_ERR_INVALID_ARG.
 *  Other arguments and rules as pmn_nvfp4_quantize.
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, once per device, with that device current).  The
 * array is shared by every call on a device and keeps the last call's
 * contents; each call clears it on `stream` before its kernel runs.  Calls
 * that overlap on the GPU (on different streams) race on it; calls on one
 * stream are ordered.
 */
PMN_API pmn_status pmn_nvfp4_quantize_per_group_noalloc(const void *x, int64_t rows, int64_t cols,
                                                        int64_t rows_per_group, int four_over_six,
                                                        uint8_t *codes, uint8_t *scales, float *outer,
                                                        void *stream);

/*
 * Dequantise -> transpose -> requantise to MXFP8 [SR]: the saved NVFP4 tensor
 * is dequantised in float32, d = (code * scale) * g, transposed, and rounded
 * to E4M3 with one E8M0 scale per 32 values along the ORIGINAL rows.  The
 * scale exponent is the smallest e with amax <= 448 * 2^e (never clips), so
 * stochastic rounding keeps E[result] = d ([SR]: E[w_q] = E[(w_q^T)^T]).
 *
 *  codes, scales  NVFP4 [batch, rows, cols] (batch = experts for weights, 1
 *           for activations).
 *  outer    float32: PMN_OUTER_PER_ROW -> [batch * rows] (tokens);
 *           PMN_OUTER_PER_GROUP -> [batch] (one per expert).
 *  rows     multiple of 32 (expert segments of activations must be padded
 *           with zero rows to multiples of 32 so blocks never straddle).
 *  cols     multiple of 64.
 *  seed, tag  stochastic rounding bits: element i of the output (row-major
 *           index over [batch, cols, rows]) takes 16 bits of one word of
 *           Philox4x32-10 (Salmon et al., SC'11) with key (seed lo, seed hi)
 *           and counter (j lo, j hi, tag, 0), j = i / 16: word (i / 4) % 4;
 *           elements 4w and 4w+1 use its low 16 bits (4w+1 in reversed bit
 *           order), 4w+2 and 4w+3 its high 16 bits (4w+3 reversed).  The
 *           bits are added to the leading 16 bits of the discarded fraction;
 *           a carry rounds away from zero (the hardware's SR conversion).
 *  rounding PMN_ROUND_SR or PMN_ROUND_RN (nearest even; bits unused).
 *  out      uint8 [batch, cols, rows] (E4M3); out_scales uint8 [batch, cols,
 *           rows/32] (E8M0).
 */
PMN_API pmn_status pmn_requant_transpose_sr_mxfp8(const uint8_t *codes, const uint8_t *scales,
                                          const float *outer, int outer_mode, int64_t batch,
                                          int64_t rows, int64_t cols, uint64_t seed, uint32_t tag,
                                          int rounding, uint8_t *out, uint8_t *out_scales,
                                          void *stream);

/*
 * Dequantise -> transpose -> requantise to NVFP4 with stochastic rounding:
 * the FP4 backward that the pages name as future work, the [SR] steps with
 * the forward's NVFP4 format.  d = (code * S) * g in float32 as above;
 * entry b of the output gets one float32 outer scale
 *   g'_b = (max over the entry's input blocks of dec(S) * g) / 448
 * (1 if every scale is zero; zero padding blocks do not count), so every
 * value fits; per 16 values along the ORIGINAL rows the E4M3 scale is the
 * smallest E4M3 value >= amax / (6 g') (saturating at 448: no value clips,
 * which keeps stochastic rounding unbiased); y = d * (1 / (dec(S') g'))
 * (float32), and the E2M1 code is y rounded stochastically with 16 random
 * bits per element (the rule, counters and bit layout of
 * pmn_requant_transpose_sr_mxfp8) or to nearest even (PMN_ROUND_RN).
 *  codes, scales, outer, outer_mode, batch, rows, cols, seed, tag, rounding
 *           as pmn_requant_transpose_sr_mxfp8 (rows % 32 == 0, cols % 64 == 0).
 *  out      uint8 [batch, cols, rows/2] (element 2i in the low nibble);
 *  out_scales uint8 [batch, cols, rows/16] (E4M3);
 *  out_outer float32 [batch] (4-byte aligned); used as scratch during the call.
 * Launches a scale reduction, the requantisation and a finalisation (three
 * kernels and one memset on `stream`).
 */
PMN_API pmn_status pmn_requant_transpose_sr_nvfp4(const uint8_t *codes, const uint8_t *scales,
                                          const float *outer, int outer_mode, int64_t batch,
                                          int64_t rows, int64_t cols, uint64_t seed, uint32_t tag,
                                          int rounding, uint8_t *out, uint8_t *out_scales,
                                          float *out_outer, void *stream);

/*
 * bf16 -> MXFP8 with round-to-nearest-even (the gradient dY; the pages ask
 * for SR on the saved forward tensors only).  Same scale rule as above.
 *  transpose 0: out [rows, cols], out_scales [rows, cols/32] (cols % 32 == 0)
 *  transpose 1: out [cols, rows], out_scales [cols, rows/32] (rows % 32 == 0,
 *               rows <= 65535 * 128, else PMN_ERR_UNSUPPORTED)
 * x and out 16-byte aligned.  One kernel on `stream`.
 */
PMN_API pmn_status pmn_mxfp8_quantize(const void *x, int64_t rows, int64_t cols, int transpose,
                              uint8_t *out, uint8_t *out_scales, void *stream);

/*
 * Both orientations of pmn_mxfp8_quantize in one pass over x [SR]: the
 * gradient's rowwise copy feeds dX / dH, its transposed copy the weight
 * gradients of the MXFP8 backward.  x is read once; the bytes equal those of
 * the two separate calls.
 *  x      bf16 [rows, cols], row-major, 16-byte aligned.
 *  rows % 32 == 0 and cols % 32 == 0 (else PMN_ERR_INVALID_ARG);
 *  rows <= 65535 * 128 (else PMN_ERR_UNSUPPORTED).
 *  out_rows [rows, cols] (16-byte aligned), out_rows_scales [rows, cols/32];
 *  out_cols [cols, rows] (16-byte aligned), out_cols_scales [cols, rows/32].
 * All buffers are the caller's device memory.  One kernel on `stream`.
 */
PMN_API pmn_status pmn_mxfp8_quantize_both(const void *x, int64_t rows, int64_t cols, uint8_t *out_rows,
                                          uint8_t *out_rows_scales, uint8_t *out_cols, uint8_t *out_cols_scales,
                                          void *stream);

/*
 * SwiGLU followed by MXFP8 quantisation (round to nearest even, E8M0 per 32
 * along the row) of h, for the forward of the last 16.6 % of layers, which
 * the pages keep in MXFP8 instead of NVFP4 [Cost]:
 *   h = bf16(silu(gate) * up), formed in float32 as in PMN_IN_BF16_SWIGLU;
 *   out = MXFP8(h) as pmn_mxfp8_quantize (transpose 0).
 *  y        bf16 [rows, 2 f]: gate = columns [0, f), up = columns [f, 2 f).
 *  f        multiple of 32;  rows * f / 32 < 2^32.
 *  out      uint8 [rows, f] (E4M3);  out_scales uint8 [rows, f / 32].
 *  h_out    optional bf16 [rows, f]: the h that was quantised (NULL to skip).
 */
PMN_API pmn_status pmn_mxfp8_quantize_swiglu(const void *y, int64_t rows, int64_t f, uint8_t *out,
                                     uint8_t *out_scales, void *h_out, void *stream);

/*
 * Grouped NVFP4 expert GEMM for the forward pass [Layers], [Cost]:
 *   Z[m, n] = (sum_k A[m, k] * B_e[n, k]) * a_outer[m] * b_outer[e]
 * for the rows m of expert e, offsets[e] <= m < offsets[e+1].  A and B are
 * NVFP4 with the contraction along their rows (K-major); the products are
 * accumulated in float32 on the tensor cores (block-scaled MMA).
 *
 *  a_codes/a_scales  NVFP4 [total_rows, k]; a_outer float32 [total_rows].
 *  b_codes/b_scales  NVFP4 [num_experts, n, k]; b_outer float32 [num_experts].
 *  offsets  DEVICE int32 [num_experts + 1], non-decreasing, 0 <= offsets[e]
 *           <= total_rows (any row counts, empty experts allowed).  They are
 *           read and checked on the device: invalid offsets run nothing and
 *           latch PMN_DEVERR_BAD_OFFSETS.  num_experts <= 1024.
 *  n        multiple of 128;  k multiple of 256.
 *  out_kind PMN_OUT_BF16 (bf16 [total_rows, n]) or PMN_OUT_F32, or
 *           PMN_OUT_SWIGLU_BF16 (n % 256 == 0): bf16 h [total_rows, n/2] with
 *           h[m, j] = silu(y[m, j]) * y[m, n/2 + j], y = Z rounded to bf16 as
 *           PMN_OUT_BF16 writes it (gate = the first n/2 rows of each B_e, up =
 *           the last n/2), formed in float32 and rounded to bf16 (nearest
 *           even): the arithmetic of pmn_nvfp4_quantize's PMN_IN_BF16_SWIGLU
 *           on the bf16 output, so h equals that unfused path's bit for bit.
 *           SwiGLU between w1 and w2 is not on the pages; the w1 shape
 *           [2F, d_model] makes the layer gated.
 * Rows outside every expert segment are not written.
 */
PMN_API pmn_status pmn_grouped_gemm_nvfp4(const uint8_t *a_codes, const uint8_t *a_scales,
                                  const float *a_outer, const uint8_t *b_codes,
                                  const uint8_t *b_scales, const float *b_outer,
                                  const int32_t *offsets, int num_experts, int64_t total_rows,
                                  int64_t n, int64_t k, int out_kind, void *out, void *stream);

/*
 * w1 GEMM with SwiGLU fused into its epilogue, then the NVFP4 quantisation
 * of h with a per-token outer scale and the optional 4/6 choice [Cost]: the
 * pages fuse quantisation into the GEMM epilogues [NVLink] and keep the
 * expert forward in NVFP4 [Layers].  Two kernels on `stream`:
 *   1. the grouped NVFP4 GEMM of pmn_grouped_gemm_nvfp4 with out_kind
 *      PMN_OUT_SWIGLU_BF16 (n = 2 f) writes bf16 h [total_rows, f];
 *   2. pmn_nvfp4_quantize(h, PER_ROW, four_over_six) of those rows; rows at
 *      or past offsets[num_experts] (outside every expert segment) are
 *      written as the quantisation of a zero row (codes 0, scales 0, outer 1).
 * The per-token outer scale needs the amax of the whole row of h, which
 * spans f / 128 tiles of the GEMM, so the codes are formed by the second
 * kernel from h instead of in the GEMM's epilogue.
 *  b_codes/b_scales/b_outer  NVFP4 W1 [num_experts, 2 f, k]: rows [0, f)
 *           gate, [f, 2 f) up.
 *  f        multiple of 128, <= 8192;  k multiple of 256.
 *  h        caller-owned bf16 [total_rows, f]: receives h (the kernels'
 *           scratch between the two steps; also a result).
 *  codes    uint8 [total_rows, f/2]; scales uint8 [total_rows, f/16];
 *  outer    float32 [total_rows].
 * Other arguments as pmn_grouped_gemm_nvfp4.
 */
PMN_API pmn_status pmn_w1_gemm_swiglu_nvfp4(const uint8_t *a_codes, const uint8_t *a_scales,
                                    const float *a_outer, const uint8_t *b_codes,
                                    const uint8_t *b_scales, const float *b_outer,
                                    const int32_t *offsets, int num_experts, int64_t total_rows,
                                    int64_t f, int64_t k, int four_over_six, void *h,
                                    uint8_t *codes, uint8_t *scales, float *outer, void *stream);

/*
 * w2 GEMM with the combine quantisation fused into its epilogue [NVLink]:
 * the grouped NVFP4 GEMM above, then for every 32 contiguous outputs of a row
 *   z = RN(1/sqrt(32)) * FWHT32(sigma . x)   (float32 butterflies h=1..16)
 *   e = smallest integer with amax(|z|) <= (127/64) * 2^e   (E8M0 byte e+127)
 *   k = round-to-nearest-even(z * 2^(6-e))                   (S2F6 int8)
 * sigma in {+-1}^32 is bit j of Philox4x32-10 word 0 at counter (0, 0, 5, 0)
 * with key (seed lo, seed hi), bit set -> -1, the same for every block.
 *  out      int8 [total_rows, n];  out_scales uint8 [total_rows, n/32].
 *  debug_acc  NULL, or float32 [total_rows, n], 16-byte aligned: receives
 *           the epilogue's input x (the accumulator times both outer
 *           scales) for the rows of the expert segments, so that the
 *           fused epilogue can be checked byte for byte against
 *           pmn_rht_s2f6_quantize or a reference of it.  The pages have no
 *           counterpart; it costs one fp32 write of the output when set.
 * Other arguments as pmn_grouped_gemm_nvfp4.
 */
PMN_API pmn_status pmn_w2_gemm_rht_s2f6(const uint8_t *a_codes, const uint8_t *a_scales,
                                const float *a_outer, const uint8_t *b_codes,
                                const uint8_t *b_scales, const float *b_outer,
                                const int32_t *offsets, int num_experts, int64_t total_rows,
                                int64_t n, int64_t k, uint64_t seed, int8_t *out,
                                uint8_t *out_scales, float *debug_acc, void *stream);

/*
 * The combine quantisation alone on a float32 tensor [NVLink] (the same
 * epilogue arithmetic as pmn_w2_gemm_rht_s2f6, for unfused use):
 *  x float32 [rows, cols], cols % 32 == 0 -> out int8 [rows, cols],
 *  out_scales uint8 [rows, cols/32].
 */
PMN_API pmn_status pmn_rht_s2f6_quantize(const float *x, int64_t rows, int64_t cols, uint64_t seed,
                                 int8_t *out, uint8_t *out_scales, void *stream);

/*
 * Receive side of the combine, back in token order [NVLink]: the pages call
 * the combine transform orthogonal and exactly invertible; each token sums
 * its k expert results, weighted by the router's gates:
 *   out[t, :] = sum_i gates[t, i] * R(row_index[t, i])
 *   R(r), per 32-block: sigma . H (k / 64 * 2^(b - 127)) / sqrt(32)
 * with (k, b) the S2F6 bytes and E8M0 scale of routed row r, H the 32-point
 * Sylvester Hadamard matrix and sigma the sign word of pmn_w2_gemm_rht_s2f6
 * for the same seed.  Computed in float32: the choices are summed before
 * the transform (u = sum_i (gate_i 2^(e_i - 6)) k_i by fma, in order i = 0 ..
 * k-1), then one FWHT32, RN(1/sqrt(32)), the signs.  How the k results are
 * merged is not on the pages; the weighted sum of an MoE combine is taken.
 *  q        int8 [rows, cols], scales uint8 [rows, cols/32]: the combine
 *           payload (rows in the routed, expert-sorted order), cols % 32 == 0.
 *  row_index  DEVICE int32 [tokens, k] (4-byte aligned): the routed row of
 *           token t's i-th choice; negative = a dropped choice (adds
 *           nothing); an index >= rows adds nothing and latches
 *           PMN_DEVERR_BAD_OFFSETS.
 *  gates    DEVICE float32 [tokens, k] (4-byte aligned).
 *  k        1 .. 64.
 *  out_kind PMN_OUT_BF16 (round to nearest even from float32) or
 *           PMN_OUT_F32;  out [tokens, cols].
 * tokens == 0 or cols == 0 returns PMN_OK before the pointers are checked.
 */
PMN_API pmn_status pmn_combine_receive_s2f6(const int8_t *q, const uint8_t *scales, int64_t rows,
                                    int64_t cols, uint64_t seed, const int32_t *row_index,
                                    const float *gates, int64_t tokens, int k, int out_kind,
                                    void *out, void *stream);

/*
 * Grouped MXFP8 GEMM for the backward pass [SR] (E4M3 operands with E8M0
 * scales per 32 along the contraction, float32 accumulation):
 *   C[m, n] = sum_k A[m, k] * B[n, k]
 * group_mode PMN_GROUP_M (dX = dY . W): A [m, k], B [num_groups, n, k];
 *           rows of group g are offsets[g] <= row < offsets[g+1]; out [m, n].
 * group_mode PMN_GROUP_K (dW = dY^T . X per expert): A [m, k], B [n, k] with k
 *           the routed-row axis; group g contracts offsets[g] <= k <
 *           offsets[g+1] (multiples of 128); out [num_groups, m, n].
 *  offsets  DEVICE int32 [num_groups + 1], non-decreasing, within [0, m]
 *           (GROUP_M) or [0, k] and multiples of 128 (GROUP_K: expert
 *           segments of the routed rows padded with zero rows to multiples of
 *           128, so every 128-deep K stage starts on a 4-scale boundary);
 *           checked on the device (invalid: nothing runs,
 *           PMN_DEVERR_BAD_OFFSETS latched).
 *  scale tensors need a row pitch that is a multiple of 16 bytes: k % 512 == 0.
 *  m        multiple of 128 for PMN_GROUP_K;  n multiple of 128;  k multiple
 *           of 512.  num_groups <= 1024.
 *  out_kind PMN_OUT_BF16 or PMN_OUT_F32.
 */
PMN_API pmn_status pmn_gemm_mxfp8(const uint8_t *a, const uint8_t *a_scales, const uint8_t *b,
                          const uint8_t *b_scales, const int32_t *offsets, int num_groups,
                          int group_mode, int64_t m, int64_t n, int64_t k, int out_kind, void *out,
                          void *stream);

#ifdef __cplusplus
}
#endif

#endif /* PMN_H */
