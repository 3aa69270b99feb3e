/*
 * nvfp4.h: C ABI of libnvfp4, the NVFP4 inference-GEMM hot path for
 * B300 (sm_103a).
 *
 * The operations follow these pages (cited by title and section):
 *  [TRT] "NVIDIA Ships TensorRT-LLM 0.16: Native FP4 Quantization for
 *        Blackwell B200", section "The Mathematical Breakthrough of
 *        Microscopic FP4 Scaling": E2M1 elements (1 sign, 2 exponent,
 *        1 mantissa bit); item 2 "Two-Level Block Scaling" (one FP8 scale per
 *        16 consecutive elements; an FP16 macro-scale per 16 micro-vectors);
 *        item 3 "Hardware-Fused Dequantization" (tensor cores apply the
 *        scales before the dot products).
 *  [LCP] "llama.cpp Put Precision Policy Inside the Model. That Matters More
 *        Than W4A4": section "One model can need more than one precision"
 *        (native W4A4 path; W4A8 for marked tensors; dense and MoE) and
 *        section "Local inference is becoming a policy engine" (q4 forces
 *        W4A4, q8 forces W4A8, auto follows per-tensor metadata).
 *  [ADA] "AdaLLM Breakthrough: First NVFP4-Only Inference Engine for RTX 4090
 *        Unveiled": fail fast, no silent fallback to a slower precision.
 *
 * Conventions shared by every entry point:
 *  - All data pointers are DEVICE pointers owned by the caller.  The library
 *    allocates no memory on these paths; scratch lives in a caller-provided
 *    workspace (see nvfp4_workspace_size / nvfp4_workspace_init).
 *  - Every call is asynchronous and stream-ordered on `stream` (a
 *    cudaStream_t; NULL is the legacy default stream).
 *  - Argument checks run on the host before anything is enqueued; a call
 *    that returns an error has enqueued no work ("fail fast", [ADA]).
 *  - Errors found on the device (non-finite input, a bounded wait that gave
 *    up) are OR-ed into a sticky status word in the workspace; read it with
 *    nvfp4_device_status.  There is no CPU or lower-precision fallback.
 *  - The entry points are not re-entrant on one workspace: two calls that
 *    overlap on the GPU must use different workspaces.
 */
#ifndef NVFP4_H
#define NVFP4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *nvfp4_stream_t; /* same type as cudaStream_t */

typedef enum nvfp4_status {
    NVFP4_OK = 0,
    NVFP4_ERR_INVALID_ARG = 1,       /* null pointer, bad enum, bad stride or alignment */
    NVFP4_ERR_UNSUPPORTED_SHAPE = 2, /* K, N or M outside what the kernels take */
    NVFP4_ERR_NONFINITE_INPUT = 3,   /* device: an input element was Inf or NaN */
    NVFP4_ERR_TIMEOUT = 4,           /* device: a bounded wait inside a kernel gave up */
    NVFP4_ERR_CUDA = 5,              /* a CUDA runtime or driver call failed */
    NVFP4_ERR_WORKSPACE = 6,         /* workspace missing, misaligned or too small */
    NVFP4_ERR_UNSUPPORTED = 7        /* valid request the library does not implement */
} nvfp4_status;

/* Per-call precision policy, [LCP] "Local inference is becoming a policy
 * engine": Q4 forces W4A4, Q8 forces W4A8, AUTO follows the layer's
 * `sensitive` flag (W4A8 when set, W4A4 otherwise). */
typedef enum nvfp4_policy {
    NVFP4_POLICY_AUTO = 0,
    NVFP4_POLICY_Q4 = 1,
    NVFP4_POLICY_Q8 = 2
} nvfp4_policy;

/* Second-level scale, [TRT] item 2.  TENSOR_FP32: one float per tensor,
 * amax / (6 * 448).  MACRO_FP16: one binary16 per 256 consecutive elements of
 * a row (16 micro-blocks), FP16(amax_256 / 2688), saturating at 65504. */
typedef enum nvfp4_scale_mode {
    NVFP4_SCALE_TENSOR_FP32 = 0,
    NVFP4_SCALE_MACRO_FP16 = 1
} nvfp4_scale_mode;

/* Layout of the E4M3 micro-scale bytes.
 *  ROW_MAJOR: byte [r][b] at r * (K/16) + b.
 *  MMA_TILED: the layout the tensor cores read.  Rows are padded to a
 *    multiple of 128 (padding bytes are written as 0) and K to a multiple
 *    of 64.  Scale b of row r lives in the 512-byte atom
 *    (r / 128) * (K/64) + (b / 4), at byte (r % 32) * 16 + ((r % 128) / 32) * 4
 *    + (b % 4) of that atom. */
typedef enum nvfp4_scale_layout {
    NVFP4_LAYOUT_ROW_MAJOR = 0,
    NVFP4_LAYOUT_MMA_TILED = 1
} nvfp4_scale_layout;

typedef enum nvfp4_out_dtype {
    NVFP4_OUT_BF16 = 0, /* round to nearest even */
    NVFP4_OUT_FP32 = 1
} nvfp4_out_dtype;

/* An NVFP4 tensor [rows, K] (activations [M, K] or weights [N, K]).
 *  codes : uint8 [rows][K/2]; element 2j in the low nibble of byte j, 2j+1
 *          in the high nibble; each nibble is an E2M1 code (bit 3 = sign).
 *          16-byte aligned.
 *  scales: E4M3 bytes, `layout` as above, 16-byte aligned.
 *  second: TENSOR_FP32 -> float[1] (for the stacked expert weights of
 *          nvfp4_grouped_gemm, float[E]); MACRO_FP16 -> binary16 [rows][K/256].
 *  Dequantised value: E2M1(code) * E4M3(scale) * second. */
typedef struct nvfp4_tensor {
    void *codes;
    void *scales;
    void *second;
    int64_t rows;
    int64_t K;
    int32_t mode;   /* nvfp4_scale_mode */
    int32_t layout; /* nvfp4_scale_layout */
} nvfp4_tensor;

/* Operation ids for nvfp4_workspace_size. */
typedef enum nvfp4_op {
    NVFP4_OP_QUANTIZE = 0,     /* M = rows, K */
    NVFP4_OP_QUANTIZE_FP8 = 1, /* M = rows, K */
    NVFP4_OP_GEMM = 2,         /* M, N, K; covers both routes and on-the-fly quantisation */
    NVFP4_OP_W4A8_GEMM = 3,    /* M, N, K */
    NVFP4_OP_GROUPED_GEMM = 4, /* M = total routed rows, N, K, E experts */
    NVFP4_OP_GROUPED_GEMM_X = 5, /* M = T activation rows (tokens), N, K, E; both routes */
    NVFP4_OP_KV_DECODE = 6       /* M = sequences, N = query heads, K = max context, E = KV heads */
} nvfp4_op;

/* ---- sizing and workspace ------------------------------------------------ */

/* Bytes of the E4M3 scale buffer of a [rows, K] tensor in `layout`.
 * Errors: INVALID_ARG for a null `bytes`, negative sizes or a bad layout;
 * UNSUPPORTED_SHAPE when K % 16 != 0 (row-major) or K % 64 != 0 (tiled). */
nvfp4_status nvfp4_scale_bytes(int64_t rows, int64_t K, int32_t layout, size_t *bytes);

/* Workspace bytes an operation needs.  Unused sizes may be 0.  The result
 * includes a 256-byte header that holds the sticky device status word. */
nvfp4_status nvfp4_workspace_size(int32_t op, int64_t M, int64_t N, int64_t K, int32_t E,
                                  size_t *bytes);

/* Zeroes a workspace (status word and the stream-K ready flags, which the
 * GEMM kernels leave zeroed after every call) on `stream`.  Call once after
 * allocating it, and again after a TIMEOUT status (an aborted kernel may leave
 * flags raised).  The status word stays sticky between calls.
 * `ws` must be 256-byte aligned. */
nvfp4_status nvfp4_workspace_init(void *ws, size_t ws_bytes, nvfp4_stream_t stream);

/* Waits for `stream`, then reads and clears the workspace's device status
 * word into *device_status (a nvfp4_status: OK, NONFINITE_INPUT or TIMEOUT;
 * NONFINITE wins when both bits are set).  The only synchronising call. */
nvfp4_status nvfp4_device_status(void *ws, nvfp4_stream_t stream, int32_t *device_status);

/* Route the policy selects for one layer: returns 4 (W4A4), 8 (W4A8) or -1
 * for an unknown policy.  Host only; nvfp4_gemm uses exactly this rule.
 * [LCP] "Local inference is becoming a policy engine". */
int32_t nvfp4_policy_route(int32_t policy, int32_t sensitive);

/* ---- the hot path ---------------------------------------------------------- */

/* NVFP4 quantisation of BF16 x [rows, K] (row stride ldx elements) into
 * `out` (caller sets out->mode and out->layout and provides the buffers;
 * out->rows and out->K must equal rows and K).  [TRT] item 2; encode order,
 * in IEEE binary32:
 *   s = amax(tensor) / 2688  (or per 256-group FP16 macro-scale)
 *   per 16-block: e = E4M3_rne_sat((amax_b / 6) / s), d = e * s,
 *   r = 1 / d (0 when d == 0, at most FLT_MAX), code = E2M1_rne_sat(x * r).
 * K % 16 == 0 (row-major scales), % 64 (tiled), % 256 (macro).  x must be
 * 16-byte aligned, ldx % 8 == 0.  Non-finite input sets NONFINITE_INPUT in
 * the device status; its outputs are then unspecified. */
nvfp4_status nvfp4_quantize(const void *x_bf16, int64_t rows, int64_t K, int64_t ldx,
                            nvfp4_tensor *out, void *ws, size_t ws_bytes, nvfp4_stream_t stream);

/* Per-token FP8 quantisation for the W4A8 route ([LCP] "One model can need
 * more than one precision"): per row, s_t = amax_row / 448 and
 * a = E4M3_rne_sat(x * (1 / s_t)).  a_fp8 is uint8 [rows][K] (dense),
 * s_t float[rows].  K % 16 == 0, x 16-byte aligned, ldx % 8 == 0. */
nvfp4_status nvfp4_quantize_fp8(const void *x_bf16, int64_t rows, int64_t K, int64_t ldx,
                                void *a_fp8, float *s_t, void *ws, size_t ws_bytes,
                                nvfp4_stream_t stream);

/* One layer Y[M, N] = X[M, K] * W[N, K]^T under the precision policy.
 *  Give exactly one of x_bf16 (BF16 [M, K], row stride ldx; quantised on the
 *  fly into the workspace by the route's quantiser) or a_q (pre-quantised
 *  NVFP4 activations, tiled scales; W4A4 route only).
 *  w: NVFP4 weights [N, K], MMA_TILED scales, TENSOR_FP32 or MACRO_FP16.
 *  Route = nvfp4_policy_route(policy, sensitive):
 *    W4A4: Y = s_a * s_w * sum_k E2M1(a)E4M3(ea) * E2M1(w)E4M3(ew)  ([TRT] item 3,
 *          [LCP] native W4A4), or per-256-group macro-scales in MACRO mode;
 *    W4A8: Y = s_t[m] * s_w * sum_k E4M3(a) * E2M1(w)E4M3(ew)   ([LCP]).
 *  y: [M, N] with row stride ldy elements, y_dtype BF16 or FP32, 16-byte
 *  aligned.  K % 64 == 0 (% 256 in macro mode).  W4A8 needs x_bf16 and
 *  TENSOR_FP32 weights.  Returns UNSUPPORTED_SHAPE for shapes the kernels do
 *  not take, UNSUPPORTED for W4A8 with pre-quantised activations. */
nvfp4_status nvfp4_gemm(const void *x_bf16, int64_t ldx, const nvfp4_tensor *a_q,
                        const nvfp4_tensor *w, void *y, int64_t ldy, int32_t y_dtype, int64_t M,
                        int32_t policy, int32_t sensitive, void *ws, size_t ws_bytes,
                        nvfp4_stream_t stream);

/* One W4A4 layer whose output is the next layer's NVFP4 activations: the
 * next layer's quantiser fused into this GEMM's epilogue, so Y never reaches
 * HBM in BF16 or FP32.  [TRT] item 2 defines the encode; the tensor scale
 * cannot be amax(Y)/2688 of this very output (Y is not complete while it is
 * being encoded), so it is a static one fixed beforehand by calibration, or
 * the previous step's, in the spirit of the calibration step [TRT]
 * describes.
 *  x_bf16/ldx or a_q: the activations, exactly as for nvfp4_gemm (W4A4 route,
 *  TENSOR_FP32 only).  w: TENSOR_FP32 weights [N, K], MMA_TILED.
 *  y_q: caller-owned output tensor: rows == M, K == N (so N % 64 == 0),
 *  mode TENSOR_FP32, layout MMA_TILED; y_q->second is a device float[1]
 *  holding the tensor scale s_y (read, not written).
 *  Each 16-element block of y = fl32(s_a * s_w) * acc (the FP32 output of
 *  nvfp4_gemm) is encoded with the nvfp4_quantize rule under s_y; blocks
 *  whose magnitude exceeds 6 * 448 * s_y saturate.  Scales of the padding
 *  rows of the last 128-row tile are written as 0.
 *  y_amax: NULL, or a device float updated to max(*y_amax, max|y|) (the
 *  amax from which a later call's s_y = amax / 2688 can be taken);
 *  initialise it to 0.  Must not alias y_q.
 *  Workspace: nvfp4_workspace_size(NVFP4_OP_GEMM, M, N, K).
 *  Errors: as nvfp4_gemm; UNSUPPORTED for MACRO_FP16 weights. */
nvfp4_status nvfp4_gemm_nvfp4_out(const void *x_bf16, int64_t ldx, const nvfp4_tensor *a_q,
                                  const nvfp4_tensor *w, nvfp4_tensor *y_q, float *y_amax, int64_t M,
                                  void *ws, size_t ws_bytes, nvfp4_stream_t stream);

/* W4A8 contraction from pre-quantised FP8 activations, the route [LCP]
 * ("One model can need more than one precision") gives tensors marked as
 * sensitive, and the FP8 activations [TRT] ("Deployment Guidelines and
 * Production Safeguards", item 2) keeps for sensitive layers:
 * Y[m, n] = s_t[m] * s_w * sum_k E4M3(a[m, k]) * E2M1(w[n, k]) * E4M3(ew[n, k/16]).
 * a_fp8 uint8 [M][K] dense, s_t float[M]; w TENSOR_FP32, MMA_TILED. */
nvfp4_status nvfp4_w4a8_gemm(const void *a_fp8, const float *s_t, const nvfp4_tensor *w,
                             void *y, int64_t ldy, int32_t y_dtype, int64_t M, void *ws,
                             size_t ws_bytes, nvfp4_stream_t stream);

/* Grouped (mixture-of-experts) W4A4, [LCP] (MoE operations):
 *  a: NVFP4 activations [T_a, K], TENSOR_FP32, MMA_TILED, quantised once.
 *  expert_offsets: device int64[E+1], non-decreasing, offsets[0] == 0,
 *    offsets[E] <= total_rows; expert e owns output rows
 *    offsets[e] .. offsets[e+1]-1.
 *  row_idx: device int32[total_rows] giving the activation row of each
 *    output row (values in [0, T_a)), or NULL for row j reading row j.
 *  w: the E experts' weights stacked as one NVFP4 tensor [E*N, K]
 *    (rows e*N .. e*N+N-1 belong to expert e), TENSOR_FP32 with
 *    second = float[E] (one tensor scale per expert), MMA_TILED, N % 128 == 0.
 *  y: [total_rows, N] with row stride ldy; rows past offsets[E] untouched.
 *  Y[j, n] = s_a * s_w[e] * sum_k a[row(j), k] * w[e*N + n, k].
 *  policy/sensitive: the layer's policy and sensitive flag as for nvfp4_gemm;
 *  `a` is NVFP4, so a request that resolves to W4A8 returns UNSUPPORTED
 *  (nvfp4_grouped_gemm_x and nvfp4_grouped_w4a8_gemm take that route).  Offsets are read on the device (no
 *  host synchronisation); invalid offsets give unspecified rows. */
nvfp4_status nvfp4_grouped_gemm(const nvfp4_tensor *a, const int32_t *row_idx,
                                const int64_t *expert_offsets, int32_t E, const nvfp4_tensor *w,
                                int64_t N, void *y, int64_t ldy, int32_t y_dtype,
                                int64_t total_rows, int32_t policy, int32_t sensitive,
                                void *ws, size_t ws_bytes, nvfp4_stream_t stream);

/* Grouped W4A8 from pre-quantised FP8 activations (the W4A8 route of [LCP]
 * covers MoE operations as well as dense ones):
 *   Y[j, n] = s_t[row(j)] * s_w[e] * sum_k E4M3(a[row(j), k]) * w[e*N + n, k]
 * with the row / offsets / expert conventions of nvfp4_grouped_gemm.
 *  a_fp8: uint8 [T, K] E4M3 (16-byte aligned), s_t: float[T] per-token
 *  scales (as nvfp4_quantize_fp8 writes them).  w: [E*N, K] TENSOR_FP32,
 *  MMA_TILED, second = float[E]; N % 128 == 0, K % 64 == 0.
 *  Routed rows whose activation index is out of range give zero rows.
 *  Workspace: nvfp4_workspace_size(NVFP4_OP_GROUPED_GEMM, total_rows, N, K, E). */
nvfp4_status nvfp4_grouped_w4a8_gemm(const void *a_fp8, const float *s_t, int64_t T,
                                     const int32_t *row_idx, const int64_t *expert_offsets,
                                     int32_t E, const nvfp4_tensor *w, int64_t N, void *y,
                                     int64_t ldy, int32_t y_dtype, int64_t total_rows, void *ws,
                                     size_t ws_bytes, nvfp4_stream_t stream);

/* Grouped GEMM of BF16 activations x [T, K] (row stride ldx) under the
 * precision policy ([LCP]: MoE operations on both routes; q4 / q8 / auto in
 * "Local inference is becoming a policy engine"): the route
 * (nvfp4_policy_route(policy, sensitive))
 * quantises x once into the workspace (NVFP4 per-tensor for W4A4, FP8
 * per-token for W4A8) and runs nvfp4_grouped_gemm's or
 * nvfp4_grouped_w4a8_gemm's contraction with the same conventions.
 * Workspace: nvfp4_workspace_size(NVFP4_OP_GROUPED_GEMM_X, T, N, K, E). */
nvfp4_status nvfp4_grouped_gemm_x(const void *x_bf16, int64_t ldx, int64_t T, const int32_t *row_idx,
                                  const int64_t *expert_offsets, int32_t E, const nvfp4_tensor *w,
                                  int64_t N, void *y, int64_t ldy, int32_t y_dtype,
                                  int64_t total_rows, int32_t policy, int32_t sensitive, void *ws,
                                  size_t ws_bytes, nvfp4_stream_t stream);

/* ---- mixture-of-experts feed-forward: fused epilogues of the grouped GEMM ----
 * The pages run MoE models (Qwen3 MoE) through the NVFP4 path ([LCP], MoE
 * operations; [ADA], model list) without printing the expert formula; the
 * reading taken is the SwiGLU expert of those models,
 *   h = SiLU(x W_gate^T) * (x W_up^T),  SiLU(v) = v / (1 + exp(-v)),
 *   y(t) = sum over the routed rows j of token t of g_j * (h_j W_down^T),
 * with both products the grouped W4A4 contraction of nvfp4_grouped_gemm
 * (same a / row_idx / expert_offsets / E / total_rows conventions; W4A4
 * route, TENSOR_FP32 only). */

/* Up projection with the SwiGLU fused into the epilogue.
 *  w_gate_up: the E experts' gate and up weights [I, K] each, stacked as one
 *    NVFP4 tensor [E * 2I, K] (one tensor scale per expert, second =
 *    float[E], MMA_TILED) in which expert e's rows e*2I + 256b + r hold gate
 *    row 128b + r for r < 128 and up row 128b + r - 128 for r >= 128 (gate
 *    and up interleaved in 128-row blocks).  I % 128 == 0.
 *  Output, exactly one of:
 *    h [total_rows, I] BF16/FP32 (h_dtype), row stride ldh elements with
 *      ldh * element size % 16 == 0, 16-byte aligned;
 *    h_q: NVFP4 [total_rows, I] (rows == total_rows, K == I, TENSOR_FP32,
 *      MMA_TILED) encoded as nvfp4_gemm_nvfp4_out does under the given
 *      device tensor scale h_q->second, with h_amax (optional) updated to
 *      max(*h_amax, max|h|); padding-row scales are zeroed.  Ready to be the
 *      `h` of nvfp4_moe_down_combine.
 *  Row j of the output is routed row j (expert e owns offsets[e] ..
 *  offsets[e+1]-1); rows past offsets[E] are untouched. */
nvfp4_status nvfp4_moe_up_swiglu(const nvfp4_tensor *a, const int32_t *row_idx,
                                 const int64_t *expert_offsets, int32_t E,
                                 const nvfp4_tensor *w_gate_up, int64_t I, void *h, int64_t ldh,
                                 int32_t h_dtype, nvfp4_tensor *h_q, float *h_amax,
                                 int64_t total_rows, void *ws, size_t ws_bytes,
                                 nvfp4_stream_t stream);

/* Down projection with the gate-weighted combine fused into the epilogue:
 *   y[token_idx[j], :] += gate_w[j] * (h[j, :] W_{e(j)}^T)
 * for every routed row j < offsets[E], e(j) the expert owning row j.
 *  h: NVFP4 routed rows [total_rows, I] (TENSOR_FP32, MMA_TILED), read in
 *    order (no index list).  w_down: [E * N, I] stacked, N % 128 == 0.
 *  token_idx: device int32[total_rows], values in [0, T) (rows with other
 *    values add nothing); gate_w: device float[total_rows].
 *  y: FP32 [T, N], row stride ldy (ldy % 4 == 0, 16-byte aligned), holding
 *    the value to add to (zeros, or the residual stream).  The additions are
 *    atomic and their order is unspecified, so the last bits of y may vary
 *    from run to run. */
nvfp4_status nvfp4_moe_down_combine(const nvfp4_tensor *h, const int64_t *expert_offsets, int32_t E,
                                    const nvfp4_tensor *w_down, int64_t N,
                                    const int32_t *token_idx, const float *gate_w, float *y,
                                    int64_t ldy, int64_t T, int64_t total_rows, void *ws,
                                    size_t ws_bytes, nvfp4_stream_t stream);

/* ---- NVFP4 paged KV cache and decode attention -------------------------------
 * "The FP4 Inflection" (serving-engine section) keeps the KV cache in FP4 with
 * paged attention as its consumer; the [TRT] engine build pages it in blocks
 * of 64 tokens; [ADA] pairs a low-precision cache with its own decode kernel.
 * Readings: every cached key / value head vector (head_dim 128) is encoded by
 * the activation block encoder ([TRT] item 2: 16 elements along head_dim, E4M3
 * block scales) under a static FP32 tensor scale per cache tensor fixed
 * beforehand (calibration), and decode attention is scaled dot-product
 * attention of one query token over its sequence's cached tokens, query head
 * h reading KV head h / (num_heads / num_kv_heads).
 *
 * An FP8 cache ([ADA]: a custom FP8 key-value cache) is the alternative
 * format: every element E4M3(x * 1/s) in binary32 (the per-token FP8 rule
 * under the static scale s), no block scales.
 *
 * Cache layout: `pages` is uint8 [num_pages][num_kv_heads][page block], one
 * contiguous block per page (64 token slots) and KV head, owned by the
 * caller; a sequence's pages are listed in its block-table row.
 * NVFP4_KV_NVFP4, 9216-byte blocks, two 32-token halves of 4608 bytes
 * (half h at byte 4608 h holds tokens 32h .. 32h + 31 of the page):
 *   [0, 2048)     key codes   [4 dim chunks][32 key slots][16]: chunk q
 *                 holds dims 32q .. 32q + 31, element 2j in the low nibble
 *                 of byte j; token k of the half sits in key slot
 *                 8*((k>>1)&3) + 2*(k>>3) + (k&1)
 *   [2048, 2304)  key scales  [32 key slots][8] E4M3
 *   [2304, 4352)  value codes [128 dims][16]   dim-major: byte j of row d
 *                 holds tokens 2j (low nibble) and 2j+1 of dimension d
 *   [4352, 4608)  value scales [8 blocks][32 tokens]
 * NVFP4_KV_FP8, 16384-byte blocks, two 32-token halves of 8192 bytes
 * (half h at byte 8192 h holds tokens 32h .. 32h + 31 of the page):
 *   [0, 4096)     keys   [8 dim chunks][32 key slots][16] E4M3: chunk q holds
 *                 dims 16q .. 16q + 15; token k of the half sits in key slot
 *                 (k&16) | ((k&2)<<2) | ((k>>1)&6) | (k&1)
 *   [4096, 8192)  values [2 token groups][128 dims][16] E4M3: byte j of row
 *                 d of group u holds token 16u + j of dimension d.
 * (The key slot orders put the 8 keys the attention reads together in 8
 * consecutive 16-byte rows.)
 * Both: k_scale, v_scale are device float[1] tensor scales.  A page belongs
 * to one sequence; slots past a sequence's length may hold anything (the
 * attention ignores them). */
typedef enum nvfp4_kv_format {
    NVFP4_KV_NVFP4 = 0,
    NVFP4_KV_FP8 = 1
} nvfp4_kv_format;

typedef struct nvfp4_kv_cache {
    void *pages;
    const float *k_scale;
    const float *v_scale;
    int32_t num_pages;
    int32_t num_kv_heads;
    int32_t head_dim;    /* 128 */
    int32_t page_tokens; /* 64 */
    int32_t format;      /* nvfp4_kv_format */
} nvfp4_kv_cache;

/* Encodes one new token per sequence into the cache: k_bf16 / v_bf16 BF16
 * [B][num_kv_heads][128]; sequence b's token goes to slot positions[b] % 64 of
 * page block_table[b * max_pages + positions[b] / 64].  Sequences whose
 * position or page is out of range are skipped.  Two sequences must not write
 * the same page in one call. */
nvfp4_status nvfp4_kv_append(const nvfp4_kv_cache *kv, const void *k_bf16, const void *v_bf16,
                             const int32_t *positions, const int32_t *block_table, int32_t max_pages,
                             int32_t B, nvfp4_stream_t stream);

/* One decode step of attention: q BF16 [B][num_heads][128]; sequence b
 * attends to its first min(ctx_lens[b], max_ctx) cached tokens;
 * out[b][h] = sum_t softmax_t(sm_scale * q[b][h] . k_t) v_t with the cached
 * keys and values decoded (E2M1 x E4M3 x tensor scale, or E4M3 x tensor
 * scale in the FP8 format), BF16 or FP32
 * [B][num_heads][128]; an empty context gives zeros.  num_heads is a multiple
 * of num_kv_heads with at most 16 query heads per KV head, and B and
 * num_kv_heads are at most 65535 (else NVFP4_ERR_UNSUPPORTED_SHAPE).  Long
 * contexts are split across CTAs and merged in a second kernel.
 * Workspace: nvfp4_workspace_size(NVFP4_OP_KV_DECODE, B, num_heads, max_ctx,
 * num_kv_heads). */
nvfp4_status nvfp4_kv_decode_attention(const nvfp4_kv_cache *kv, const void *q_bf16, int32_t num_heads,
                                       const int32_t *ctx_lens, const int32_t *block_table,
                                       int32_t max_pages, int32_t B, int32_t max_ctx, float sm_scale,
                                       void *out, int32_t out_dtype, void *ws, size_t ws_bytes,
                                       nvfp4_stream_t stream);

/* ---- no-allocation variant --------------------------------------------------- */

/* W4A4 product Y[M, N] = A[M, K] * W[N, K]^T of pre-quantised NVFP4
 * activations a_q (TENSOR_FP32, MMA_TILED) and weights w, for callers that
 * cannot allocate device memory at call time: a host framework that owns all
 * device memory through its own pool and forbids cudaMalloc, a plugin without
 * allocation rights, or a serving loop that must never reach the allocator.
 * The pages have no counterpart to this entry point; it is the nvfp4_gemm
 * W4A4 kernel with its scratch moved into the library.
 *  - Takes no workspace and allocates nothing (no cudaMalloc, no cudaFree, no
 *    allocating library call).  Its scratch (status word, stream-K FP32
 *    partial tiles and ready flags) is a fixed 4 MiB array inside the
 *    library, which every GPU that loads the library holds until exit.
 *  - A shape whose scratch would exceed 4 MiB (M <= 128 shapes that use
 *    stream-K need about 1 KiB * M per SM for their partial tiles) is
 *    rejected with NVFP4_ERR_WORKSPACE before anything is enqueued.
 *  - The first call on a device looks up the array's device address for that
 *    device (with that device current); make that first call before any
 *    stream capture.
 *  - Every call shares the one array and zeroes the part it uses on `stream`
 *    before the kernel runs; calls that overlap on the GPU (other streams,
 *    other threads) race on it and must be serialised by the caller.
 *  - Device-side status (a bounded wait that ran out, leaving part of y
 *    unspecified) is kept in that array: read it with
 *    nvfp4_gemm_w4a4_noalloc_status before the next call clears it.
 *  y: [M, N] with row stride ldy, y_dtype BF16 or FP32, 16-byte aligned.
 *  The tensors are checked as nvfp4_gemm checks them (same error codes);
 *  NVFP4_SCALE_MACRO_FP16 tensors give NVFP4_ERR_UNSUPPORTED. */
nvfp4_status nvfp4_gemm_w4a4_noalloc(const nvfp4_tensor *a_q, const nvfp4_tensor *w, void *y, int64_t ldy,
                                     int32_t y_dtype, nvfp4_stream_t stream);

/* Device status of the most recent nvfp4_gemm_w4a4_noalloc call(s) on the
 * current device: waits for `stream`'s earlier work, then writes NVFP4_OK,
 * NVFP4_ERR_TIMEOUT (a bounded wait ran out; part of y is unspecified) or
 * NVFP4_ERR_NONFINITE_INPUT to *device_status (host memory) and clears the
 * word.  Allocates nothing.  Like the calls themselves, it shares the
 * library's scratch array: calls on other streams race with it. */
nvfp4_status nvfp4_gemm_w4a4_noalloc_status(nvfp4_stream_t stream, int32_t *device_status);

/* ---- diagnostics ----------------------------------------------------------- */

/* Runs the kernels' own element conversions on n floats: out_e2m1[i] is the
 * E2M1 code of in[i] (round to nearest even, saturating at 6, sign kept) and
 * out_e4m3[i] the E4M3 code (round to nearest even, saturating at 448).
 * Used to check the device conversions exhaustively against the oracle. */
nvfp4_status nvfp4_probe_convert(const float *in, int64_t n, uint8_t *out_e2m1, uint8_t *out_e4m3,
                                 nvfp4_stream_t stream);

/* Dense FP4 tensor-core rate of this GPU, the denominator of the W4A4 GEMM
 * roofline ("NVIDIA Ships TensorRT-LLM 0.16: Native FP4 Quantization for
 * Blackwell B200", section "The Mathematical Breakthrough of Microscopic FP4
 * Scaling", item 3: the tensor cores take FP4 codes and their micro-scales).
 * Launches one CTA per SM; each issues `iters` x 4 back-to-back block-scaled
 * MMAs (kind::mxf4nvf4, M = 128, N = 256, K = 64: 4194304 FLOP each) on
 * operands held in shared memory and TMEM, so nothing but the tensor core
 * limits it, and writes its cycle count (clock64) to cycles[cta] (device
 * memory, nvfp4_sm_count() entries, 8-byte aligned; ~0 if its bounded wait
 * ran out).  FLOP per cycle and SM = iters * 4 * 4194304 / cycles; time the
 * launch with events on `stream` for FLOP/s at the clock it ran at.
 * iters in 1 .. 2^24.  Asynchronous; the caller owns `cycles`. */
nvfp4_status nvfp4_diag_fp4_mma_rate(int32_t iters, uint64_t *cycles, nvfp4_stream_t stream);

/* Diagnostic: the copy engine's streaming rate as the W4A4 GEMM's weight
 * operand sees it.  Streams the rows x row_bytes byte matrix w (device,
 * 16-byte aligned, row-major; rows a multiple of 256 up to 2^31, row_bytes a
 * multiple of 128 in 128 .. 2^20) into shared memory with the GEMM's weight
 * boxes (128 bytes x 256 rows, 128-byte swizzle) through a 6-deep ring of
 * 32 KB stages on `grid` CTAs (1 .. 4096, one warp each), each CTA taking an
 * equal contiguous range of the boxes, and does nothing else with them.
 * Time the launch with events on `stream`: rows x row_bytes bytes over that
 * time is the streaming ceiling of the decode GEMM (whose weights arrive
 * exactly so).  A bounded wait that runs out ORs NVFP4's timeout bit (2)
 * into *status (a device word, 4-byte aligned, caller-owned).
 * Asynchronous. */
nvfp4_status nvfp4_diag_tma_stream(const uint8_t *w, int64_t rows, int64_t row_bytes, int32_t grid,
                                   uint32_t *status, nvfp4_stream_t stream);

/* Test-only failure injection for the device-side failure detection: runs the
 * W4A4 GEMM of pre-quantised a_q (TENSOR_FP32, MMA_TILED) and w on a shape
 * that uses stream-K, with CTA `skip_cta` never raising its ready flag, and
 * every bounded wait limited to timeout_ns (1 .. 1e10).  If skip_cta's range
 * starts inside a tile, that tile's owner gives up waiting after timeout_ns,
 * sets TIMEOUT in the workspace status word and exits cleanly (no fault, no
 * hang; the context stays usable); that tile of y is then unspecified.
 * Afterwards call nvfp4_workspace_init: the abandoned flags stay raised.
 * Returns UNSUPPORTED_SHAPE for a shape that does not run stream-K. */
nvfp4_status nvfp4_diag_streamk_skip_flag(const nvfp4_tensor *a_q, const nvfp4_tensor *w, void *y,
                                          int64_t ldy, int32_t y_dtype, int32_t skip_cta,
                                          uint64_t timeout_ns, void *ws, size_t ws_bytes,
                                          nvfp4_stream_t stream);

/* Number of streaming multiprocessors of the current device (0 on error). */
int32_t nvfp4_sm_count(void);

/* How the W4A4 route of nvfp4_gemm (tensor-scale mode) spreads the work for
 * M activation rows, N weight rows and depth K: NVFP4_PATH_WHOLE_TILES (each
 * persistent CTA takes whole 128-row output tiles) or NVFP4_PATH_STREAMK
 * (M <= 128 with too few N tiles to fill the SMs: the K stages are spread over
 * the SMs and partial tiles meet in the workspace).  -1 for sizes nvfp4_gemm
 * rejects.  Host-side query; launches nothing. */
enum { NVFP4_PATH_WHOLE_TILES = 1, NVFP4_PATH_STREAMK = 2 };
int32_t nvfp4_gemm_kernel_path(int64_t M, int64_t N, int64_t K);

/* Bounds-checked build.  libnvfp4_checked.so is the same library compiled
 * with NVFP4_CHECK_BOUNDS: before each access its kernels test that shared
 * memory destinations and operands lie in the CTA's dynamic shared memory
 * (bulk and tensor copies aligned, tensor-map x a multiple of 16 bytes),
 * TMEM column ranges within the 512 columns, and global loads and stores
 * within the byte range the call's arguments grant each tensor (its rows
 * and leading dimension in the layout this header documents).  A failed test
 * skips its access and is counted; the first failure of each translation unit
 * keeps its site (file and line), the offending value and its limit.
 * Outputs of a call with a failed test are unspecified (the call's bounded
 * waits may also record TIMEOUT for copies that were skipped).
 *
 * nvfp4_diag_bounds_checked: 1 in the checked build, 0 in the normal one.
 * nvfp4_diag_bounds_record: synchronises the device, then writes the total
 * number of failed tests since the last clear to *failures and, when there is
 * one, the first recorded failure's site ("unit.cu:line", or
 * "unit.cu via ptx.cuh:line" for a test inside a shared wrapper) to `where`
 * (NUL-terminated, at most where_len bytes; may be null) and its value and
 * limit to *value and *limit (may be null); clear != 0 resets the records.
 * Returns NVFP4_ERR_UNSUPPORTED in the normal build.
 *
 * nvfp4_diag_bounds_selftest: stores the byte 1 to every offset of
 * [0, span_bytes + 64) of the device buffer buf (buf_bytes >= span_bytes +
 * 64, so every store is inside buf) from a kernel that tests each store
 * against a span of span_bytes (1 .. 2^30): the checked build skips and
 * counts the last 64 stores, the normal build makes them all.  Asynchronous
 * on `stream`; the caller owns buf. */
int32_t nvfp4_diag_bounds_checked(void);
nvfp4_status nvfp4_diag_bounds_record(uint64_t *failures, char *where, int32_t where_len, uint64_t *value,
                                      uint64_t *limit, int32_t clear);
nvfp4_status nvfp4_diag_bounds_selftest(uint8_t *buf, uint64_t buf_bytes, uint64_t span_bytes,
                                        nvfp4_stream_t stream);

/* Library version string. */
const char *nvfp4_version(void);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_H */
