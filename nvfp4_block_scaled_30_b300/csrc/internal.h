// Host-side declarations shared by the library's translation units.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/nvfp4.h"

namespace nv4 {

// Workspace header: the first 256 bytes; word 0 is the sticky device status.
constexpr size_t WS_HEADER = 256;
constexpr uint32_t ST_NONFINITE = 1u;
constexpr uint32_t ST_TIMEOUT = 2u;
// Partial maxima written by the first quantiser pass (one word per CTA).
constexpr int AMAX_MAX_CTAS = 1024;
constexpr size_t WS_AMAX_BYTES = AMAX_MAX_CTAS * sizeof(uint32_t);

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
// Bytes of the MMA-tiled scale layout of rows x cols elements (atoms of 128
// rows x 64 columns, 512 bytes each).
inline uint64_t tiled_scale_bytes(int64_t rows, int64_t cols)
{
    return rows > 0 ? (uint64_t)ceil_div(rows, 128) * (uint64_t)(cols / 64) * 512u : 0u;
}
// Bytes of a rows x cols matrix of esz-byte elements with row pitch ld
// (elements), the last row ending at its last element.
inline uint64_t matrix_bytes(int64_t rows, int64_t cols, int64_t ld, int64_t esz)
{
    return rows > 0 && cols > 0 ? (uint64_t)((rows - 1) * ld + cols) * (uint64_t)esz : 0u;
}

int device_sm_count();

// A byte range [lo, lo + bytes) of global memory that a call's arguments
// grant a tensor (the bounds-checked build tests accesses against it).
struct Span {
    uint64_t lo = 0, bytes = 0;
};

__host__ __device__ __forceinline__ Span span_of(const void *p, uint64_t bytes)
{
    Span s;
    s.lo = reinterpret_cast<uint64_t>(p);
    s.bytes = p ? bytes : 0;
    return s;
}

// Argument checks of an nvfp4_tensor shared by the entry points (null or
// misaligned pointers, enums, sizes: NVFP4_ERR_INVALID_ARG; K not a multiple
// of 16, of 64 for the MMA-tiled layout or of 256 in macro mode:
// NVFP4_ERR_UNSUPPORTED_SHAPE); need_tiled requires the MMA-tiled layout.
nvfp4_status check_tensor(const nvfp4_tensor *t, bool need_tiled);

// Launch with programmatic stream serialisation: the grid may start while
// the previous grid in the stream is still running.  Every kernel launched
// this way executes griddepcontrol.wait before it touches memory that the
// previous grid reads or writes, so its completion still implies that of
// the previous grid.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), int grid, int block, size_t smem, cudaStream_t stream, Args &&...args)
{
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

// ---- quantisers (quantize.cu) ------------------------------------------------
// zero_pad: also zero the scales of the tiled layout's padding rows (the
// public quantiser promises them; the GEMM never reads them into stored
// output, and its workspace keeps them zero from initialisation).
cudaError_t launch_nvfp4_quantize(const uint16_t *x, int64_t rows, int64_t K, int64_t ldx, uint8_t *codes,
                                  uint8_t *scales, void *second, int mode, int layout, uint32_t *amax_partial,
                                  uint32_t *status, cudaStream_t stream, bool zero_pad = true);
cudaError_t launch_fp8_quantize(const uint16_t *x, int64_t rows, int64_t K, int64_t ldx, uint8_t *a, float *s_t,
                                uint32_t *status, cudaStream_t stream);
cudaError_t launch_fp4_mma_rate(int iters, uint64_t *cycles, cudaStream_t stream);
cudaError_t launch_bounds_selftest(uint8_t *buf, uint64_t span_bytes, cudaStream_t stream);
cudaError_t launch_tma_stream(const uint8_t *w, int64_t rows, int64_t row_bytes, int grid, uint32_t *status,
                              cudaStream_t stream);
cudaError_t launch_probe_convert(const float *in, int64_t n, uint8_t *o2, uint8_t *o3, cudaStream_t stream);
cudaError_t launch_finalize_bf16(const float *acc, int64_t rows, int64_t cols, int64_t ld_acc, uint16_t *y,
                                 int64_t ldy, cudaStream_t stream);

// ---- GEMMs (gemm.cu) -----------------------------------------------------------
struct DenseGemmArgs {
    // MMA operand A (M side, tiles of 128 rows) and B (N side).
    const uint8_t *a_codes;
    const uint8_t *a_scales; // tiled
    const float *a_second;
    int64_t a_rows;
    const uint8_t *b_codes;
    const uint8_t *b_scales; // tiled
    const float *b_second;
    int64_t b_rows;
    int64_t K;
    // output element (i, j) of the accumulator tile goes to out[i*ld_i + j*ld_j]
    void *out;
    int64_t ld_i, ld_j;
    int out_dtype;           // 0 bf16, 1 fp32
    // stream-K (spread K stages evenly over the SMs, only when a_rows <= 128):
    // slots holds one FP32 partial tile [a_rows][N tile] per CTA of the grid
    // (streamk_slot_floats each) and flags one word per CTA; the flags are
    // zero between calls and left zero by the kernel.
    bool streamk;
    float *slots;
    uint32_t *flags;
    // the previous grid in the stream is this call's activation quantiser:
    // the first stages' weight copies may start before waiting for it
    bool b_early;
    // test-only: stream-K CTA that skips raising its ready flag (-1: none)
    int diag_skip_flag = -1;
    // NVFP4 output instead of out (whole tiles only, b_rows % 64 == 0):
    // codes [a_rows][b_rows/2], MMA-tiled scales, encoded under the device
    // tensor scale *yq_scale; the largest |Y| (float bits) is max-reduced
    // into *yq_amax when yq_amax is set
    uint8_t *yq_codes;
    uint8_t *yq_scales;
    const float *yq_scale;
    uint32_t *yq_amax;
    uint32_t *status;
    uint64_t timeout_ns;
};
cudaError_t launch_w4a4_dense(const DenseGemmArgs &g, cudaStream_t stream);
int w4a4_dense_bn(int64_t b_rows);
// Stream-K launch shape of the dense W4A4 GEMM: whether it is used, the grid
// size, and the workspace it needs (partial slots, then flags).
struct StreamKPlan {
    bool used = false;
    int grid = 0;
    size_t slot_bytes = 0; // all slots, 256-aligned
    size_t flag_bytes = 0; // all flags, 256-aligned
};
StreamKPlan w4a4_streamk_plan(int64_t M, int64_t N, int64_t K, int sms);

struct GroupedGemmArgs {
    const uint8_t *a_codes;
    const uint8_t *a_scales; // tiled, rows padded to 128
    const float *a_second;
    int64_t a_rows;
    const int32_t *row_idx;  // may be null
    const int64_t *offsets;  // device [E+1]
    int E;
    const uint8_t *w_codes;  // [E*N][K/2]
    const uint8_t *w_scales; // tiled over E*N rows
    const float *w_second;   // [E]
    int64_t N, K;
    void *out;
    int64_t ldy;
    int out_dtype;
    int64_t total_rows;
    uint32_t *status;
    uint64_t timeout_ns;
    // epilogue: EPI_PLAIN (out = alpha * acc), EPI_SWIGLU (N = 2I stacked
    // rows per expert interleaving 128-row gate and up blocks; out, or the
    // NVFP4 output yq_* when yq_codes is set, gets SiLU(gate) * up, [rows, I])
    // or EPI_COMBINE (out FP32 [tokens][ldy]: row comb_idx[j] += comb_w[j] *
    // alpha * acc of routed row j, atomically)
    int epi;
    const int32_t *comb_idx;
    const float *comb_w;
    int64_t comb_rows;       // tokens; rows with other token indices add nothing
    uint8_t *yq_codes;
    uint8_t *yq_scales;
    const float *yq_scale;
    uint32_t *yq_amax;
};
enum { EPI_PLAIN = 0, EPI_SWIGLU = 1, EPI_COMBINE = 2 };
cudaError_t launch_w4a4_grouped(const GroupedGemmArgs &g, cudaStream_t stream);

struct W4A8GemmArgs {
    const uint8_t *a_fp8;    // [M][K]
    const float *s_t;        // [M]
    int64_t M;
    const uint8_t *w_codes;  // [N][K/2] ([E*N][K/2] grouped)
    const uint8_t *w_scales; // tiled
    const float *w_second;   // [1] ([E] grouped)
    int64_t N, K;
    void *out;
    int64_t ldy;
    int out_dtype;
    uint32_t *status;
    uint64_t timeout_ns;
    // grouped (E > 0): N per expert (% 128 == 0); expert e owns output rows
    // offsets[e] .. offsets[e+1]-1, routed row j reads activation row
    // row_idx[j] (or j when row_idx is null)
    int E;
    const int64_t *offsets;
    const int32_t *row_idx;
    int64_t total_rows;
};
cudaError_t launch_w4a8(const W4A8GemmArgs &g, cudaStream_t stream);

// ---- NVFP4 / FP8 paged KV cache (kv_attention.cu) ------------------------------------
// head_dim 128, 64 tokens per page; layouts in include/nvfp4.h (nvfp4_kv_cache)
enum { KV_FMT_NVFP4 = 0, KV_FMT_FP8 = 1 };
struct KvAppendArgs {
    int fmt;
    const uint16_t *k_new, *v_new; // BF16 [B][H_kv][128]
    const int32_t *positions;      // [B] slot of the new token in its sequence
    const int32_t *block_table;    // [B][max_pages]
    int B, H_kv, max_pages, num_pages;
    uint8_t *pages;                // [num_pages][H_kv][page block]
    const float *k_scale, *v_scale;
    Span sp_k_new, sp_v_new, sp_positions, sp_block_table, sp_pages, sp_k_scale, sp_v_scale; // set by the launch
};
cudaError_t launch_kv_append(const KvAppendArgs &a, cudaStream_t stream);

struct KvAttnArgs {
    int fmt;
    const uint16_t *q;             // BF16 [B][H][128]
    const int32_t *ctx_lens;       // [B]
    const int32_t *block_table;    // [B][max_pages]
    int B, H, H_kv, max_pages, num_pages, max_ctx;
    const uint8_t *pages;          // [num_pages][H_kv][page block]
    const float *k_scale, *v_scale;
    float sm_scale;
    int keys_per_split, n_splits;  // keys_per_split % 64 == 0
    void *out;                     // [B][H][128]
    int out_dtype;
    float *partial;                // [B][H][n_splits][130] when n_splits > 1
    uint32_t *status;
    uint64_t timeout_ns;
    Span sp_q, sp_ctx_lens, sp_block_table, sp_pages, sp_k_scale, sp_v_scale, sp_out, sp_partial; // set by the launch
};
size_t kv_attn_partial_bytes(int B, int H, int n_splits);
// Context splits of one decode-attention call: one wave of ctas_per_sm CTAs
// per SM, at least 256 keys per split.  kv_ctas_per_sm: the attention
// kernel's occupancy for a cache format and query heads per KV head.
int kv_ctas_per_sm(int fmt, int64_t group);
void kv_attn_splits(int64_t B, int64_t H_kv, int64_t max_ctx, int sms, int ctas_per_sm, int &n_splits,
                    int &keys_per_split);
cudaError_t launch_kv_decode(const KvAttnArgs &a, cudaStream_t stream);

struct MacroGemmArgs {
    const uint8_t *a_codes;
    const uint8_t *a_scales;  // tiled
    const uint16_t *a_macro;  // [M][K/256] binary16
    int64_t M;
    const uint8_t *w_codes;
    const uint8_t *w_scales;  // tiled
    const uint16_t *w_macro;  // [N][K/256]
    int64_t N, K;
    void *out;
    int64_t ldy;
    int out_dtype;
    uint32_t *status;
    uint64_t timeout_ns;
};
cudaError_t launch_w4a4_macro(const MacroGemmArgs &g, cudaStream_t stream);

// Tensor-map creation through the driver entry point (no libcuda link).
CUresult make_tmap_2d_u8(CUtensorMap *map, const void *base, uint64_t inner_bytes, uint64_t rows,
                         uint64_t row_pitch_bytes, uint32_t box_inner, uint32_t box_rows, bool swizzle128);
CUresult make_tmap_2d_u8_swizzle(CUtensorMap *map, const void *base, uint64_t inner_bytes, uint64_t rows,
                                 uint64_t row_pitch_bytes, uint32_t box_inner, uint32_t box_rows,
                                 CUtensorMapSwizzle swizzle);
// The MMA-tiled scale atoms of a [groups x 128 rows][k64 x 64] tensor viewed
// as a 4-D tensor [groups][k64][4][128 bytes]: one box of box_k64 atoms of
// box_groups consecutive row groups lands as [group][atom][512 bytes].
CUresult make_tmap_scale_atoms(CUtensorMap *map, const void *scales, uint64_t groups, uint64_t k64,
                               uint32_t box_k64, uint32_t box_groups);


} // namespace nv4
