// C ABI of libnvfp4: argument checks, workspace layout, precision-policy
// routing and launch configuration.  Declarations and contracts are in
// include/nvfp4.h.  Every check runs before any work is enqueued, so an
// error return means nothing was launched ("fail fast, no silent fallback",
// "AdaLLM Breakthrough: First NVFP4-Only Inference Engine for RTX 4090
// Unveiled").
#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <cudaTypedefs.h>
#include <mutex>

#include "internal.h"

namespace nv4 {

static constexpr uint64_t DEFAULT_TIMEOUT_NS = 2000000000ull; // bounded waits: 2 s
static constexpr int64_t MAX_DIM = (int64_t)1 << 30;

int device_sm_count()
{
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return 148;
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
        cache[dev] = n;
    }
    return cache[dev];
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

CUresult make_tmap_2d_u8_swizzle(CUtensorMap *map, const void *base, uint64_t inner_bytes, uint64_t rows,
                                 uint64_t row_pitch_bytes, uint32_t box_inner, uint32_t box_rows,
                                 CUtensorMapSwizzle swizzle)
{
    auto fn = encode_fn();
    if (!fn)
        return CUDA_ERROR_NOT_FOUND;
    cuuint64_t dims[2] = {inner_bytes, rows};
    cuuint64_t strides[1] = {row_pitch_bytes};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

CUresult make_tmap_scale_atoms(CUtensorMap *map, const void *scales, uint64_t groups, uint64_t k64,
                               uint32_t box_k64, uint32_t box_groups)
{
    auto fn = encode_fn();
    if (!fn)
        return CUDA_ERROR_NOT_FOUND;
    cuuint64_t dims[4] = {128, 4, k64, groups};
    cuuint64_t strides[3] = {128, 512, k64 * 512};
    cuuint32_t box[4] = {128, 4, box_k64, box_groups};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void *>(scales), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

CUresult make_tmap_2d_u8(CUtensorMap *map, const void *base, uint64_t inner_bytes, uint64_t rows,
                         uint64_t row_pitch_bytes, uint32_t box_inner, uint32_t box_rows, bool swizzle128)
{
    return make_tmap_2d_u8_swizzle(map, base, inner_bytes, rows, row_pitch_bytes, box_inner, box_rows,
                                   swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE);
}

// ---- workspace layout ------------------------------------------------------------

struct WsLayout {
    size_t amax = 0;      // partial maxima of the first quantiser pass
    size_t a_codes = 0;   // on-the-fly NVFP4 activations
    size_t a_scales = 0;
    size_t a_second = 0;  // float (tensor mode) or binary16 [M][K/256] (macro)
    size_t a_fp8 = 0;     // on-the-fly FP8 activations (W4A8 route)
    size_t a_st = 0;
    size_t sk_slots = 0;  // stream-K FP32 partial tiles, one per CTA
    size_t sk_flags = 0;  // stream-K ready flags, one per CTA, kept zero between calls
    size_t kv_partial = 0; // decode attention: per-split partial outputs
    size_t total = 0;
};

static WsLayout ws_layout(int op, int64_t M, int64_t N, int64_t K, int64_t E = 0)
{
    WsLayout L;
    size_t off = WS_HEADER;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off = align_up(off + bytes, 256);
        return o;
    };
    L.amax = take(WS_AMAX_BYTES);
    if (op == NVFP4_OP_GEMM || op == NVFP4_OP_GROUPED_GEMM_X) {
        const int64_t mpad = ceil_div(M, 128) * 128;
        const int64_t kpad = ceil_div(K, 64) * 64;
        L.a_codes = take((size_t)(M * (K / 2)));
        L.a_scales = take((size_t)(mpad * (kpad / 16)));
        L.a_second = take(std::max<size_t>(16, (size_t)(M * (K / 256) * 2)));
        L.a_fp8 = take((size_t)(M * K));
        L.a_st = take((size_t)(M * 4));
    }
    if (op == NVFP4_OP_KV_DECODE) {
        // M = sequences, N = query heads, K = max context, E = KV heads
        int ns = 1, kps = 64;
        // sized for the format with the most splits
        kv_attn_splits(M, E, K, device_sm_count(), kv_ctas_per_sm(KV_FMT_NVFP4, E > 0 ? N / E : N), ns, kps);
        const size_t pb = kv_attn_partial_bytes((int)M, (int)N, ns);
        if (pb)
            L.kv_partial = take(pb);
    }
    if (op == NVFP4_OP_GEMM) {
        const StreamKPlan pl = w4a4_streamk_plan(M, N, K, device_sm_count());
        if (pl.used) {
            L.sk_slots = take(pl.slot_bytes);
            L.sk_flags = take(pl.flag_bytes);
        }
    }
    L.total = off;
    return L;
}

static uint32_t *status_word(void *ws) { return static_cast<uint32_t *>(ws); }

static uint8_t *ws_at(void *ws, size_t off) { return static_cast<uint8_t *>(ws) + off; }

static bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

static nvfp4_status check_ws(void *ws, size_t ws_bytes, size_t need)
{
    if (!ws || !aligned(ws, 256) || ws_bytes < need)
        return NVFP4_ERR_WORKSPACE;
    return NVFP4_OK;
}

nvfp4_status check_tensor(const nvfp4_tensor *t, bool need_tiled)
{
    if (!t || !t->second || (t->rows > 0 && (!t->codes || !t->scales)))
        return NVFP4_ERR_INVALID_ARG;
    if (!aligned(t->codes, 16) || !aligned(t->scales, 16) || !aligned(t->second, 4))
        return NVFP4_ERR_INVALID_ARG;
    if (t->mode != NVFP4_SCALE_TENSOR_FP32 && t->mode != NVFP4_SCALE_MACRO_FP16)
        return NVFP4_ERR_INVALID_ARG;
    if (t->layout != NVFP4_LAYOUT_ROW_MAJOR && t->layout != NVFP4_LAYOUT_MMA_TILED)
        return NVFP4_ERR_INVALID_ARG;
    if (need_tiled && t->layout != NVFP4_LAYOUT_MMA_TILED)
        return NVFP4_ERR_INVALID_ARG;
    if (t->rows < 0 || t->K <= 0 || t->rows > MAX_DIM || t->K > MAX_DIM)
        return NVFP4_ERR_INVALID_ARG;
    if (t->K % 16 != 0 || (t->layout == NVFP4_LAYOUT_MMA_TILED && t->K % 64 != 0) ||
        (t->mode == NVFP4_SCALE_MACRO_FP16 && t->K % 256 != 0))
        return NVFP4_ERR_UNSUPPORTED_SHAPE;
    return NVFP4_OK;
}

static nvfp4_status from_cuda(cudaError_t e)
{
    if (e == cudaSuccess)
        return NVFP4_OK;
    return e == cudaErrorNotSupported ? NVFP4_ERR_UNSUPPORTED : NVFP4_ERR_CUDA;
}

// Stream-K pays off when whole tiles fill the SMs poorly (wave efficiency
// below 90%) and there are enough K stages to spread.
// W4A4 dense product of NVFP4 activations `a` ([M, K], tiled scales, tensor
// mode) and weights `w` ([N, K]) into y.
// With yq set, the output is NVFP4 (codes, tiled scales) under the device
// tensor scale yq->second instead of y; stream-K is then not used.
static nvfp4_status run_w4a4_dense(const uint8_t *a_codes, const uint8_t *a_scales, const float *a_second,
                                   int64_t M, const nvfp4_tensor *w, void *y, int64_t ldy, int y_dtype, void *ws,
                                   const WsLayout &L, bool after_quantiser, cudaStream_t stream,
                                   const nvfp4_tensor *yq = nullptr, float *y_amax = nullptr,
                                   int diag_skip_flag = -1, uint64_t timeout_ns = DEFAULT_TIMEOUT_NS)
{
    const int64_t N = w->rows, K = w->K;
    DenseGemmArgs g{};
    g.a_codes = a_codes;
    g.a_scales = a_scales;
    g.a_second = a_second;
    g.a_rows = M;
    g.b_codes = static_cast<const uint8_t *>(w->codes);
    g.b_scales = static_cast<const uint8_t *>(w->scales);
    g.b_second = static_cast<const float *>(w->second);
    g.b_rows = N;
    g.K = K;
    g.status = status_word(ws);
    g.timeout_ns = timeout_ns;
    g.diag_skip_flag = diag_skip_flag;
    g.out = y;
    g.out_dtype = y_dtype;
    g.ld_i = ldy;
    g.ld_j = 1;
    // stream-K when the plan (the same one that sized the workspace) says
    // so: partial tiles meet in the workspace slots; the kernel writes y
    // itself and leaves the flags zeroed
    g.b_early = after_quantiser;
    if (yq) {
        g.yq_codes = static_cast<uint8_t *>(yq->codes);
        g.yq_scales = static_cast<uint8_t *>(yq->scales);
        g.yq_scale = static_cast<const float *>(yq->second);
        g.yq_amax = reinterpret_cast<uint32_t *>(y_amax);
        return from_cuda(launch_w4a4_dense(g, stream));
    }
    g.streamk = L.sk_slots != 0;
    if (g.streamk) {
        g.slots = reinterpret_cast<float *>(ws_at(ws, L.sk_slots));
        g.flags = reinterpret_cast<uint32_t *>(ws_at(ws, L.sk_flags));
    }
    (void)N;
    return from_cuda(launch_w4a4_dense(g, stream));
}

// Records of the bounds-checked build, one per translation unit with
// kernels (registered by their static initialisers; constant-initialised
// here, so registration order does not matter).
#ifdef NVFP4_CHECK_BOUNDS
constexpr bool kCheckBounds = true;
#else
constexpr bool kCheckBounds = false;
#endif
namespace {
struct BoundsUnit {
    const void *symbol;
    const char *unit;
};
constexpr int MAX_BOUNDS_UNITS = 32;
BoundsUnit g_bounds_units[MAX_BOUNDS_UNITS];
int g_bounds_n = 0;
} // namespace

void register_bounds_record(const void *symbol, const char *unit)
{
    if (g_bounds_n < MAX_BOUNDS_UNITS)
        g_bounds_units[g_bounds_n++] = BoundsUnit{symbol, unit};
}

} // namespace nv4

using namespace nv4;

extern "C" {

const char *nvfp4_version(void) { return "nvfp4-b300 0.1 (sm_103a)"; }

int32_t nvfp4_sm_count(void)
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    return n;
}

int32_t nvfp4_gemm_kernel_path(int64_t M, int64_t N, int64_t K)
{
    if (M <= 0 || N <= 0 || K <= 0 || M > MAX_DIM || N > MAX_DIM || K > MAX_DIM || K % 64 != 0)
        return -1;
    const WsLayout L = ws_layout(NVFP4_OP_GEMM, M, N, K);
    return L.sk_slots != 0 ? NVFP4_PATH_STREAMK : NVFP4_PATH_WHOLE_TILES;
}

int32_t nvfp4_policy_route(int32_t policy, int32_t sensitive)
{
    switch (policy) {
    case NVFP4_POLICY_AUTO: return sensitive ? 8 : 4;
    case NVFP4_POLICY_Q4: return 4;
    case NVFP4_POLICY_Q8: return 8;
    default: return -1;
    }
}

nvfp4_status nvfp4_scale_bytes(int64_t rows, int64_t K, int32_t layout, size_t *bytes)
{
    if (!bytes || rows < 0 || K < 0 || rows > MAX_DIM || K > MAX_DIM)
        return NVFP4_ERR_INVALID_ARG;
    if (layout == NVFP4_LAYOUT_ROW_MAJOR) {
        if (K % 16 != 0)
            return NVFP4_ERR_UNSUPPORTED_SHAPE;
        *bytes = (size_t)rows * (size_t)(K / 16);
        return NVFP4_OK;
    }
    if (layout == NVFP4_LAYOUT_MMA_TILED) {
        if (K % 64 != 0)
            return NVFP4_ERR_UNSUPPORTED_SHAPE;
        *bytes = (size_t)ceil_div(rows, 128) * 128 * (size_t)(K / 16);
        return NVFP4_OK;
    }
    return NVFP4_ERR_INVALID_ARG;
}

nvfp4_status nvfp4_workspace_size(int32_t op, int64_t M, int64_t N, int64_t K, int32_t E, size_t *bytes)
{
    if (!bytes || M < 0 || N < 0 || K < 0 || E < 0 || M > MAX_DIM || N > MAX_DIM || K > MAX_DIM)
        return NVFP4_ERR_INVALID_ARG;
    if (op < NVFP4_OP_QUANTIZE || op > NVFP4_OP_KV_DECODE)
        return NVFP4_ERR_INVALID_ARG;
    *bytes = ws_layout(op, M, N, K, E).total;
    return NVFP4_OK;
}

nvfp4_status nvfp4_workspace_init(void *ws, size_t ws_bytes, nvfp4_stream_t stream)
{
    if (!ws || !aligned(ws, 256) || ws_bytes < WS_HEADER)
        return NVFP4_ERR_WORKSPACE;
    return from_cuda(cudaMemsetAsync(ws, 0, ws_bytes, (cudaStream_t)stream));
}

nvfp4_status nvfp4_device_status(void *ws, nvfp4_stream_t stream, int32_t *device_status)
{
    if (!ws || !device_status || !aligned(ws, 256))
        return NVFP4_ERR_INVALID_ARG;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    uint32_t w = 0;
    if (cudaMemcpy(&w, ws, 4, cudaMemcpyDeviceToHost) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    if (cudaMemset(ws, 0, 4) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    *device_status = (w & ST_NONFINITE) ? NVFP4_ERR_NONFINITE_INPUT : (w & ST_TIMEOUT) ? NVFP4_ERR_TIMEOUT : NVFP4_OK;
    return NVFP4_OK;
}

nvfp4_status nvfp4_quantize(const void *x_bf16, int64_t rows, int64_t K, int64_t ldx, nvfp4_tensor *out, void *ws,
                            size_t ws_bytes, nvfp4_stream_t stream)
{
    nvfp4_status st = check_tensor(out, false);
    if (st != NVFP4_OK)
        return st;
    if (rows < 0 || out->rows != rows || out->K != K || ldx < K || ldx % 8 != 0)
        return NVFP4_ERR_INVALID_ARG;
    if (rows > 0 && (!x_bf16 || !aligned(x_bf16, 16)))
        return NVFP4_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(NVFP4_OP_QUANTIZE, rows, 0, K);
    if ((st = check_ws(ws, ws_bytes, L.total)) != NVFP4_OK)
        return st;
    cudaStream_t s = (cudaStream_t)stream;
    if (rows == 0) {
        if (out->mode == NVFP4_SCALE_TENSOR_FP32)
            return from_cuda(cudaMemsetAsync(out->second, 0, 4, s));
        return NVFP4_OK;
    }
    return from_cuda(launch_nvfp4_quantize(static_cast<const uint16_t *>(x_bf16), rows, K, ldx,
                                           static_cast<uint8_t *>(out->codes), static_cast<uint8_t *>(out->scales),
                                           out->second, out->mode, out->layout,
                                           reinterpret_cast<uint32_t *>(ws_at(ws, L.amax)), status_word(ws), s));
}

nvfp4_status nvfp4_quantize_fp8(const void *x_bf16, int64_t rows, int64_t K, int64_t ldx, void *a_fp8, float *s_t,
                                void *ws, size_t ws_bytes, nvfp4_stream_t stream)
{
    if (rows < 0 || K <= 0 || rows > MAX_DIM || K > MAX_DIM || ldx < K || ldx % 8 != 0)
        return NVFP4_ERR_INVALID_ARG;
    if (K % 16 != 0)
        return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (rows > 0 && (!x_bf16 || !aligned(x_bf16, 16) || !a_fp8 || !aligned(a_fp8, 16) || !s_t))
        return NVFP4_ERR_INVALID_ARG;
    nvfp4_status st = check_ws(ws, ws_bytes, ws_layout(NVFP4_OP_QUANTIZE_FP8, rows, 0, K).total);
    if (st != NVFP4_OK)
        return st;
    return from_cuda(launch_fp8_quantize(static_cast<const uint16_t *>(x_bf16), rows, K, ldx,
                                         static_cast<uint8_t *>(a_fp8), s_t, status_word(ws), (cudaStream_t)stream));
}

static nvfp4_status check_out(const void *y, int64_t ldy, int32_t y_dtype, int64_t N)
{
    if (y_dtype != NVFP4_OUT_BF16 && y_dtype != NVFP4_OUT_FP32)
        return NVFP4_ERR_INVALID_ARG;
    if (!y || !aligned(y, 16) || ldy < N)
        return NVFP4_ERR_INVALID_ARG;
    return NVFP4_OK;
}

nvfp4_status nvfp4_w4a8_gemm(const void *a_fp8, const float *s_t, const nvfp4_tensor *w, void *y, int64_t ldy,
                             int32_t y_dtype, int64_t M, void *ws, size_t ws_bytes, nvfp4_stream_t stream)
{
    nvfp4_status st = check_tensor(w, true);
    if (st != NVFP4_OK)
        return st;
    if (w->mode != NVFP4_SCALE_TENSOR_FP32)
        return NVFP4_ERR_UNSUPPORTED;
    if (M < 0 || M > MAX_DIM || (M > 0 && (!a_fp8 || !aligned(a_fp8, 16) || !s_t)))
        return NVFP4_ERR_INVALID_ARG;
    if ((st = check_out(y, ldy, y_dtype, w->rows)) != NVFP4_OK)
        return st;
    const WsLayout L = ws_layout(NVFP4_OP_W4A8_GEMM, M, w->rows, w->K);
    if ((st = check_ws(ws, ws_bytes, L.total)) != NVFP4_OK)
        return st;
    if (M == 0 || w->rows == 0)
        return NVFP4_OK;
    W4A8GemmArgs g{};
    g.a_fp8 = static_cast<const uint8_t *>(a_fp8);
    g.s_t = s_t;
    g.M = M;
    g.w_codes = static_cast<const uint8_t *>(w->codes);
    g.w_scales = static_cast<const uint8_t *>(w->scales);
    g.w_second = static_cast<const float *>(w->second);
    g.N = w->rows;
    g.K = w->K;
    g.out = y;
    g.ldy = ldy;
    g.out_dtype = y_dtype;
    g.status = status_word(ws);
    g.timeout_ns = DEFAULT_TIMEOUT_NS;
    return from_cuda(launch_w4a8(g, (cudaStream_t)stream));
}

nvfp4_status nvfp4_gemm(const void *x_bf16, int64_t ldx, const nvfp4_tensor *a_q, const nvfp4_tensor *w, void *y,
                        int64_t ldy, int32_t y_dtype, int64_t M, int32_t policy, int32_t sensitive, void *ws,
                        size_t ws_bytes, nvfp4_stream_t stream)
{
    const int32_t route = nvfp4_policy_route(policy, sensitive);
    if (route < 0)
        return NVFP4_ERR_INVALID_ARG;
    if ((x_bf16 == nullptr) == (a_q == nullptr))
        return NVFP4_ERR_INVALID_ARG;
    nvfp4_status st = check_tensor(w, true);
    if (st != NVFP4_OK)
        return st;
    const int64_t N = w->rows, K = w->K;
    if (M < 0 || M > MAX_DIM)
        return NVFP4_ERR_INVALID_ARG;
    if ((st = check_out(y, ldy, y_dtype, N)) != NVFP4_OK)
        return st;
    if (x_bf16) {
        if (ldx < K || ldx % 8 != 0 || (M > 0 && !aligned(x_bf16, 16)))
            return NVFP4_ERR_INVALID_ARG;
    } else {
        if ((st = check_tensor(a_q, true)) != NVFP4_OK)
            return st;
        if (a_q->rows != M || a_q->K != K || a_q->mode != w->mode)
            return NVFP4_ERR_INVALID_ARG;
        if (route == 8)
            return NVFP4_ERR_UNSUPPORTED; // W4A8 needs the BF16 activations
    }
    const WsLayout L = ws_layout(NVFP4_OP_GEMM, M, N, K);
    if ((st = check_ws(ws, ws_bytes, L.total)) != NVFP4_OK)
        return st;
    if (route == 8 && w->mode != NVFP4_SCALE_TENSOR_FP32)
        return NVFP4_ERR_UNSUPPORTED;
    if (M == 0 || N == 0)
        return NVFP4_OK;
    cudaStream_t s = (cudaStream_t)stream;

    if (route == 8) {
        uint8_t *a8 = ws_at(ws, L.a_fp8);
        float *st_ = reinterpret_cast<float *>(ws_at(ws, L.a_st));
        cudaError_t e = launch_fp8_quantize(static_cast<const uint16_t *>(x_bf16), M, K, ldx, a8, st_,
                                            status_word(ws), s);
        if (e != cudaSuccess)
            return NVFP4_ERR_CUDA;
        W4A8GemmArgs g{};
        g.a_fp8 = a8;
        g.s_t = st_;
        g.M = M;
        g.w_codes = static_cast<const uint8_t *>(w->codes);
        g.w_scales = static_cast<const uint8_t *>(w->scales);
        g.w_second = static_cast<const float *>(w->second);
        g.N = N;
        g.K = K;
        g.out = y;
        g.ldy = ldy;
        g.out_dtype = y_dtype;
        g.status = status_word(ws);
        g.timeout_ns = DEFAULT_TIMEOUT_NS;
        return from_cuda(launch_w4a8(g, s));
    }

    const uint8_t *ac, *as;
    const void *asec;
    if (x_bf16) {
        uint8_t *c = ws_at(ws, L.a_codes), *sc = ws_at(ws, L.a_scales);
        void *sec = ws_at(ws, L.a_second);
        cudaError_t e = launch_nvfp4_quantize(static_cast<const uint16_t *>(x_bf16), M, K, ldx, c, sc, sec, w->mode,
                                              NVFP4_LAYOUT_MMA_TILED, reinterpret_cast<uint32_t *>(ws_at(ws, L.amax)),
                                              status_word(ws), s, false);
        if (e != cudaSuccess)
            return NVFP4_ERR_CUDA;
        ac = c;
        as = sc;
        asec = sec;
    } else {
        ac = static_cast<const uint8_t *>(a_q->codes);
        as = static_cast<const uint8_t *>(a_q->scales);
        asec = a_q->second;
    }
    if (w->mode == NVFP4_SCALE_MACRO_FP16) {
        MacroGemmArgs g{};
        g.a_codes = ac;
        g.a_scales = as;
        g.a_macro = static_cast<const uint16_t *>(asec);
        g.M = M;
        g.w_codes = static_cast<const uint8_t *>(w->codes);
        g.w_scales = static_cast<const uint8_t *>(w->scales);
        g.w_macro = static_cast<const uint16_t *>(w->second);
        g.N = N;
        g.K = K;
        g.out = y;
        g.ldy = ldy;
        g.out_dtype = y_dtype;
        g.status = status_word(ws);
        g.timeout_ns = DEFAULT_TIMEOUT_NS;
        return from_cuda(launch_w4a4_macro(g, s));
    }
    return run_w4a4_dense(ac, as, static_cast<const float *>(asec), M, w, y, ldy, y_dtype, ws, L, x_bf16 != nullptr,
                          s);
}

nvfp4_status nvfp4_gemm_nvfp4_out(const void *x_bf16, int64_t ldx, const nvfp4_tensor *a_q, const nvfp4_tensor *w,
                                  nvfp4_tensor *y_q, float *y_amax, int64_t M, void *ws, size_t ws_bytes,
                                  nvfp4_stream_t stream)
{
    if ((x_bf16 == nullptr) == (a_q == nullptr))
        return NVFP4_ERR_INVALID_ARG;
    nvfp4_status st = check_tensor(w, true);
    if (st != NVFP4_OK)
        return st;
    if (w->mode != NVFP4_SCALE_TENSOR_FP32)
        return NVFP4_ERR_UNSUPPORTED;
    const int64_t N = w->rows, K = w->K;
    if (M < 0 || M > MAX_DIM || (y_amax && !aligned(y_amax, 4)))
        return NVFP4_ERR_INVALID_ARG;
    if ((st = check_tensor(y_q, true)) != NVFP4_OK)
        return st;
    if (y_q->mode != NVFP4_SCALE_TENSOR_FP32 || y_q->rows != M || y_q->K != N)
        return NVFP4_ERR_INVALID_ARG;
    if (x_bf16) {
        if (ldx < K || ldx % 8 != 0 || (M > 0 && !aligned(x_bf16, 16)))
            return NVFP4_ERR_INVALID_ARG;
    } else {
        if ((st = check_tensor(a_q, true)) != NVFP4_OK)
            return st;
        if (a_q->rows != M || a_q->K != K || a_q->mode != NVFP4_SCALE_TENSOR_FP32)
            return NVFP4_ERR_INVALID_ARG;
    }
    const WsLayout L = ws_layout(NVFP4_OP_GEMM, M, N, K);
    if ((st = check_ws(ws, ws_bytes, L.total)) != NVFP4_OK)
        return st;
    if (M == 0 || N == 0)
        return NVFP4_OK;
    cudaStream_t s = (cudaStream_t)stream;
    const uint8_t *ac, *as;
    const void *asec;
    if (x_bf16) {
        uint8_t *c = ws_at(ws, L.a_codes), *sc = ws_at(ws, L.a_scales);
        void *sec = ws_at(ws, L.a_second);
        cudaError_t e = launch_nvfp4_quantize(static_cast<const uint16_t *>(x_bf16), M, K, ldx, c, sc, sec,
                                              NVFP4_SCALE_TENSOR_FP32, NVFP4_LAYOUT_MMA_TILED,
                                              reinterpret_cast<uint32_t *>(ws_at(ws, L.amax)), status_word(ws), s,
                                              false);
        if (e != cudaSuccess)
            return NVFP4_ERR_CUDA;
        ac = c;
        as = sc;
        asec = sec;
    } else {
        ac = static_cast<const uint8_t *>(a_q->codes);
        as = static_cast<const uint8_t *>(a_q->scales);
        asec = a_q->second;
    }
    return run_w4a4_dense(ac, as, static_cast<const float *>(asec), M, w, nullptr, 0, NVFP4_OUT_FP32, ws, L,
                          x_bf16 != nullptr, s, y_q, y_amax);
}

// Checks shared by the grouped entry points (activations, stacked weights of
// E experts with n_rows rows each, offsets, index list) and the argument
// block they fill.
static nvfp4_status grouped_args(const nvfp4_tensor *a, const int32_t *row_idx, const int64_t *expert_offsets,
                                 int32_t E, const nvfp4_tensor *w, int64_t n_rows, int64_t total_rows, void *ws,
                                 size_t ws_bytes, GroupedGemmArgs &g)
{
    nvfp4_status st = check_tensor(a, true);
    if (st != NVFP4_OK)
        return st;
    if ((st = check_tensor(w, true)) != NVFP4_OK)
        return st;
    if (a->mode != NVFP4_SCALE_TENSOR_FP32 || w->mode != NVFP4_SCALE_TENSOR_FP32)
        return NVFP4_ERR_UNSUPPORTED;
    if (E <= 0 || E > 1024 || !expert_offsets || !aligned(expert_offsets, 8))
        return NVFP4_ERR_INVALID_ARG;
    if (n_rows <= 0 || n_rows % 128 != 0)
        return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (w->rows != (int64_t)E * n_rows || w->K != a->K)
        return NVFP4_ERR_INVALID_ARG;
    if (total_rows < 0 || total_rows > MAX_DIM)
        return NVFP4_ERR_INVALID_ARG;
    if (row_idx == nullptr && total_rows > a->rows)
        return NVFP4_ERR_INVALID_ARG;
    if (row_idx != nullptr && !aligned(row_idx, 4))
        return NVFP4_ERR_INVALID_ARG;
    if ((st = check_ws(ws, ws_bytes, ws_layout(NVFP4_OP_GROUPED_GEMM, total_rows, n_rows, a->K).total)) != NVFP4_OK)
        return st;
    g = GroupedGemmArgs{};
    g.a_codes = static_cast<const uint8_t *>(a->codes);
    g.a_scales = static_cast<const uint8_t *>(a->scales);
    g.a_second = static_cast<const float *>(a->second);
    g.a_rows = a->rows;
    g.row_idx = row_idx;
    g.offsets = expert_offsets;
    g.E = E;
    g.w_codes = static_cast<const uint8_t *>(w->codes);
    g.w_scales = static_cast<const uint8_t *>(w->scales);
    g.w_second = static_cast<const float *>(w->second);
    g.N = n_rows;
    g.K = a->K;
    g.total_rows = total_rows;
    g.status = status_word(ws);
    g.timeout_ns = DEFAULT_TIMEOUT_NS;
    g.epi = EPI_PLAIN;
    return NVFP4_OK;
}

nvfp4_status nvfp4_grouped_gemm(const nvfp4_tensor *a, const int32_t *row_idx, const int64_t *expert_offsets,
                                int32_t E, const nvfp4_tensor *w, int64_t N, void *y, int64_t ldy, int32_t y_dtype,
                                int64_t total_rows, int32_t policy, int32_t sensitive, void *ws,
                                size_t ws_bytes, nvfp4_stream_t stream)
{
    const int32_t route = nvfp4_policy_route(policy, sensitive);
    if (route < 0)
        return NVFP4_ERR_INVALID_ARG;
    if (route == 8)
        return NVFP4_ERR_UNSUPPORTED; // W4A8 needs FP8 activations: nvfp4_grouped_gemm_x / _w4a8_gemm
    GroupedGemmArgs g;
    nvfp4_status st = grouped_args(a, row_idx, expert_offsets, E, w, N, total_rows, ws, ws_bytes, g);
    if (st != NVFP4_OK)
        return st;
    if ((st = check_out(y, ldy, y_dtype, N)) != NVFP4_OK)
        return st;
    if (total_rows == 0)
        return NVFP4_OK;
    g.out = y;
    g.ldy = ldy;
    g.out_dtype = y_dtype;
    return from_cuda(launch_w4a4_grouped(g, (cudaStream_t)stream));
}

// Checks of the grouped W4A8 operands; fills the argument block.
static nvfp4_status grouped_w4a8_args(const void *a_fp8, const float *s_t, int64_t T, const int32_t *row_idx,
                                      const int64_t *expert_offsets, int32_t E, const nvfp4_tensor *w, int64_t N,
                                      void *y, int64_t ldy, int32_t y_dtype, int64_t total_rows, W4A8GemmArgs &g)
{
    nvfp4_status st = check_tensor(w, true);
    if (st != NVFP4_OK)
        return st;
    if (w->mode != NVFP4_SCALE_TENSOR_FP32)
        return NVFP4_ERR_UNSUPPORTED;
    if (E <= 0 || E > 1024 || !expert_offsets || !aligned(expert_offsets, 8))
        return NVFP4_ERR_INVALID_ARG;
    if (N <= 0 || N % 128 != 0)
        return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (w->rows != (int64_t)E * N)
        return NVFP4_ERR_INVALID_ARG;
    if (T < 0 || T > MAX_DIM || total_rows < 0 || total_rows > MAX_DIM)
        return NVFP4_ERR_INVALID_ARG;
    if (T > 0 && (!a_fp8 || !aligned(a_fp8, 16) || !s_t || !aligned(s_t, 4)))
        return NVFP4_ERR_INVALID_ARG;
    if ((row_idx == nullptr && total_rows > T) || (row_idx != nullptr && !aligned(row_idx, 4)))
        return NVFP4_ERR_INVALID_ARG;
    if ((st = check_out(y, ldy, y_dtype, N)) != NVFP4_OK)
        return st;
    g = W4A8GemmArgs{};
    g.a_fp8 = static_cast<const uint8_t *>(a_fp8);
    g.s_t = s_t;
    g.M = T;
    g.w_codes = static_cast<const uint8_t *>(w->codes);
    g.w_scales = static_cast<const uint8_t *>(w->scales);
    g.w_second = static_cast<const float *>(w->second);
    g.N = N;
    g.K = w->K;
    g.out = y;
    g.ldy = ldy;
    g.out_dtype = y_dtype;
    g.timeout_ns = DEFAULT_TIMEOUT_NS;
    g.E = E;
    g.offsets = expert_offsets;
    g.row_idx = row_idx;
    g.total_rows = total_rows;
    return NVFP4_OK;
}

nvfp4_status nvfp4_grouped_w4a8_gemm(const void *a_fp8, const float *s_t, int64_t T, const int32_t *row_idx,
                                     const int64_t *expert_offsets, int32_t E, const nvfp4_tensor *w, int64_t N,
                                     void *y, int64_t ldy, int32_t y_dtype, int64_t total_rows, void *ws,
                                     size_t ws_bytes, nvfp4_stream_t stream)
{
    W4A8GemmArgs g;
    nvfp4_status st =
        grouped_w4a8_args(a_fp8, s_t, T, row_idx, expert_offsets, E, w, N, y, ldy, y_dtype, total_rows, g);
    if (st != NVFP4_OK)
        return st;
    if ((st = check_ws(ws, ws_bytes, ws_layout(NVFP4_OP_GROUPED_GEMM, total_rows, N, w->K).total)) != NVFP4_OK)
        return st;
    if (total_rows == 0 || T == 0)
        return NVFP4_OK;
    g.status = status_word(ws);
    return from_cuda(launch_w4a8(g, (cudaStream_t)stream));
}

nvfp4_status nvfp4_grouped_gemm_x(const void *x_bf16, int64_t ldx, int64_t T, const int32_t *row_idx,
                                  const int64_t *expert_offsets, int32_t E, const nvfp4_tensor *w, int64_t N,
                                  void *y, int64_t ldy, int32_t y_dtype, int64_t total_rows, int32_t policy,
                                  int32_t sensitive, void *ws, size_t ws_bytes, nvfp4_stream_t stream)
{
    const int32_t route = nvfp4_policy_route(policy, sensitive);
    if (route < 0 || !w)
        return NVFP4_ERR_INVALID_ARG;
    const int64_t K = w->K;
    if (T < 0 || T > MAX_DIM || ldx < K || ldx % 8 != 0 || (T > 0 && (!x_bf16 || !aligned(x_bf16, 16))))
        return NVFP4_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(NVFP4_OP_GROUPED_GEMM_X, T, N, K);
    cudaStream_t s = (cudaStream_t)stream;
    if (route == 8) {
        uint8_t *a8 = ws_at(ws, L.a_fp8);
        float *st_ = reinterpret_cast<float *>(ws_at(ws, L.a_st));
        W4A8GemmArgs g;
        nvfp4_status st =
            grouped_w4a8_args(a8, st_, T, row_idx, expert_offsets, E, w, N, y, ldy, y_dtype, total_rows, g);
        if (st != NVFP4_OK)
            return st;
        if ((st = check_ws(ws, ws_bytes, L.total)) != NVFP4_OK)
            return st;
        if (total_rows == 0 || T == 0)
            return NVFP4_OK;
        g.status = status_word(ws);
        if (launch_fp8_quantize(static_cast<const uint16_t *>(x_bf16), T, K, ldx, a8, st_, status_word(ws), s) !=
            cudaSuccess)
            return NVFP4_ERR_CUDA;
        return from_cuda(launch_w4a8(g, s));
    }
    // W4A4: the NVFP4 activations live in the workspace
    nvfp4_tensor a{};
    a.codes = ws_at(ws, L.a_codes);
    a.scales = ws_at(ws, L.a_scales);
    a.second = ws_at(ws, L.a_second);
    a.rows = T;
    a.K = K;
    a.mode = NVFP4_SCALE_TENSOR_FP32;
    a.layout = NVFP4_LAYOUT_MMA_TILED;
    if (!ws || !aligned(ws, 256))
        return NVFP4_ERR_WORKSPACE;
    GroupedGemmArgs g;
    nvfp4_status st = grouped_args(&a, row_idx, expert_offsets, E, w, N, total_rows, ws, ws_bytes, g);
    if (st != NVFP4_OK)
        return st;
    if ((st = check_out(y, ldy, y_dtype, N)) != NVFP4_OK)
        return st;
    if ((st = check_ws(ws, ws_bytes, L.total)) != NVFP4_OK)
        return st;
    if (total_rows == 0 || T == 0)
        return NVFP4_OK;
    g.out = y;
    g.ldy = ldy;
    g.out_dtype = y_dtype;
    cudaError_t e = launch_nvfp4_quantize(static_cast<const uint16_t *>(x_bf16), T, K, ldx,
                                          static_cast<uint8_t *>(a.codes), static_cast<uint8_t *>(a.scales), a.second,
                                          NVFP4_SCALE_TENSOR_FP32, NVFP4_LAYOUT_MMA_TILED,
                                          reinterpret_cast<uint32_t *>(ws_at(ws, L.amax)), status_word(ws), s, false);
    if (e != cudaSuccess)
        return NVFP4_ERR_CUDA;
    return from_cuda(launch_w4a4_grouped(g, s));
}

static nvfp4_status check_kv(const nvfp4_kv_cache *kv)
{
    if (!kv || (kv->format != NVFP4_KV_NVFP4 && kv->format != NVFP4_KV_FP8))
        return NVFP4_ERR_INVALID_ARG;
    if (!kv->pages || !kv->k_scale || !kv->v_scale)
        return NVFP4_ERR_INVALID_ARG;
    if (kv->head_dim != 128 || kv->page_tokens != 64)
        return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (kv->num_pages <= 0 || kv->num_kv_heads <= 0 || !aligned(kv->pages, 16) || !aligned(kv->k_scale, 4) ||
        !aligned(kv->v_scale, 4))
        return NVFP4_ERR_INVALID_ARG;
    return NVFP4_OK;
}

nvfp4_status nvfp4_kv_append(const nvfp4_kv_cache *kv, const void *k_bf16, const void *v_bf16,
                             const int32_t *positions, const int32_t *block_table, int32_t max_pages, int32_t B,
                             nvfp4_stream_t stream)
{
    nvfp4_status st = check_kv(kv);
    if (st != NVFP4_OK)
        return st;
    if (B < 0 || max_pages <= 0)
        return NVFP4_ERR_INVALID_ARG;
    if (B == 0)
        return NVFP4_OK;
    if (!k_bf16 || !v_bf16 || !positions || !block_table || !aligned(k_bf16, 2) || !aligned(v_bf16, 2) ||
        !aligned(positions, 4) || !aligned(block_table, 4))
        return NVFP4_ERR_INVALID_ARG;
    KvAppendArgs a{};
    a.fmt = kv->format;
    a.k_new = static_cast<const uint16_t *>(k_bf16);
    a.v_new = static_cast<const uint16_t *>(v_bf16);
    a.positions = positions;
    a.block_table = block_table;
    a.B = B;
    a.H_kv = kv->num_kv_heads;
    a.max_pages = max_pages;
    a.num_pages = kv->num_pages;
    a.pages = static_cast<uint8_t *>(kv->pages);
    a.k_scale = kv->k_scale;
    a.v_scale = kv->v_scale;
    return from_cuda(launch_kv_append(a, (cudaStream_t)stream));
}

nvfp4_status nvfp4_kv_decode_attention(const nvfp4_kv_cache *kv, const void *q_bf16, int32_t num_heads,
                                       const int32_t *ctx_lens, const int32_t *block_table, int32_t max_pages,
                                       int32_t B, int32_t max_ctx, float sm_scale, void *out, int32_t out_dtype,
                                       void *ws, size_t ws_bytes, nvfp4_stream_t stream)
{
    nvfp4_status st = check_kv(kv);
    if (st != NVFP4_OK)
        return st;
    const int H_kv = kv->num_kv_heads;
    if (B < 0 || max_pages <= 0 || max_ctx < 0 || num_heads <= 0 || num_heads % H_kv != 0)
        return NVFP4_ERR_INVALID_ARG;
    if (num_heads / H_kv > 16 || B > 65535 || H_kv > 65535)
        return NVFP4_ERR_UNSUPPORTED_SHAPE; // up to 16 query heads per KV head; grid y = KV heads, z = sequences
    if (out_dtype != NVFP4_OUT_BF16 && out_dtype != NVFP4_OUT_FP32)
        return NVFP4_ERR_INVALID_ARG;
    if (!(sm_scale == sm_scale) || sm_scale < 0.0f || sm_scale > 1e30f)
        return NVFP4_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(NVFP4_OP_KV_DECODE, B, num_heads, max_ctx, H_kv);
    if ((st = check_ws(ws, ws_bytes, L.total)) != NVFP4_OK)
        return st;
    if (B == 0)
        return NVFP4_OK;
    if (!q_bf16 || !ctx_lens || !block_table || !out || !aligned(q_bf16, 2) || !aligned(ctx_lens, 4) ||
        !aligned(block_table, 4) || !aligned(out, 4))
        return NVFP4_ERR_INVALID_ARG;
    KvAttnArgs a{};
    a.fmt = kv->format;
    a.q = static_cast<const uint16_t *>(q_bf16);
    a.ctx_lens = ctx_lens;
    a.block_table = block_table;
    a.B = B;
    a.H = num_heads;
    a.H_kv = H_kv;
    a.max_pages = max_pages;
    a.num_pages = kv->num_pages;
    a.max_ctx = max_ctx;
    a.pages = static_cast<const uint8_t *>(kv->pages);
    a.k_scale = kv->k_scale;
    a.v_scale = kv->v_scale;
    a.sm_scale = sm_scale;
    kv_attn_splits(B, H_kv, max_ctx, device_sm_count(), kv_ctas_per_sm(a.fmt, num_heads / H_kv), a.n_splits,
                   a.keys_per_split);
    a.out = out;
    a.out_dtype = out_dtype;
    a.partial = L.kv_partial ? reinterpret_cast<float *>(ws_at(ws, L.kv_partial)) : nullptr;
    a.status = status_word(ws);
    a.timeout_ns = DEFAULT_TIMEOUT_NS;
    return from_cuda(launch_kv_decode(a, (cudaStream_t)stream));
}

nvfp4_status nvfp4_moe_up_swiglu(const nvfp4_tensor *a, const int32_t *row_idx, const int64_t *expert_offsets,
                                 int32_t E, const nvfp4_tensor *w_gate_up, int64_t I, void *h, int64_t ldh,
                                 int32_t h_dtype, nvfp4_tensor *h_q, float *h_amax, int64_t total_rows, void *ws,
                                 size_t ws_bytes, nvfp4_stream_t stream)
{
    if ((h == nullptr) == (h_q == nullptr) || I <= 0 || I % 128 != 0)
        return I > 0 && I % 128 != 0 ? NVFP4_ERR_UNSUPPORTED_SHAPE : NVFP4_ERR_INVALID_ARG;
    GroupedGemmArgs g;
    nvfp4_status st = grouped_args(a, row_idx, expert_offsets, E, w_gate_up, 2 * I, total_rows, ws, ws_bytes, g);
    if (st != NVFP4_OK)
        return st;
    if (h) {
        if ((st = check_out(h, ldh, h_dtype, I)) != NVFP4_OK)
            return st;
        if ((ldh * (h_dtype == NVFP4_OUT_BF16 ? 2 : 4)) % 16 != 0)
            return NVFP4_ERR_INVALID_ARG;
    } else {
        if ((st = check_tensor(h_q, true)) != NVFP4_OK)
            return st;
        if (h_q->mode != NVFP4_SCALE_TENSOR_FP32 || h_q->rows != total_rows || h_q->K != I)
            return NVFP4_ERR_INVALID_ARG;
        if (h_amax && !aligned(h_amax, 4))
            return NVFP4_ERR_INVALID_ARG;
    }
    if (total_rows == 0)
        return NVFP4_OK;
    cudaStream_t s = (cudaStream_t)stream;
    g.epi = EPI_SWIGLU;
    if (h) {
        g.out = h;
        g.ldy = ldh;
        g.out_dtype = h_dtype;
    } else {
        g.yq_codes = static_cast<uint8_t *>(h_q->codes);
        g.yq_scales = static_cast<uint8_t *>(h_q->scales);
        g.yq_scale = static_cast<const float *>(h_q->second);
        g.yq_amax = reinterpret_cast<uint32_t *>(h_amax);
        g.out_dtype = NVFP4_OUT_FP32;
        if (total_rows % 128 != 0) {
            // the last 128-row scale tile holds padding rows: zero it, the
            // kernel then writes the rows that exist
            const size_t atom_row = (size_t)(I / 64) * 512;
            if (cudaMemsetAsync(g.yq_scales + (size_t)(total_rows / 128) * atom_row, 0, atom_row, s) != cudaSuccess)
                return NVFP4_ERR_CUDA;
        }
    }
    return from_cuda(launch_w4a4_grouped(g, s));
}

nvfp4_status nvfp4_moe_down_combine(const nvfp4_tensor *h, const int64_t *expert_offsets, int32_t E,
                                    const nvfp4_tensor *w_down, int64_t N, const int32_t *token_idx,
                                    const float *gate_w, float *y, int64_t ldy, int64_t T, int64_t total_rows,
                                    void *ws, size_t ws_bytes, nvfp4_stream_t stream)
{
    GroupedGemmArgs g;
    nvfp4_status st = grouped_args(h, nullptr, expert_offsets, E, w_down, N, total_rows, ws, ws_bytes, g);
    if (st != NVFP4_OK)
        return st;
    if (T < 0 || T > MAX_DIM || !token_idx || !gate_w || !aligned(token_idx, 4) || !aligned(gate_w, 4))
        return NVFP4_ERR_INVALID_ARG;
    if ((st = check_out(y, ldy, NVFP4_OUT_FP32, N)) != NVFP4_OK)
        return st;
    if (ldy % 4 != 0)
        return NVFP4_ERR_INVALID_ARG;
    if (total_rows == 0 || T == 0)
        return NVFP4_OK;
    g.epi = EPI_COMBINE;
    g.out = y;
    g.ldy = ldy;
    g.out_dtype = NVFP4_OUT_FP32;
    g.comb_idx = token_idx;
    g.comb_w = gate_w;
    g.comb_rows = T;
    return from_cuda(launch_w4a4_grouped(g, (cudaStream_t)stream));
}

nvfp4_status nvfp4_diag_streamk_skip_flag(const nvfp4_tensor *a_q, const nvfp4_tensor *w, void *y, int64_t ldy,
                                          int32_t y_dtype, int32_t skip_cta, uint64_t timeout_ns, void *ws,
                                          size_t ws_bytes, nvfp4_stream_t stream)
{
    nvfp4_status st = check_tensor(w, true);
    if (st != NVFP4_OK)
        return st;
    if ((st = check_tensor(a_q, true)) != NVFP4_OK)
        return st;
    if (w->mode != NVFP4_SCALE_TENSOR_FP32 || a_q->mode != NVFP4_SCALE_TENSOR_FP32 || a_q->K != w->K)
        return NVFP4_ERR_INVALID_ARG;
    const int64_t M = a_q->rows, N = w->rows, K = w->K;
    if ((st = check_out(y, ldy, y_dtype, N)) != NVFP4_OK)
        return st;
    if (skip_cta < 0 || timeout_ns == 0 || timeout_ns > 10000000000ull)
        return NVFP4_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(NVFP4_OP_GEMM, M, N, K);
    if ((st = check_ws(ws, ws_bytes, L.total)) != NVFP4_OK)
        return st;
    if (L.sk_slots == 0)
        return NVFP4_ERR_UNSUPPORTED_SHAPE; // the shape does not run stream-K
    return run_w4a4_dense(static_cast<const uint8_t *>(a_q->codes), static_cast<const uint8_t *>(a_q->scales),
                          static_cast<const float *>(a_q->second), M, w, y, ldy, y_dtype, ws, L, false,
                          (cudaStream_t)stream, nullptr, nullptr, skip_cta, timeout_ns);
}

nvfp4_status nvfp4_diag_fp4_mma_rate(int32_t iters, uint64_t *cycles, nvfp4_stream_t stream)
{
    if (iters < 1 || iters > (1 << 24) || !cycles || !aligned(cycles, 8))
        return NVFP4_ERR_INVALID_ARG;
    return from_cuda(launch_fp4_mma_rate(iters, cycles, (cudaStream_t)stream));
}

int32_t nvfp4_diag_bounds_checked(void) { return kCheckBounds ? 1 : 0; }

nvfp4_status nvfp4_diag_bounds_selftest(uint8_t *buf, uint64_t buf_bytes, uint64_t span_bytes, nvfp4_stream_t stream)
{
    if (!buf || span_bytes == 0 || span_bytes > (uint64_t(1) << 30) || buf_bytes < span_bytes + 64)
        return NVFP4_ERR_INVALID_ARG;
    return from_cuda(launch_bounds_selftest(buf, span_bytes, (cudaStream_t)stream));
}

nvfp4_status nvfp4_diag_bounds_record(uint64_t *failures, char *where, int32_t where_len, uint64_t *value,
                                      uint64_t *limit, int32_t clear)
{
    if (!kCheckBounds)
        return NVFP4_ERR_UNSUPPORTED;
    if (!failures || where_len < 0 || (where_len > 0 && !where))
        return NVFP4_ERR_INVALID_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess)
        return NVFP4_ERR_CUDA;
    uint64_t total = 0;
    bool have = false;
    for (int u = 0; u < g_bounds_n; ++u) {
        unsigned long long rec[4];
        if (cudaMemcpyFromSymbol(rec, g_bounds_units[u].symbol, sizeof(rec)) != cudaSuccess)
            return NVFP4_ERR_CUDA;
        total += rec[0];
        if (rec[0] != 0 && !have) {
            have = true;
            if (value)
                *value = rec[2];
            if (limit)
                *limit = rec[3];
            if (where && where_len > 0) {
                const char *name = g_bounds_units[u].unit;
                const char *slash = std::strrchr(name, '/');
                name = slash ? slash + 1 : name;
                static const char *const shared_files[] = {"", " via ptx.cuh", " via epilogue.cuh"};
                const unsigned file = (unsigned)(rec[1] >> 16);
                std::snprintf(where, (size_t)where_len, "%s%s:%u", name, file < 3 ? shared_files[file] : " via ?",
                              (unsigned)(rec[1] & 0xFFFFu));
            }
        }
        if (clear) {
            const unsigned long long zero[4] = {0, 0, 0, 0};
            if (cudaMemcpyToSymbol(g_bounds_units[u].symbol, zero, sizeof(zero)) != cudaSuccess)
                return NVFP4_ERR_CUDA;
        }
    }
    *failures = total;
    if (!have && where && where_len > 0)
        where[0] = '\0';
    return NVFP4_OK;
}

nvfp4_status nvfp4_diag_tma_stream(const uint8_t *w, int64_t rows, int64_t row_bytes, int32_t grid, uint32_t *status,
                                   nvfp4_stream_t stream)
{
    if (!w || !aligned(w, 16) || rows <= 0 || rows % 256 != 0 || rows > ((int64_t)1 << 31) || row_bytes < 128 ||
        row_bytes % 128 != 0 || row_bytes > ((int64_t)1 << 20) || grid < 1 || grid > 4096 || !status ||
        !aligned(status, 4))
        return NVFP4_ERR_INVALID_ARG;
    return from_cuda(launch_tma_stream(w, rows, row_bytes, grid, status, (cudaStream_t)stream));
}

nvfp4_status nvfp4_probe_convert(const float *in, int64_t n, uint8_t *out_e2m1, uint8_t *out_e4m3,
                                 nvfp4_stream_t stream)
{
    if (n < 0 || (n > 0 && (!in || !out_e2m1 || !out_e4m3)))
        return NVFP4_ERR_INVALID_ARG;
    return from_cuda(launch_probe_convert(in, n, out_e2m1, out_e4m3, (cudaStream_t)stream));
}

} // extern "C"
