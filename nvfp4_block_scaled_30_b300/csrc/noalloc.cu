// nvfp4_gemm_w4a4_noalloc: the W4A4 GEMM for callers that cannot allocate.
//
// Some callers have no way to obtain device memory at the point of the call:
// a host framework that owns every byte of device memory through its own
// pool and forbids direct cudaMalloc, a plugin running inside another
// runtime without allocation rights, or a latency-critical serving loop that
// must never reach the allocator.  nvfp4_gemm needs a caller-allocated
// workspace for its stream-K partial sums; this entry point instead keeps
// that scratch in a fixed array inside the library (see the header for the
// contract).  It allocates nothing: no cudaMalloc, no cudaFree, no
// allocating library routine.
#include <mutex>

#include "internal.h"

namespace nv4 {

namespace {

// Scratch of the no-allocation entry point: every GPU that loads the library
// holds these bytes until the process exits.  Layout: [0, 256) status word,
// then the stream-K partial slots (one FP32 tile per CTA), then the flags.
constexpr size_t NOALLOC_SCRATCH_BYTES = size_t(4) << 20;
static __device__ __align__(256) uint8_t g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

constexpr uint64_t NOALLOC_TIMEOUT_NS = 2000000000ull;

std::mutex g_mu;
void *g_scratch_addr[64] = {nullptr};

// Device address of the scratch array on the current device.  The symbol's
// host-side name is only a stand-in; the address comes from
// cudaGetSymbolAddress, looked up once per device with that device current.
cudaError_t scratch_address(void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= 64)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess)
            return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

} // namespace

} // namespace nv4

using namespace nv4;

extern "C" nvfp4_status nvfp4_gemm_w4a4_noalloc(const nvfp4_tensor *a_q, const nvfp4_tensor *w, void *y,
                                                 int64_t ldy, int32_t y_dtype, nvfp4_stream_t stream)
{
    nvfp4_status st = check_tensor(a_q, true);
    if (st == NVFP4_OK)
        st = check_tensor(w, true);
    if (st != NVFP4_OK)
        return st;
    if (a_q->mode != NVFP4_SCALE_TENSOR_FP32 || w->mode != NVFP4_SCALE_TENSOR_FP32)
        return NVFP4_ERR_UNSUPPORTED;
    if (a_q->K != w->K)
        return NVFP4_ERR_INVALID_ARG;
    if (y_dtype != NVFP4_OUT_BF16 && y_dtype != NVFP4_OUT_FP32)
        return NVFP4_ERR_INVALID_ARG;
    const int64_t M = a_q->rows, N = w->rows, K = w->K;
    if (M == 0 || N == 0)
        return NVFP4_OK;
    if (!y || (reinterpret_cast<uintptr_t>(y) % 16) != 0 || ldy < N)
        return NVFP4_ERR_INVALID_ARG;

    // the same launch shape nvfp4_gemm picks: stream-K when whole tiles fill
    // the SMs poorly
    DenseGemmArgs g{};
    g.a_codes = static_cast<const uint8_t *>(a_q->codes);
    g.a_scales = static_cast<const uint8_t *>(a_q->scales);
    g.a_second = static_cast<const float *>(a_q->second);
    g.a_rows = M;
    g.b_codes = static_cast<const uint8_t *>(w->codes);
    g.b_scales = static_cast<const uint8_t *>(w->scales);
    g.b_second = static_cast<const float *>(w->second);
    g.b_rows = N;
    g.K = K;
    const StreamKPlan pl = w4a4_streamk_plan(M, N, K, device_sm_count());

    // scratch needed by this call; larger requests are rejected
    const size_t need = WS_HEADER + (pl.used ? pl.slot_bytes + pl.flag_bytes : 0);
    if (need > NOALLOC_SCRATCH_BYTES)
        return NVFP4_ERR_WORKSPACE;

    void *scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    // the array keeps the previous call's contents: zero the status word and
    // the stream-K flags this call relies on (the partial slots are always
    // written before they are read)
    uint8_t *base = static_cast<uint8_t *>(scratch);
    if (cudaMemsetAsync(base, 0, WS_HEADER, s) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    if (pl.used && cudaMemsetAsync(base + WS_HEADER + pl.slot_bytes, 0, pl.flag_bytes, s) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    g.status = reinterpret_cast<uint32_t *>(base);
    g.timeout_ns = NOALLOC_TIMEOUT_NS;
    g.out = y;
    g.out_dtype = y_dtype;
    g.ld_i = ldy;
    g.ld_j = 1;
    g.streamk = pl.used;
    if (pl.used) {
        g.slots = reinterpret_cast<float *>(base + WS_HEADER);
        g.flags = reinterpret_cast<uint32_t *>(base + WS_HEADER + pl.slot_bytes);
    }
    const cudaError_t e = launch_w4a4_dense(g, s);
    if (e == cudaSuccess)
        return NVFP4_OK;
    return e == cudaErrorNotSupported ? NVFP4_ERR_UNSUPPORTED : NVFP4_ERR_CUDA;
}

extern "C" nvfp4_status nvfp4_gemm_w4a4_noalloc_status(nvfp4_stream_t stream, int32_t *device_status)
{
    if (!device_status)
        return NVFP4_ERR_INVALID_ARG;
    void *scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    uint32_t word = 0;
    // the copy into pageable host memory returns once the stream's earlier
    // work (the calls being asked about) has finished
    if (cudaMemcpyAsync(&word, scratch, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    if (cudaMemsetAsync(scratch, 0, sizeof(word), s) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    *device_status = (word & ST_NONFINITE) ? NVFP4_ERR_NONFINITE_INPUT : (word & ST_TIMEOUT) ? NVFP4_ERR_TIMEOUT
                                                                                           : NVFP4_OK;
    return NVFP4_OK;
}
