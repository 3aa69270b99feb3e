// What the copy engine delivers to a kernel that only streams: the bytes of
// a [rows][row_bytes] matrix brought into shared memory with the same tiled
// TMA boxes as the W4A4 GEMM's weight operand (128 bytes x 256 rows, 128-byte
// swizzle) through a 6-deep ring of 32 KB stages, and nothing else.  The
// decode GEMM streams its weights this way, so this rate, at the decode
// kernel's grid and at one CTA per SM, is the ceiling that kernel's HBM
// roofline fraction is measured against in practice.
#include "internal.h"
#include "ptx.cuh"

namespace nv4 {

namespace {

constexpr int ST_ROWS = 256;
constexpr int ST_STAGES = 6;
constexpr int ST_BYTES = ST_ROWS * 128; // one box
constexpr int ST_SMEM = ST_STAGES * ST_BYTES + 1024;

// CTA b takes the contiguous range [b U / G, (b + 1) U / G) of the U =
// (rows / 256) x (row_bytes / 128) boxes, row-tile major, so a CTA's boxes
// run along its row tiles as the GEMM's K stages do.
__global__ void __launch_bounds__(32, 1)
    tma_stream_kernel(const __grid_constant__ CUtensorMap map, int64_t tiles, int kboxes, uint32_t *status,
                      uint64_t timeout_ns)
{
    extern __shared__ uint8_t raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t full[ST_STAGES];
    const int lane = threadIdx.x;
    if (lane == 0) {
        for (int s = 0; s < ST_STAGES; ++s)
            mbar_init(&full[s], 1);
        fence_mbar_init();
        prefetch_tmap(&map);
    }
    __syncwarp();
    const int64_t U = tiles * kboxes;
    const int64_t u0 = (int64_t)blockIdx.x * U / gridDim.x, u1 = (int64_t)(blockIdx.x + 1) * U / gridDim.x;
    bool ok = true;
    int i = 0;
    for (int64_t u = u0; ok && u < u1; ++u, ++i) {
        const int s = i % ST_STAGES;
        if (i >= ST_STAGES)
            ok = mbar_wait(&full[s], (uint32_t)((i / ST_STAGES) - 1) & 1u, timeout_ns, nullptr);
        ok = __all_sync(0xFFFFFFFFu, ok);
        if (!ok)
            break;
        // copies of one thread are served in order: rotate the issuing lane
        if (lane == (i & 7)) {
            mbar_arrive_expect_tx(&full[s], ST_BYTES);
            tma_load_2d(sm + (size_t)s * ST_BYTES, &map, (int)(u % kboxes) * 128, (int)(u / kboxes) * ST_ROWS,
                        &full[s], ST_BYTES);
        }
        __syncwarp();
    }
    // every copy issued lands before the CTA exits
    for (int j = i - ST_STAGES; j < i; ++j)
        if (j >= 0 && !mbar_wait(&full[j % ST_STAGES], (uint32_t)(j / ST_STAGES) & 1u, timeout_ns, nullptr))
            ok = false;
    if (!ok && lane == 0)
        atomicOr(status, ST_TIMEOUT);
}

} // namespace

cudaError_t launch_tma_stream(const uint8_t *w, int64_t rows, int64_t row_bytes, int grid, uint32_t *status,
                              cudaStream_t stream)
{
    CUtensorMap map;
    if (make_tmap_2d_u8(&map, w, (uint64_t)row_bytes, (uint64_t)rows, (uint64_t)row_bytes, 128, ST_ROWS, true) !=
        CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(tma_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, ST_SMEM);
    if (e != cudaSuccess)
        return e;
    tma_stream_kernel<<<grid, 32, ST_SMEM, stream>>>(map, rows / ST_ROWS, (int)(row_bytes / 128), status,
                                                     2000000000ull);
    return cudaGetLastError();
}

} // namespace nv4
