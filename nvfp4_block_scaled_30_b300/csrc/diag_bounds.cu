// Self-test of the bounds-checked build: a kernel stores one byte to every
// offset of [0, span_bytes + 64) of a caller buffer while the span it tests
// against grants only span_bytes, so in the checked build the last 64 stores
// fail their test, are counted and skipped, and in the normal build all of
// them happen.  The caller's buffer holds at least span_bytes + 64 bytes, so
// every store lies inside memory the caller owns whichever build runs.
#include "internal.h"
#include "ptx.cuh"

namespace nv4 {

namespace {

__global__ void bounds_selftest_kernel(uint8_t *buf, uint64_t n, const Span granted)
{
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (uint64_t)gridDim.x * blockDim.x)
        if (in_span(NV4_SITE(0), granted, buf + i, 1))
            buf[i] = 1;
}

} // namespace

cudaError_t launch_bounds_selftest(uint8_t *buf, uint64_t span_bytes, cudaStream_t stream)
{
    bounds_selftest_kernel<<<1, 256, 0, stream>>>(buf, span_bytes + 64, span_of(buf, span_bytes));
    return cudaGetLastError();
}

} // namespace nv4
