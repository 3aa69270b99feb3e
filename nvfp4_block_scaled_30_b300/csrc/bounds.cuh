// Bounds-checked build.  Compiled with -DNVFP4_CHECK_BOUNDS (the library
// libnvfp4_checked.so), the copy, tensor-memory and MMA wrappers and the
// kernels' plain global accesses test every address before it is used:
//   - a shared-memory destination or operand must lie inside the CTA's
//     dynamic shared memory (and bulk/TMA destinations be aligned);
//   - a tensor-map x coordinate must be a multiple of 16 bytes;
//   - a TMEM column range must lie within the 512 columns of an SM;
//   - a global load or store must lie inside the byte range that the call's
//     arguments grant the tensor (rows x leading dimension, as the header
//     documents each layout), computed once per kernel from the arguments,
//     not from the per-element index arithmetic under test.
// A failed test counts, records (site, value, limit) if it is the first of
// its translation unit, and skips the access; nvfp4_diag_bounds_record reads
// the records.  In the normal build every test folds to `true`.
#pragma once
#include <cstdint>

#include "internal.h"

// site of a test: which file it sits in (0 the kernel's own .cu file,
// 1 ptx.cuh, 2 epilogue.cuh) and its line
#define NV4_SITE(file) ((uint32_t)(((file) << 16) | (__LINE__ & 0xFFFF)))

namespace nv4 {

#ifdef NVFP4_CHECK_BOUNDS
constexpr bool kCheckBounds = true;

// Host: registers one translation unit's record (a __device__ symbol) so
// that the reader can find it.
void register_bounds_record(const void *symbol, const char *unit);

namespace {
// failures, first failure's site, value, limit
__device__ unsigned long long bounds_rec[4];

struct BoundsRecordRegistrar {
    BoundsRecordRegistrar() { register_bounds_record(&bounds_rec, __BASE_FILE__); }
};
BoundsRecordRegistrar bounds_registrar;

__device__ __noinline__ void bounds_fail(uint32_t site, uint64_t value, uint64_t limit)
{
    if (atomicAdd(&bounds_rec[0], 1ull) == 0ull) {
        bounds_rec[1] = site;
        bounds_rec[2] = value;
        bounds_rec[3] = limit;
    }
}
} // namespace

// value < limit, unsigned (a negative value wrapped to 64 bits fails)
__device__ __forceinline__ bool in_bounds(uint32_t site, uint64_t value, uint64_t limit)
{
    if (value < limit)
        return true;
    bounds_fail(site, value, limit);
    return false;
}

// value % align == 0 (align a power of two)
__device__ __forceinline__ bool aligned_to(uint32_t site, uint64_t value, uint64_t align)
{
    if ((value & (align - 1)) == 0)
        return true;
    bounds_fail(site, value, align);
    return false;
}
#else
constexpr bool kCheckBounds = false;
__device__ __forceinline__ void bounds_fail(uint32_t, uint64_t, uint64_t) {}
__device__ __forceinline__ bool in_bounds(uint32_t, uint64_t, uint64_t) { return true; }
__device__ __forceinline__ bool aligned_to(uint32_t, uint64_t, uint64_t) { return true; }
#endif

// Whether [p, p + n) lies inside s (n >= 1).  The recorded value is the
// offset of p from s.lo (wrapped to 64 bits when p < s.lo), the limit
// s.bytes.
__device__ __forceinline__ bool in_span(uint32_t site, const Span &s, const void *p, uint64_t n)
{
    if (!kCheckBounds)
        return true;
    const uint64_t off = reinterpret_cast<uint64_t>(p) - s.lo;
    if (off < s.bytes && n <= s.bytes - off)
        return true;
    bounds_fail(site, off, s.bytes);
    return false;
}

// Whether the shared-memory range [saddr, saddr + n) lies inside this CTA's
// dynamic shared memory (every extern __shared__ array starts at its base).
__device__ __forceinline__ bool in_dyn_smem(uint32_t site, uint32_t saddr, uint32_t n)
{
    if (!kCheckBounds)
        return true;
    extern __shared__ uint8_t nv4_dynamic_smem_base[];
    const uint32_t base = static_cast<uint32_t>(__cvta_generic_to_shared(nv4_dynamic_smem_base));
    uint32_t size;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(size));
    const uint32_t off = saddr - base;
    if (off < size && n <= size - off)
        return true;
    bounds_fail(site, off, size);
    return false;
}

} // namespace nv4
