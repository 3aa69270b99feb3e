// Dense FP4 tensor-core peak of this GPU, measured: one CTA per SM issues
// tcgen05.mma kind::mxf4nvf4 (M = 128, N = 256, K = 64, UE4M3 scales per 16
// elements) back to back on operands resident in shared memory and scales
// resident in TMEM, so no global memory traffic limits it.  The contraction
// is the block-scaled FP4 x FP4 product that "NVIDIA Ships TensorRT-LLM 0.16:
// Native FP4 Quantization for Blackwell B200", section "The Mathematical
// Breakthrough of Microscopic FP4 Scaling", item 3 "Hardware-Fused
// Dequantization" describes; the GEMMs' roofline divides by this rate.
#include "internal.h"
#include "ptx.cuh"

namespace nv4 {

namespace {

constexpr int PEAK_THREADS = 128;
constexpr int PEAK_N = 256;
constexpr int PEAK_A_BYTES = 128 * 128;      // 128 rows x 256 FP4
constexpr int PEAK_B_BYTES = PEAK_N * 128;   // 256 rows x 256 FP4
constexpr int PEAK_SF_BYTES = 12 * 512;      // 4 A atoms + 8 B atoms
// more shared memory than two CTAs can share, so the grid runs one CTA per SM
constexpr int PEAK_SMEM = 160 * 1024;

__global__ void __launch_bounds__(PEAK_THREADS, 1) fp4_mma_rate_kernel(int iters, uint64_t *cycles, const Span sp_cycles)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = sm;
    uint8_t *sB = sA + PEAK_A_BYTES;
    uint8_t *sSF = sB + PEAK_B_BYTES;
    __shared__ uint64_t bar;
    __shared__ uint32_t tmem_slot;
    const int warp = threadIdx.x >> 5;
    // codes: a fixed hash of the byte index (all 16 E2M1 codes occur);
    // scales 0x30 = 0.5 keep the accumulators finite
    for (int i = threadIdx.x; i < PEAK_A_BYTES + PEAK_B_BYTES; i += PEAK_THREADS) {
        uint32_t h = (uint32_t)i * 2654435761u;
        h ^= h >> 15;
        sA[i] = (uint8_t)h;
    }
    for (int i = threadIdx.x; i < PEAK_SF_BYTES; i += PEAK_THREADS)
        sSF[i] = 0x30;
    fence_proxy_async_smem();
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    if (threadIdx.x == 0) {
        const uint32_t sf_col = tmem + PEAK_N;
        for (int kk = 0; kk < 4; ++kk) {
            tc_cp_32x128b_warpx4(sf_col + 4 * kk, sdesc_sf(smem_u32(sSF + kk * 512)));
            for (int h = 0; h < 2; ++h)
                tc_cp_32x128b_warpx4(sf_col + 16 + 8 * kk + 4 * h, sdesc_sf(smem_u32(sSF + 2048 + h * 2048 + kk * 512)));
        }
        tc_commit(&bar);
        bool ok = mbar_wait(&bar, 0, 2000000000ull, nullptr);
        tc_fence_after();
        const uint32_t idesc = idesc_mxf4nvf4(PEAK_N);
        const uint64_t adesc = sdesc_sw128(smem_u32(sA));
        const uint64_t bdesc = sdesc_sw128(smem_u32(sB));
        const uint64_t t0 = clock64();
        for (int it = 0; ok && it < iters; ++it) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_mxf4nvf4(tmem, adesc + (uint64_t)(kk * 2), bdesc + (uint64_t)(kk * 2), idesc, sf_col + 4 * kk,
                             sf_col + 16 + 8 * kk, (it | kk) != 0 ? 1u : 0u);
        }
        tc_commit(&bar);
        ok = ok && mbar_wait(&bar, 1, 4000000000ull, nullptr);
        const uint64_t t1 = clock64();
        if (in_span(NV4_SITE(0), sp_cycles, cycles + blockIdx.x, 8))
            cycles[blockIdx.x] = ok ? t1 - t0 : ~0ull;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

} // namespace

cudaError_t launch_fp4_mma_rate(int iters, uint64_t *cycles, cudaStream_t stream)
{
    cudaError_t e = cudaFuncSetAttribute(fp4_mma_rate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, PEAK_SMEM);
    if (e != cudaSuccess)
        return e;
    const int sms = device_sm_count();
    fp4_mma_rate_kernel<<<sms, PEAK_THREADS, PEAK_SMEM, stream>>>(iters, cycles, span_of(cycles, 8u * (uint64_t)sms));
    return cudaGetLastError();
}

} // namespace nv4
