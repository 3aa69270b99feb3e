// W4A4 GEMM with FP16 macro-scales, the second scaling level of "NVIDIA Ships
// TensorRT-LLM 0.16: Native FP4 Quantization for Blackwell B200", section
// "The Mathematical Breakthrough of Microscopic FP4 Scaling", item 2
// "Two-Level Block Scaling": 16 consecutive micro-vectors (256 elements of
// a row) share one FP16 macro-scale.  With macro-scales the product is
//
//   Y[m][n] = sum_g S_A[m][g] * S_W[n][g] * P_g[m][n],
//   P_g[m][n] = sum_{k in group g} E2M1(a)E4M3(ea) * E2M1(w)E4M3(ew),
//
// so the macro-scales cannot be folded into one epilogue factor.  One
// pipeline stage covers exactly one group (256 elements of K): the tensor
// cores compute P_g into one of two TMEM buffers (tcgen05.mma kind::mxf4nvf4,
// 4 x K=64) while eight epilogue warps rescale the previous P_{g-1} by
// S_A * S_W and accumulate it in registers (FP32).
//
// Roles (one CTA per SM, persistent, 352 threads): warp 0 copy producer,
// warp 1 TMEM allocation + MMA issue, warp 2 scale copies into TMEM, warps
// 3..10 epilogue (warp w covers TMEM lane quarter w % 4 and columns
// 64 * ((w - 3) / 4) .. +63 of the 128-wide tile).
#include <algorithm>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "epilogue.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace nv4 {

namespace {

constexpr int BM = 128;
constexpr int BN = 128;               // B tiles start on a 128-row scale atom
constexpr int STAGE_K_BYTES = 128; // 256 FP4 = one macro group
constexpr int STAGES = 5;
constexpr int EPI_WARPS = 8;
constexpr int EPI_FIRST_WARP = 3;
constexpr int THREADS = 32 * EPI_FIRST_WARP + 32 * EPI_WARPS;
constexpr int A_BYTES = BM * STAGE_K_BYTES;
constexpr int B_BYTES = BN * STAGE_K_BYTES;
constexpr int SFA_BYTES = 2048;
constexpr int SFB_BYTES = 2048;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
constexpr int SF_COLS = 32;            // 16 (A) + 16 (B) TMEM columns per stage
constexpr int P_BUFS = 2;
constexpr int SF_BASE = P_BUFS * BN;
constexpr int TMEM_COLS = 512;
// W macro-scales of the current tile for WT_G groups at a time, FP32
// [group][BN + 4] (the 4-float pad spreads a column's writes over banks and
// keeps rows 16-byte aligned for the epilogue's float4 reads)
constexpr int WT_G = 32;
constexpr int WT_PITCH = BN + 4;
constexpr int TAB_BYTES = WT_G * WT_PITCH * 4;
constexpr int TAB_LOADS = WT_G * BN / (32 * 8);   // table entries per epilogue thread (8 warps)
static_assert(WT_G * BN % (32 * 8) == 0, "table fill mapping");
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + TAB_BYTES + 256 + 1024;
static_assert(SF_BASE + STAGES * SF_COLS <= TMEM_COLS, "TMEM");
static_assert(STAGE_BYTES % 1024 == 0, "alignment");
static_assert(SMEM_BYTES <= 232448, "shared memory");

struct Params {
    CUtensorMap tmap_a;
    CUtensorMap tmap_b;
    const uint8_t *sfa;
    const uint8_t *sfb;
    const uint16_t *a_macro; // [M][K/256]
    const uint16_t *w_macro; // [N][K/256]
    void *out;
    int64_t ldy, M, N;
    int32_t m_tiles, n_tiles, k64, groups, out_dtype, vec_ok;
    uint32_t *status;
    uint64_t timeout_ns;
    // the bytes the call's arguments grant each tensor (tested before each
    // plain access in the bounds-checked build)
    Span sp_sfa, sp_sfb, sp_a_macro, sp_w_macro, sp_out;
};

__device__ __forceinline__ void tile_of(const Params &p, int item, int &tm, int &tn)
{
    constexpr int G = 8;
    const int band = G * p.n_tiles;
    const int bid = item / band;
    const int first = bid * G;
    const int gs = min(p.m_tiles - first, G);
    const int r = item - bid * band;
    tm = first + r % gs;
    tn = r / gs;
}

__device__ __forceinline__ void timeout(const Params &p, volatile int *abort_flag)
{
    *abort_flag = 1;
    atomicOr(p.status, ST_TIMEOUT);
}

// Named barrier 1 across the epilogue warps.
__device__ __forceinline__ void epi_bar_sync()
{
    asm volatile("bar.sync 1, %0;" ::"n"(32 * EPI_WARPS) : "memory");
}

// Named barrier 1 across the epilogue warps returning the AND of `pred`, so
// every epilogue warp takes the same exit decision.
__device__ __forceinline__ bool epi_bar_all(bool pred)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "bar.red.and.pred po, 1, %2, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "n"(32 * EPI_WARPS)
        : "memory");
    return r != 0;
}

__global__ void __launch_bounds__(THREADS, 1) macro_kernel(const __grid_constant__ Params p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *wtab = reinterpret_cast<float *>(smem + STAGES * STAGE_BYTES);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + STAGES * STAGE_BYTES + TAB_BYTES);
    uint64_t *empty = full + STAGES;
    uint64_t *pfull = empty + STAGES;
    uint64_t *pempty = pfull + P_BUFS;
    uint64_t *sf_full = pempty + P_BUFS;
    uint64_t *sf_ready = sf_full + STAGES;
    uint64_t *drain = sf_ready + STAGES;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            mbar_init(&sf_full[s], 1);
            mbar_init(&sf_ready[s], 1);
        }
        for (int b = 0; b < P_BUFS; ++b) {
            mbar_init(&pfull[b], 1);
            mbar_init(&pempty[b], EPI_WARPS);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int total = p.m_tiles * p.n_tiles;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // The four copies of a stage (A codes, B codes, A scales, B scales)
        // go out from four different lanes: copies issued by one thread are
        // served one after another, copies from different threads overlap.
        // Lanes 8r .. 8r+3 serve stages r, r + 4, ..., so each lane has at
        // most one copy of four consecutive stages outstanding.
        int st = 0, issued = 0;
        uint32_t ph = 0;
        bool ok = true;
        for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
            int tm, tn;
            tile_of(p, item, tm, tn);
            for (int g = 0; g < p.groups; ++g) {
                const bool got = mbar_wait(&empty[st], ph ^ 1u, p.timeout_ns, abort_flag);
                if (!__all_sync(0xFFFFFFFFu, got)) {
                    if (lane == 0)
                        timeout(p, abort_flag);
                    ok = false;
                    break;
                }
                uint8_t *sA = smem + st * STAGE_BYTES;
                uint8_t *sB = sA + A_BYTES;
                if (lane == 0)
                    mbar_arrive_expect_tx(&full[st], A_BYTES + B_BYTES);
                else if (lane == 1)
                    mbar_arrive_expect_tx(&sf_full[st], SFA_BYTES + SFB_BYTES);
                __syncwarp();
                const int op = lane - 8 * (issued & 3);
                if (op == 0) {
                    tma_load_2d(sA, &p.tmap_a, g * STAGE_K_BYTES, tm * BM, &full[st], A_BYTES);
                } else if (op == 1) {
                    tma_load_2d(sB, &p.tmap_b, g * STAGE_K_BYTES, tn * BN, &full[st], B_BYTES);
                } else if (op == 2) {
                    const uint8_t *sfa_src = p.sfa + ((size_t)tm * p.k64 + 4 * g) * 512;
                    if (in_span(NV4_SITE(0), p.sp_sfa, sfa_src, SFA_BYTES))
                        bulk_load(sB + B_BYTES, sfa_src, SFA_BYTES, &sf_full[st]);
                } else if (op == 3) {
                    const uint8_t *sfb_src = p.sfb + ((size_t)tn * p.k64 + 4 * g) * 512;
                    if (in_span(NV4_SITE(0), p.sp_sfb, sfb_src, SFB_BYTES))
                        bulk_load(sB + B_BYTES + SFA_BYTES, sfb_src, SFB_BYTES, &sf_full[st]);
                }
                ++issued;
                if (++st == STAGES) {
                    st = 0;
                    ph ^= 1u;
                }
            }
        }
        // every copy issued lands before the CTA exits
        if (lane == 0) {
            const int n = min(issued, STAGES);
            for (int q = 0; q < n; ++q) {
                if (--st < 0) {
                    st = STAGES - 1;
                    ph ^= 1u;
                }
                mbar_wait(&full[st], ph, p.timeout_ns, nullptr);
                mbar_wait(&sf_full[st], ph, p.timeout_ns, nullptr);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_mxf4nvf4(BN);
            int st = 0, pb = 0;
            uint32_t ph = 0, pph = 0;
            bool ok = true;
            for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
                int tm, tn;
                tile_of(p, item, tm, tn);
                for (int g = 0; g < p.groups; ++g) {
                    if (!mbar_wait(&full[st], ph, p.timeout_ns, abort_flag) ||
                        !mbar_wait(&sf_ready[st], ph, p.timeout_ns, abort_flag) ||
                        !mbar_wait(&pempty[pb], pph ^ 1u, p.timeout_ns, abort_flag)) {
                        timeout(p, abort_flag);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint8_t *sA = smem + st * STAGE_BYTES;
                    const uint8_t *sB = sA + A_BYTES;
                    const uint32_t sf = tmem + SF_BASE + st * SF_COLS;
                    const uint64_t ad = sdesc_sw128(smem_u32(sA)), bd = sdesc_sw128(smem_u32(sB));
                    const uint32_t d = tmem + pb * BN;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_mxf4nvf4(d, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), idesc, sf + kk * 4,
                                     sf + 16 + kk * 4, kk > 0 ? 1u : 0u);
                    tc_commit(&empty[st]);
                    tc_commit(&pfull[pb]);
                    if (++st == STAGES) {
                        st = 0;
                        ph ^= 1u;
                    }
                    if (++pb == P_BUFS) {
                        pb = 0;
                        pph ^= 1u;
                    }
                }
            }
            tc_commit(drain);
            mbar_wait(drain, 0, p.timeout_ns, nullptr);
        }
        __syncwarp();
    } else if (warp == 2) {
        // ------------------------------------------------------------ scale warp
        // The stage's scale atoms go to its TMEM scale columns as soon as they
        // land (separate barrier from the codes), committed to sf_ready; the
        // MMA thread only issues MMAs.  The stage's previous MMAs have
        // completed (the producer refills a stage after its empty commit).
        int st = 0, issued = 0;
        uint32_t ph = 0;
        bool ok = true;
        for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
            for (int g = 0; g < p.groups; ++g) {
                const bool got = mbar_wait(&sf_full[st], ph, p.timeout_ns, abort_flag);
                if (!__all_sync(0xFFFFFFFFu, got)) {
                    if (lane == 0)
                        timeout(p, abort_flag);
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    tc_fence_after();
                    const uint8_t *sSFA = smem + st * STAGE_BYTES + A_BYTES + B_BYTES;
                    const uint8_t *sSFB = sSFA + SFA_BYTES;
                    const uint32_t sf = tmem + SF_BASE + st * SF_COLS;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        tc_cp_32x128b_warpx4(sf + kk * 4, sdesc_sf(smem_u32(sSFA + kk * 512)));
                        tc_cp_32x128b_warpx4(sf + 16 + kk * 4, sdesc_sf(smem_u32(sSFB + kk * 512)));
                    }
                    tc_commit(&sf_ready[st]);
                }
                __syncwarp();
                ++issued;
                if (++st == STAGES) {
                    st = 0;
                    ph ^= 1u;
                }
            }
        }
        // the copies this warp issued complete before TMEM is freed
        if (lane == 0) {
            const int n = min(issued, STAGES);
            for (int q = 0; q < n; ++q) {
                if (--st < 0) {
                    st = STAGES - 1;
                    ph ^= 1u;
                }
                mbar_wait(&sf_ready[st], ph, p.timeout_ns, nullptr);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;
        const int half = (warp - EPI_FIRST_WARP) >> 2;
        const int row = q * 32 + lane;
        const int et = threadIdx.x - 32 * EPI_FIRST_WARP; // 0 .. 32 * EPI_WARPS - 1
        const OutDesc out_desc{p.out, p.ldy, 1, p.out_dtype, p.vec_ok, p.sp_out};
        int pb = 0;
        uint32_t pph = 0;
        bool ok = true;
        for (int item = blockIdx.x; item < total; item += gridDim.x) {
            int tm, tn;
            tile_of(p, item, tm, tn);
            const int64_t i = (int64_t)tm * BM + row;
            const int64_t j0 = (int64_t)tn * BN + half * 64;
            float acc[64];
#pragma unroll
            for (int c = 0; c < 64; ++c)
                acc[c] = 0.0f;
            // this row's A macro-scale, one group ahead
            auto a_scale = [&](int g) -> float {
                return i < p.M && in_span(NV4_SITE(0), p.sp_a_macro, p.a_macro + i * p.groups + g, 2)
                           ? __half2float(__ushort_as_half(__ldg(p.a_macro + i * p.groups + g)))
                           : 0.0f;
            };
            float sa_next = a_scale(0);
            for (int g0 = 0; g0 < p.groups; g0 += WT_G) {
                // every epilogue warp takes the same exit decision and is done
                // with the previous table before it is overwritten
                ok = epi_bar_all(ok);
                if (!ok)
                    break;
                const int ng = min(WT_G, p.groups - g0);
                // W macro-scales of the tile's BN columns for groups g0 ..
                // g0 + ng - 1 (consecutive threads read consecutive groups of
                // one column: the row-major [N][K/256] layout), every load in
                // flight before the first store
                float wv[TAB_LOADS];
#pragma unroll
                for (int u = 0; u < TAB_LOADS; ++u) {
                    const int e = et + u * 32 * EPI_WARPS;
                    const int r = e / ng, gg = e - r * ng;
                    wv[u] = 0.0f;
                    if (e < ng * BN) {
                        const int64_t j = (int64_t)tn * BN + r;
                        const uint16_t *ws = p.w_macro + j * p.groups + g0 + gg;
                        if (j < p.N && in_span(NV4_SITE(0), p.sp_w_macro, ws, 2))
                            wv[u] = __half2float(__ushort_as_half(__ldg(ws)));
                    }
                }
#pragma unroll
                for (int u = 0; u < TAB_LOADS; ++u) {
                    const int e = et + u * 32 * EPI_WARPS;
                    const int r = e / ng, gg = e - r * ng;
                    if (e < ng * BN)
                        wtab[gg * WT_PITCH + r] = wv[u];
                }
                epi_bar_sync();
                for (int g = g0; g < g0 + ng; ++g) {
                    const bool got = mbar_wait(&pfull[pb], pph, p.timeout_ns, abort_flag);
                    if (!__all_sync(0xFFFFFFFFu, got)) {
                        if (lane == 0)
                            timeout(p, abort_flag);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const float sa = sa_next;
                    const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + pb * BN + half * 64;
                    uint32_t va[32], vb[32];
                    tc_ld_32x32b_x32(ta, va);
                    tc_ld_32x32b_x32(ta + 32, vb);
                    tc_wait_ld();
                    // both halves are in registers: the buffer can take the next group
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&pempty[pb]);
                    if (++pb == P_BUFS) {
                        pb = 0;
                        pph ^= 1u;
                    }
                    if (g + 1 < p.groups)
                        sa_next = a_scale(g + 1);
                    const float4 *sw4 = reinterpret_cast<const float4 *>(wtab + (g - g0) * WT_PITCH + half * 64);
#pragma unroll
                    for (int c4 = 0; c4 < 8; ++c4) {
                        const float4 w = sw4[c4];
                        acc[4 * c4 + 0] = fmaf(sa * w.x, __uint_as_float(va[4 * c4 + 0]), acc[4 * c4 + 0]);
                        acc[4 * c4 + 1] = fmaf(sa * w.y, __uint_as_float(va[4 * c4 + 1]), acc[4 * c4 + 1]);
                        acc[4 * c4 + 2] = fmaf(sa * w.z, __uint_as_float(va[4 * c4 + 2]), acc[4 * c4 + 2]);
                        acc[4 * c4 + 3] = fmaf(sa * w.w, __uint_as_float(va[4 * c4 + 3]), acc[4 * c4 + 3]);
                    }
#pragma unroll
                    for (int c4 = 0; c4 < 8; ++c4) {
                        const float4 w = sw4[8 + c4];
                        acc[32 + 4 * c4 + 0] = fmaf(sa * w.x, __uint_as_float(vb[4 * c4 + 0]), acc[32 + 4 * c4 + 0]);
                        acc[32 + 4 * c4 + 1] = fmaf(sa * w.y, __uint_as_float(vb[4 * c4 + 1]), acc[32 + 4 * c4 + 1]);
                        acc[32 + 4 * c4 + 2] = fmaf(sa * w.z, __uint_as_float(vb[4 * c4 + 2]), acc[32 + 4 * c4 + 2]);
                        acc[32 + 4 * c4 + 3] = fmaf(sa * w.w, __uint_as_float(vb[4 * c4 + 3]), acc[32 + 4 * c4 + 3]);
                    }
                }
            }
            ok = epi_bar_all(ok);
            if (!ok)
                break;
            // the warp's 32 rows together (32-byte stores of whole row runs)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t v[32];
#pragma unroll
                for (int k = 0; k < 32; ++k)
                    v[k] = __float_as_uint(acc[32 * h + k]);
                store_chunk32_warp(out_desc, v, i - lane, 0, p.M, j0 + 32 * h, 1.0f, p.N, lane);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

} // namespace

cudaError_t launch_w4a4_macro(const MacroGemmArgs &g, cudaStream_t stream)
{
    if (g.K % 256 != 0)
        return cudaErrorInvalidValue;
    Params p{};
    CUresult r = make_tmap_2d_u8(&p.tmap_a, g.a_codes, (uint64_t)(g.K / 2), (uint64_t)g.M, (uint64_t)(g.K / 2),
                                 STAGE_K_BYTES, BM, true);
    if (r != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    r = make_tmap_2d_u8(&p.tmap_b, g.w_codes, (uint64_t)(g.K / 2), (uint64_t)g.N, (uint64_t)(g.K / 2), STAGE_K_BYTES,
                        BN, true);
    if (r != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    p.sfa = g.a_scales;
    p.sfb = g.w_scales;
    p.a_macro = g.a_macro;
    p.w_macro = g.w_macro;
    p.out = g.out;
    p.ldy = g.ldy;
    p.M = g.M;
    p.N = g.N;
    p.m_tiles = (int)ceil_div(g.M, BM);
    p.n_tiles = (int)ceil_div(g.N, BN);
    p.k64 = (int)(g.K / 64);
    p.groups = (int)(g.K / 256);
    p.out_dtype = g.out_dtype;
    const int esz = g.out_dtype == NVFP4_OUT_BF16 ? 2 : 4;
    p.vec_ok = out_vec_level(g.out, g.ldy, 1, esz);
    p.status = g.status;
    p.timeout_ns = g.timeout_ns;
    p.sp_sfa = span_of(g.a_scales, tiled_scale_bytes(g.M, g.K));
    p.sp_sfb = span_of(g.w_scales, tiled_scale_bytes(g.N, g.K));
    p.sp_a_macro = span_of(g.a_macro, 2u * (uint64_t)g.M * (uint64_t)p.groups);
    p.sp_w_macro = span_of(g.w_macro, 2u * (uint64_t)g.N * (uint64_t)p.groups);
    p.sp_out = span_of(g.out, matrix_bytes(g.M, g.N, g.ldy, esz));
    cudaError_t e = cudaFuncSetAttribute(macro_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess)
        return e;
    const int total = p.m_tiles * p.n_tiles;
    const int grid = std::max(1, std::min(total, device_sm_count()));
    macro_kernel<<<grid, THREADS, SMEM_BYTES, stream>>>(p);
    return cudaGetLastError();
}

} // namespace nv4
