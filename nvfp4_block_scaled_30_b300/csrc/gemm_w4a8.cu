// W4A8 GEMM: FP8 (E4M3, per-token FP32 scale) activations x NVFP4 weights, the
// route "llama.cpp Put Precision Policy Inside the Model. That Matters More
// Than W4A4", section "One model can need more than one precision", gives the
// layers its metadata marks as sensitive.
//
//   Y[m][n] = s_t[m] * s_w * sum_k E4M3(a[m][k]) * E2M1(w[n][k]) * E4M3(ew[n][k/16])
//
// Exactness: an E4M3 value and an E2M1 x E4M3 product (at most 6 significant
// bits, magnitudes 2^-10 .. 2688) are both exact in FP16, so converter warps
// expand both operands to FP16 and tcgen05.mma kind::f16 (FP16 x FP16 ->
// FP32) contracts them; no requantisation of the weights.  The activations
// go to TMEM (the MMA's A operand may come from there) and only the weights
// through shared memory: the kernel is bound by shared-memory traffic, and
// the FP16 activations would be a third of it.
// The block-scaled FP8 MMA kinds use power-of-two scales per 32 elements and
// cannot carry the weights' E4M3 scales per 16 elements exactly.
//
// Pipeline (persistent, one CTA per SM, 576 threads, tile 128 x 256):
//   warp 0      TMA: raw FP8 A tile [128 x 64 B], raw FP4 W tile [256 x 32 B]
//               and the W scale atoms per 64-element K step (raw ring); each
//               copy of a step from its own lane (one thread's copies are
//               served one after another, different threads' in parallel)
//   warp 1      TMEM alloc (one 256-column accumulator, then the FP16 A
//               stages); lane 0 issues 4 x tcgen05.mma kind::f16 (M 128,
//               N 256, K 16, A from TMEM) per step
//   warps 2..9  converters: raw ring -> FP16.  Warp w expands its TMEM lane
//               quarter's 32 A rows, K half (w - 2) / 4, into the step's TMEM
//               A stage (tcgen05.st, 16 columns per lane); threads 2i, 2i+1
//               expand the halves of W rows i and 128 + i into 128-byte
//               swizzled shared-memory rows (no bank conflicts)
//   warps 10..17 epilogue: TMEM -> registers 32 columns at a time,
//               * s_t[m] * s_w, BF16/FP32 store
// The grouped (mixture-of-experts) variant runs the same pipeline over the
// experts' routed rows: work items are (expert, 128-row block of its rows,
// N tile); gathered token rows are copied into the raw ring with 16-byte
// cp.async by all producer lanes (contiguous rows by TMA), each row takes
// its token's scale and the expert's weight scale.
#include <algorithm>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "epilogue.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace nv4 {

namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int NG = BN / 128;    // 128-row scale groups per W tile
constexpr int KSTEP = 64;       // K elements per pipeline step
constexpr int RAW_STAGES = 4;
constexpr int CONV_STAGES = 4;
constexpr int ACC_BUFS = 1;
constexpr int CONV_WARPS = 8;
constexpr int EPI_WARPS = 8;
constexpr int EPI_FIRST_WARP = 2 + CONV_WARPS;
constexpr int THREADS = 64 + 32 * (CONV_WARPS + EPI_WARPS);
constexpr int RAW_A = BM * KSTEP;           // 8192 B of FP8
constexpr int RAW_W = BN * KSTEP / 2;       // 8192 B of FP4 codes
constexpr int RAW_S = NG * 512;             // scale atoms
constexpr int RAW_BYTES = RAW_A + RAW_W + RAW_S;
constexpr int CONV_B = BN * 128;            // FP16 W rows of 128 bytes
constexpr int CONV_BYTES = CONV_B;
constexpr int TMEM_COLS = 512;
constexpr int A_COLS = KSTEP / 2;           // TMEM columns of one FP16 A stage (2 per column)
constexpr int A_BASE = ACC_BUFS * BN;       // first A stage column
constexpr int MAX_EXPERTS = 1024;
static_assert(CONV_WARPS * 32 == 2 * BM && CONV_WARPS * 32 == BN, "converter thread mapping");
constexpr int SMEM_BYTES = CONV_STAGES * CONV_BYTES + RAW_STAGES * RAW_BYTES + 256 + 1024;
static_assert(RAW_BYTES % 1024 == 0 && CONV_BYTES % 1024 == 0, "alignment");
static_assert(SMEM_BYTES + 4 * (MAX_EXPERTS + 2) <= 232448, "shared memory");
static_assert(A_BASE + CONV_STAGES * A_COLS <= TMEM_COLS, "TMEM");

struct Params {
    CUtensorMap tmap_a; // FP8 [M][K]
    CUtensorMap tmap_w; // FP4 codes [N][K/2]
    const uint8_t *w_scales;
    const float *s_t;
    const float *w_second;
    void *out;
    int64_t ldy, M, N;
    int32_t m_tiles, n_tiles, ksteps, k64_total, out_dtype, vec_ok, w_groups;
    uint32_t *status;
    uint64_t timeout_ns;
    // grouped mode: N is per expert, W holds E * N rows
    const uint8_t *a_fp8;     // gathered rows are copied from here
    int64_t K;
    const int64_t *offsets;
    const int32_t *row_idx;   // null: routed row j reads activation row j
    int32_t E;
    int64_t total_rows;
    // the bytes the call's arguments grant each tensor (tested before each
    // plain access in the bounds-checked build)
    Span sp_w_scales, sp_s_t, sp_w_second, sp_out, sp_a_fp8, sp_offsets, sp_row_idx;
};

struct Item {
    int tn, expert;
    int64_t row0, row_end;    // first output row of the tile, end of its rows
};

// Expert e's routed rows [lo, hi), offsets clamped to [0, total_rows] and
// made non-decreasing.
__device__ __forceinline__ void expert_rows(const Params &p, int e, int64_t &lo, int64_t &hi)
{
    if (!in_span(NV4_SITE(0), p.sp_offsets, p.offsets + e, 16)) {
        lo = hi = 0;
        return;
    }
    lo = min(max(p.offsets[e], (int64_t)0), p.total_rows);
    hi = min(max(p.offsets[e + 1], lo), p.total_rows);
}

__device__ __forceinline__ void decode_dense(const Params &p, int item, int &tm, int &tn)
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

// prefix[e] = 128-row blocks of experts 0..e-1 (grouped); items are the
// expert's blocks, N tiles outermost within an expert.
template <bool GROUPED>
__device__ __forceinline__ void decode(const Params &p, const int *prefix, int item, Item &it)
{
    if (!GROUPED) {
        int tm;
        decode_dense(p, item, tm, it.tn);
        it.expert = 0;
        it.row0 = (int64_t)tm * BM;
        it.row_end = p.M;
        return;
    }
    const int blk = item / p.n_tiles;
    int lo = 0, hi = p.E;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (prefix[mid] <= blk)
            lo = mid;
        else
            hi = mid;
    }
    const int e = lo;
    const int mt_e = prefix[e + 1] - prefix[e];
    const int local = item - prefix[e] * p.n_tiles;
    it.expert = e;
    it.tn = local / mt_e;
    int64_t r_lo, r_hi;
    expert_rows(p, e, r_lo, r_hi);
    it.row0 = r_lo + (int64_t)(local - it.tn * mt_e) * BM;
    it.row_end = r_hi;
}

__device__ __forceinline__ uint32_t f16x2_from_e4m3x2(uint32_t two_bytes)
{
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"((uint16_t)two_bytes));
    return r;
}

__device__ __forceinline__ uint32_t f16x2_from_e2m1x2(uint32_t byte)
{
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(r) : "r"(byte));
    return r;
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b)
{
    __half2 r = __hmul2(*reinterpret_cast<__half2 *>(&a), *reinterpret_cast<__half2 *>(&b));
    return *reinterpret_cast<uint32_t *>(&r);
}

__device__ __forceinline__ void timeout(const Params &p, volatile int *abort_flag)
{
    *abort_flag = 1;
    atomicOr(p.status, ST_TIMEOUT);
}

template <bool GROUPED>
__global__ void __launch_bounds__(THREADS, 1) w4a8_kernel(const __grid_constant__ Params p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *conv = smem;
    uint8_t *raw = smem + CONV_STAGES * CONV_BYTES;
    uint64_t *raw_full = reinterpret_cast<uint64_t *>(raw + RAW_STAGES * RAW_BYTES);
    uint64_t *raw_empty = raw_full + RAW_STAGES;
    uint64_t *conv_full = raw_empty + RAW_STAGES;
    uint64_t *conv_empty = conv_full + CONV_STAGES;
    uint64_t *acc_full = conv_empty + CONV_STAGES;
    uint64_t *acc_empty = acc_full + ACC_BUFS;
    uint64_t *drain = acc_empty + ACC_BUFS;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    __shared__ int prefix[GROUPED ? MAX_EXPERTS + 1 : 1];
    __shared__ int total_s;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr unsigned FULLMASK = 0xFFFFFFFFu;
    const bool indexed = GROUPED && p.row_idx != nullptr;
    if (threadIdx.x == 0) {
        for (int s = 0; s < RAW_STAGES; ++s) {
            // gathered rows: one more arrival per producer lane (its cp.async)
            mbar_init(&raw_full[s], indexed ? 33 : 1);
            mbar_init(&raw_empty[s], CONV_WARPS);
        }
        for (int s = 0; s < CONV_STAGES; ++s) {
            mbar_init(&conv_full[s], CONV_WARPS);
            mbar_init(&conv_empty[s], 1);
        }
        for (int b = 0; b < ACC_BUFS; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], EPI_WARPS);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    if (GROUPED) {
        if (warp == 2) {
            // 128-row blocks per expert, prefix-summed by one warp: lane l
            // owns a contiguous run of experts, a shuffle scan joins the runs
            const int per = (p.E + 31) / 32;
            const int e0 = min(lane * per, p.E), e1 = min(e0 + per, p.E);
            int run = 0;
            for (int e = e0; e < e1; ++e) {
                int64_t lo, hi;
                expert_rows(p, e, lo, hi);
                run += (int)((hi - lo + BM - 1) / BM);
            }
            int incl = run;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(FULLMASK, incl, o);
                if (lane >= o)
                    incl += v;
            }
            int acc = incl - run;
            if (lane == 0)
                prefix[0] = 0;
            for (int e = e0; e < e1; ++e) {
                int64_t lo, hi;
                expert_rows(p, e, lo, hi);
                acc += (int)((hi - lo + BM - 1) / BM);
                prefix[e + 1] = acc;
            }
            if (lane == 31)
                total_s = incl * p.n_tiles;
        }
    } else if (threadIdx.x == 0) {
        total_s = p.m_tiles * p.n_tiles;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int total = total_s;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        int st = 0, issued = 0;
        uint32_t ph = 0;
        bool ok = true;
        for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
            Item it;
            decode<GROUPED>(p, prefix, item, it);
            const int64_t w_row0 = (int64_t)it.expert * p.N + (int64_t)it.tn * BN;
            const int g0 = (int)(w_row0 / 128); // first 128-row scale group of the W tile
            // gathered rows: source rows of this lane's 4 tile rows (row 0,
            // zero-filled, past the expert or for out-of-range indices)
            int64_t src[4] = {0, 0, 0, 0};
            bool live[4] = {false, false, false, false};
            if (indexed) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int64_t g = it.row0 + lane + 32 * q;
                    const int r = g < it.row_end && in_span(NV4_SITE(0), p.sp_row_idx, p.row_idx + g, 4)
                                      ? p.row_idx[g]
                                      : -1;
                    live[q] = r >= 0 && r < p.M;
                    src[q] = live[q] ? r : 0;
                }
            }
            int ng = 0;
#pragma unroll
            for (int h = 0; h < NG; ++h)
                ng += (g0 + h < p.w_groups) ? 1 : 0;
            for (int ks = 0; ks < p.ksteps; ++ks) {
                const bool got = mbar_wait(&raw_empty[st], ph ^ 1u, p.timeout_ns, abort_flag);
                if (!__all_sync(FULLMASK, got)) {
                    if (lane == 0)
                        timeout(p, abort_flag);
                    ok = false;
                    break;
                }
                uint8_t *r = raw + st * RAW_BYTES;
                if (lane == 0)
                    mbar_arrive_expect_tx(&raw_full[st], (indexed ? 0 : RAW_A) + RAW_W + ng * 512);
                __syncwarp();
                // op 0: A, 1: W codes, 2..2+NG-1: W scale atoms; lanes 8r.. serve steps r, r+4, ...
                const int op = lane - 8 * (issued & 3);
                if (op == 0 && !indexed)
                    tma_load_2d(r, &p.tmap_a, ks * KSTEP, (int)it.row0, &raw_full[st], RAW_A);
                else if (op == 1)
                    tma_load_2d(r + RAW_A, &p.tmap_w, ks * (KSTEP / 2), (int)w_row0, &raw_full[st], RAW_W);
                else if (op >= 2 && op < 2 + NG && g0 + op - 2 < p.w_groups &&
                         in_span(NV4_SITE(0), p.sp_w_scales,
                                 p.w_scales + ((size_t)(g0 + op - 2) * p.k64_total + ks) * 512, 512))
                    bulk_load(r + RAW_A + RAW_W + (op - 2) * 512,
                              p.w_scales + ((size_t)(g0 + op - 2) * p.k64_total + ks) * 512, 512, &raw_full[st]);
                if (indexed) {
                    // gathered FP8 rows: 64 bytes per row and step, plain
                    // row-major like the TMA box; every lane's copies
                    // complete the stage's barrier on their own
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint8_t *srow = p.a_fp8 + src[q] * p.K + (int64_t)ks * KSTEP;
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const bool in = live[q] && in_span(NV4_SITE(0), p.sp_a_fp8, srow + 16 * c, 16);
                            // the TMA's 64-byte swizzle, applied by hand
                            const int row = lane + 32 * q;
                            cp_async_16(r + row * KSTEP + ((c ^ ((row >> 1) & 3)) << 4), srow + 16 * c, in ? 16u : 0u);
                        }
                    }
                    cp_async_arrive_noinc(&raw_full[st]);
                }
                ++issued;
                if (++st == RAW_STAGES) {
                    st = 0;
                    ph ^= 1u;
                }
            }
        }
        if (lane == 0) {
            const int n = min(issued, RAW_STAGES);
            for (int q = 0; q < n; ++q) {
                if (--st < 0) {
                    st = RAW_STAGES - 1;
                    ph ^= 1u;
                }
                mbar_wait(&raw_full[st], ph, p.timeout_ns, nullptr);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_f16(BN);
            int cs = 0, acc = 0;
            uint32_t cph = 0, aph = 0;
            bool ok = true;
            for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
                if (!mbar_wait(&acc_empty[acc], aph ^ 1u, p.timeout_ns, abort_flag)) {
                    timeout(p, abort_flag);
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + acc * BN;
                uint32_t accumulate = 0;
                for (int ks = 0; ks < p.ksteps; ++ks) {
                    if (!mbar_wait(&conv_full[cs], cph, p.timeout_ns, abort_flag)) {
                        timeout(p, abort_flag);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t bd = sdesc_sw128(smem_u32(conv + cs * CONV_BYTES));
                    const uint32_t ta = tmem + A_BASE + cs * A_COLS;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) { // 16 FP16 per MMA: 8 A columns, 32 B bytes
                        mma_f16_ta(d, ta + 8 * kk, bd + (uint64_t)(kk * 2), idesc, accumulate);
                        accumulate = 1;
                    }
                    tc_commit(&conv_empty[cs]);
                    if (++cs == CONV_STAGES) {
                        cs = 0;
                        cph ^= 1u;
                    }
                }
                if (!ok)
                    break;
                tc_commit(&acc_full[acc]);
                if (++acc == ACC_BUFS) {
                    acc = 0;
                    aph ^= 1u;
                }
            }
            tc_commit(drain);
            mbar_wait(drain, 0, p.timeout_ns, nullptr);
        }
        __syncwarp();
    } else if (warp < 2 + CONV_WARPS) {
        // ------------------------------------------------------------ converters
        const int t = threadIdx.x - 64; // 0..255
        int rs = 0, cs = 0;
        uint32_t rph = 0, cph = 0;
        for (int item = blockIdx.x; item < total; item += gridDim.x) {
            bool ok = true;
            for (int ks = 0; ks < p.ksteps; ++ks) {
                const bool g1 = mbar_wait(&raw_full[rs], rph, p.timeout_ns, abort_flag);
                const bool g2 = g1 && mbar_wait(&conv_empty[cs], cph ^ 1u, p.timeout_ns, abort_flag);
                if (!__all_sync(FULLMASK, g2)) {
                    if (lane == 0)
                        timeout(p, abort_flag);
                    ok = false;
                    break;
                }
                const uint8_t *r = raw + rs * RAW_BYTES;
                uint8_t *cB = conv + cs * CONV_BYTES;
                // A rows of this warp's TMEM lane quarter, K half ah: 32 FP8
                // -> 32 FP16 = 16 columns of the step's A stage in TMEM
                {
                    const int quarter = warp & 3, ah = (warp - 2) >> 2;
                    const int ar = quarter * 32 + lane;
                    uint32_t o[16];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        // chunk 2 ah + h of the row, 64-byte swizzled
                        const uint4 v = *reinterpret_cast<const uint4 *>(
                            r + ar * KSTEP + (((2 * ah + h) ^ ((ar >> 1) & 3)) << 4)); // 16 FP8 -> 8 columns
                        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            o[8 * h + 2 * q] = f16x2_from_e4m3x2(w[q] & 0xFFFFu);
                            o[8 * h + 2 * q + 1] = f16x2_from_e4m3x2(w[q] >> 16);
                        }
                    }
                    tc_st_32x32b_x16(tmem + ((uint32_t)(quarter * 32) << 16) + A_BASE + cs * A_COLS + 16 * ah, o);
                }
                // W: two threads per row, each half a row (16 code bytes = two
                // 16-element blocks) x their E4M3 scales -> 32 FP16, rows
                // t / 2 and 128 + t / 2.  Eight threads of a load cover four
                // whole 32-byte rows, and their stores land in eight
                // different 16-byte chunk positions: no bank conflicts
#pragma unroll
                for (int pass = 0; pass < 2; ++pass) {
                    const int wrow = pass * 128 + (t >> 1), hw = t & 1;
                    const uint4 v = *reinterpret_cast<const uint4 *>(r + RAW_A + wrow * (KSTEP / 2) + hw * 16);
                    const uint32_t sc = *reinterpret_cast<const uint32_t *>(
                        r + RAW_A + RAW_W + (wrow >> 7) * 512 + (wrow & 31) * 16 + ((wrow & 127) >> 5) * 4);
                    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int bb = 0; bb < 2; ++bb) { // 16-element block b = 2 hw + bb uses scale byte b
                        const int b = 2 * hw + bb;
                        const uint32_t s2 = f16x2_from_e4m3x2(((sc >> (8 * b)) & 0xFFu) * 0x0101u);
                        uint32_t o[8];
#pragma unroll
                        for (int q = 0; q < 2; ++q)
#pragma unroll
                            for (int y = 0; y < 4; ++y)
                                o[4 * q + y] = hmul2_u32(f16x2_from_e2m1x2((w4[2 * bb + q] >> (8 * y)) & 0xFFu), s2);
                        const int c0 = 2 * b, c1 = 2 * b + 1;
                        *reinterpret_cast<uint4 *>(cB + wrow * 128 + ((c0 ^ (wrow & 7)) << 4)) =
                            make_uint4(o[0], o[1], o[2], o[3]);
                        *reinterpret_cast<uint4 *>(cB + wrow * 128 + ((c1 ^ (wrow & 7)) << 4)) =
                            make_uint4(o[4], o[5], o[6], o[7]);
                    }
                }
                // A (TMEM stores) and W (shared memory) reach the tensor core
                // before this warp's arrival
                tc_wait_st();
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&conv_full[cs]);
                    mbar_arrive(&raw_empty[rs]);
                }
                if (++rs == RAW_STAGES) {
                    rs = 0;
                    rph ^= 1u;
                }
                if (++cs == CONV_STAGES) {
                    cs = 0;
                    cph ^= 1u;
                }
            }
            if (!ok)
                break;
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;                     // the TMEM lane quarter this warp may access
        const int chalf = (warp - EPI_FIRST_WARP) >> 2; // which 128 accumulator columns
        const OutDesc out_desc{p.out, p.ldy, 1, p.out_dtype, p.vec_ok, p.sp_out};
        const int row = q * 32 + lane;
        int acc = 0;
        uint32_t aph = 0;
        for (int item = blockIdx.x; item < total; item += gridDim.x) {
            Item it;
            decode<GROUPED>(p, prefix, item, it);
            const int tn = it.tn;
            const bool got = mbar_wait(&acc_full[acc], aph, p.timeout_ns, abort_flag);
            if (!__all_sync(FULLMASK, got)) {
                if (lane == 0)
                    timeout(p, abort_flag);
                break;
            }
            tc_fence_after();
            const int64_t i = it.row0 + row;
            const bool row_ok = i < it.row_end;
            int64_t tok = i;
            if (indexed && row_ok) {
                const int r = in_span(NV4_SITE(0), p.sp_row_idx, p.row_idx + i, 4) ? p.row_idx[i] : -1;
                tok = (r >= 0 && r < p.M) ? r : -1;
            }
            const bool scales_in = row_ok && tok >= 0 && in_span(NV4_SITE(0), p.sp_s_t, p.s_t + tok, 4) &&
                                   in_span(NV4_SITE(0), p.sp_w_second, p.w_second + it.expert, 4);
            const float alpha = scales_in ? p.s_t[tok] * p.w_second[it.expert] : 0.0f;
            const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16) + acc * BN;
            for (int c0 = chalf * (BN / 2); c0 < (chalf + 1) * (BN / 2); c0 += 32) {
                uint32_t v[32];
                tc_ld_32x32b_x32(tb + c0, v);
                tc_wait_ld();
                // the warp's 32 rows together (32-byte stores of whole row
                // runs; each lane scales its own row by its alpha)
                store_chunk32_warp(out_desc, v, it.row0 + q * 32, it.row0, it.row_end, (int64_t)tn * BN + c0,
                                   alpha, p.N, lane);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&acc_empty[acc]);
            if (++acc == ACC_BUFS) {
                acc = 0;
                aph ^= 1u;
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

cudaError_t launch_w4a8(const W4A8GemmArgs &g, cudaStream_t stream)
{
    if (g.K % KSTEP != 0)
        return cudaErrorInvalidValue;
    const bool grouped = g.E > 0;
    const int64_t w_rows = grouped ? (int64_t)g.E * g.N : g.N;
    Params p{};
    // the raw FP8 A tile with the 64-byte swizzle: 16-byte chunk c of row r
    // lands at chunk c ^ ((r / 2) % 4), so the converters' per-row reads hit
    // every bank once
    CUresult r = make_tmap_2d_u8_swizzle(&p.tmap_a, g.a_fp8, (uint64_t)g.K, (uint64_t)g.M, (uint64_t)g.K, KSTEP, BM,
                                         CU_TENSOR_MAP_SWIZZLE_64B);
    if (r != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    r = make_tmap_2d_u8(&p.tmap_w, g.w_codes, (uint64_t)(g.K / 2), (uint64_t)w_rows, (uint64_t)(g.K / 2), KSTEP / 2,
                        BN, false);
    if (r != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    p.w_scales = g.w_scales;
    p.s_t = g.s_t;
    p.w_second = g.w_second;
    p.out = g.out;
    p.ldy = g.ldy;
    p.M = g.M;
    p.N = g.N;
    p.m_tiles = (int)ceil_div(g.M, BM);
    p.n_tiles = (int)ceil_div(g.N, BN);
    p.ksteps = (int)(g.K / KSTEP);
    p.k64_total = (int)(g.K / 64);
    p.w_groups = (int)ceil_div(w_rows, 128);
    p.out_dtype = g.out_dtype;
    const int esz = g.out_dtype == NVFP4_OUT_BF16 ? 2 : 4;
    p.vec_ok = out_vec_level(g.out, g.ldy, 1, esz);
    p.status = g.status;
    p.timeout_ns = g.timeout_ns;
    p.a_fp8 = g.a_fp8;
    p.K = g.K;
    p.offsets = g.offsets;
    p.row_idx = g.row_idx;
    p.E = g.E;
    p.total_rows = g.total_rows;
    p.sp_w_scales = span_of(g.w_scales, tiled_scale_bytes(w_rows, g.K));
    p.sp_s_t = span_of(g.s_t, 4u * (uint64_t)g.M);
    p.sp_w_second = span_of(g.w_second, 4u * (uint64_t)(grouped ? g.E : 1));
    p.sp_out = span_of(g.out, matrix_bytes(grouped ? g.total_rows : g.M, g.N, g.ldy, esz));
    p.sp_a_fp8 = span_of(g.a_fp8, (uint64_t)g.M * (uint64_t)g.K);
    p.sp_offsets = span_of(g.offsets, 8u * (uint64_t)(g.E + 1));
    p.sp_row_idx = span_of(g.row_idx, 4u * (uint64_t)g.total_rows);
    auto kern = grouped ? w4a8_kernel<true> : w4a8_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess)
        return e;
    // grouped: an upper bound of the items (every expert's rows in 128-row
    // blocks, plus one partial block per expert); the kernel counts them
    const int64_t items = grouped ? (ceil_div(g.total_rows, BM) + g.E) * p.n_tiles : (int64_t)p.m_tiles * p.n_tiles;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(items, device_sm_count()));
    kern<<<grid, THREADS, SMEM_BYTES, stream>>>(p);
    return cudaGetLastError();
}

} // namespace nv4
