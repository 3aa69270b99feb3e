// W4A4 block-scaled GEMM on 5th-generation tensor cores (tcgen05, sm_103a).
//
// Computes D[i][j] = alpha * sum_k A[i][k] * B[j][k] where A and B are NVFP4
// (E2M1 codes with one UE4M3 scale per 16 elements of K), the contraction
// that "NVIDIA Ships TensorRT-LLM 0.16: Native FP4 Quantization for Blackwell
// B200", section "The Mathematical Breakthrough of Microscopic FP4 Scaling",
// item 3 "Hardware-Fused Dequantization" describes: the tensor cores take the
// FP4 codes and the micro-scales directly and apply the scales before the
// dot products.  alpha is the product of the two FP32 second-level scales.
// The grouped variant serves the mixture-of-experts operations of "llama.cpp
// Put Precision Policy Inside the Model. That Matters More Than W4A4",
// section "One model can need more than one precision".
//
// Design (one CTA per SM, persistent, warp-specialised, 384 threads):
//   warp 0      producer: A/B code tiles by TMA (128-byte rows = 256 FP4,
//               128-byte swizzle), A's compact 512-byte scale atoms by a bulk
//               copy and B's (the stage's atoms of both 128-row groups) by
//               one 4-D TMA copy, into a STAGES-deep ring; each copy of a
//               stage is issued by its own lane (one thread's copies are
//               served in order, different threads' copies in parallel).
//   warp 1      allocates TMEM; lane 0 issues tcgen05.mma kind::mxf4nvf4
//               (M = 128, N = BN, K = 64; 4 per stage) and tcgen05.commit.
//   warp 2      scale warp: moves each stage's compact scale atoms from the
//               ring to TMEM with tcgen05.cp.32x128b.warpx4 (the copy engine
//               replicates every 32-row atom into all four TMEM lane
//               quarters, which is what each quarter of the tensor core
//               reads: row m of A at lane m, column address + m / 32; B in
//               every quarter), off the MMA thread.  Measured on B300 this
//               beats rebuilding replicated copy sources in shared memory
//               with the threads: shared-memory bandwidth, not the copy
//               engine, limits a stage.
//   warps 3-10  epilogue: tcgen05.ld of the FP32 accumulator into registers,
//               release of the accumulator, then alpha scale and BF16/FP32
//               stores (with 32-byte aligned rows, whole 64-byte row runs:
//               each warp exchanges its 32 rows' words by shuffles so every
//               256-bit store covers 16 rows).  Stream-K partial tiles: a
//               CTA whose range starts inside a tile parks its FP32 partial
//               in its own workspace slot and raises its flag; the CTA
//               holding the tile's first K stages (its last work item)
//               parks its accumulator in the idle ring, adds the flagged
//               contributors' slots and stores the tile.
//   warp 11     grouped with routing indices only, gather warp: the
//               activation rows of a work item (gathered through the
//               indices) and their scale bytes by 16- and 4-byte cp.async
//               into the stages the producer arms, so those many small
//               copies do not hold up the producer's bulk copies.
//               Contiguous grouped rows need no gather: an expert's tiles
//               start at the 128-row boundary at or below its first row,
//               so they load like dense tiles (TMA codes, bulk-copied scale
//               atoms) and the leading rows of the previous expert are
//               computed but not stored.
// The dense launch is a programmatic dependent launch: set-up, tensor-map
// fetch and the first weight stages' L2 prefetch overlap the previous grid
// (normally the activation quantiser); every access to memory the previous
// grid touches comes after griddepcontrol.wait.
// Every mbarrier wait is bounded; on timeout the CTA records NVFP4 TIMEOUT in
// the status word, drains its in-flight copies and MMAs, frees TMEM and
// exits (epilogue warps decide together through a barrier reduction).
#include <algorithm>
#include <cuda_bf16.h>

#include "epilogue.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace nv4 {

namespace {

constexpr int BM = 128;
constexpr int STAGE_K_BYTES = 128; // per row and stage: 256 FP4 elements
constexpr int EPI_WARPS = 8;
constexpr int EPI_FIRST_WARP = 3;
constexpr int GATHER_WARP = EPI_FIRST_WARP + EPI_WARPS; // grouped: activation row / scale gathers
constexpr int THREADS = 32 * (GATHER_WARP + 1);
constexpr int MAX_EXPERTS = 1024;

// AR: activation rows one stage holds.  128 in general; 16 for the decode
// shapes (M <= 16), whose stages then take 14 KB less shared memory, which
// buys a deeper ring (more weight bytes in flight per SM).  The MMA still
// reads 128 rows; rows past the 16 loaded ones read whatever follows in
// shared memory and only feed output rows that are never stored.
template <int BN, int AR = BM>
struct Cfg {
    static_assert(BN == 128 || BN == 256, "N tile");
    static_assert(AR == BM || AR == 16, "activation rows per stage");
    static constexpr int NB = BN / 128;                 // 128-row scale groups per B tile
    static constexpr int STAGES = AR == BM ? (BN == 256 ? 4 : 6) : (BN == 256 ? 5 : 8);
    static constexpr int ACC_BUFS = BN == 256 ? 1 : 2;
    static constexpr int A_BYTES = AR * STAGE_K_BYTES;
    static constexpr int B_BYTES = BN * STAGE_K_BYTES;
    static constexpr int SFA_BYTES = 4 * 512;           // compact atoms as loaded
    static constexpr int SFB_BYTES = NB * 4 * 512;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
    static constexpr int SF_COLS = 16 + 16 * NB;        // TMEM scale columns per stage
    static constexpr int SF_BASE = ACC_BUFS * BN;
    static constexpr int TMEM_COLS = 512;
    static constexpr int BAR_BYTES = 512;
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + BAR_BYTES + 1024;
    static constexpr int EPI_COLS = BN / 2;              // accumulator columns per epilogue warp
    static_assert(SF_BASE + STAGES * SF_COLS <= TMEM_COLS, "TMEM budget");
    static_assert(STAGE_BYTES % 1024 == 0, "alignment");
    static_assert(SMEM_BYTES + 4 * (2 * MAX_EXPERTS + 3) <= 232448, "shared memory budget");
};

struct Params {
    CUtensorMap tmap_a;  // MMA operand A codes [a_rows][K/2]
    CUtensorMap tmap_b;  // MMA operand B codes
    CUtensorMap tmap_sfb; // B's scale atoms, [groups][k64][4][128 B]: one box per stage
    const uint8_t *a_codes; // indexed grouped rows are copied from here with cp.async
    const uint8_t *sfa;  // tiled scales of A (row-padded to 128)
    const uint8_t *sfb;  // tiled scales of B
    const float *a_second;
    const float *b_second; // [1] dense, [E] grouped
    void *out;
    int64_t ld_i, ld_j;
    float *slots;            // stream-K: one FP32 partial tile [a_rows][BN] per CTA
    uint32_t *flags;         // stream-K: one ready flag per CTA, zero between calls
    int64_t a_rows, b_rows; // valid extents (b_rows = N per expert in grouped mode)
    int64_t slot_stride;    // stream-K: floats per partial slot (a_rows * BN)
    int32_t m_tiles, n_tiles, k64, kstages, streamk, group_m;
    int32_t out_dtype, vec_ok;
    int32_t b_row_tiles;    // 128-row scale atoms available in B (total)
    int32_t a_box_rows;     // rows of A one stage loads (128, or M rounded up to 16 when M < 128)
    int32_t b_early;        // issue the first stages' B copies before waiting for the previous grid
    int32_t diag_skip_flag; // stream-K: the CTA that does not raise its ready flag (-1: none)
    // NVFP4 output (the next layer's quantiser fused into the epilogue):
    // codes [a_rows][b_rows/2], MMA-tiled scales, under the given tensor
    // scale; the largest |Y| is max-reduced into yq_amax when it is set
    int32_t out_q;
    int64_t yq_n;            // columns of the NVFP4 output
    uint8_t *yq_codes;
    uint8_t *yq_scales;
    const float *yq_scale;
    uint32_t *yq_amax;
    // grouped mode
    int32_t epi;             // EPI_PLAIN, EPI_SWIGLU or EPI_COMBINE
    const int32_t *comb_idx; // combine: token of each routed row
    const float *comb_w;     // combine: routing weight of each routed row
    int64_t comb_rows;       // combine: token rows of the output
    const int64_t *offsets;
    const int32_t *row_idx;
    int32_t E;
    int64_t total_rows;      // rows of the index list / output (offsets are clamped to it)
    uint32_t *status;
    uint64_t timeout_ns;
    // the bytes the call's arguments grant each tensor (tested before each
    // plain access in the bounds-checked build)
    Span sp_a_codes, sp_sfa, sp_sfb, sp_b_second, sp_out, sp_slots, sp_flags, sp_yq_codes, sp_yq_scales;
    Span sp_comb_idx, sp_comb_w, sp_offsets, sp_row_idx;
};

struct Tile {
    int tile, tile_m, tile_n, kst0, kst1;
    int expert;            // grouped
    int64_t row0, row_end; // grouped: first output row of the tile, end of the expert's rows
    int64_t row_lo;        // grouped: the expert's first row (rows below it are not stored)
};

// Tiles in bands of group_m M-tiles, M fastest inside a band, so CTAs running
// at the same time share weight tiles (L2) and, when the band holds every
// M-tile, each weight tile comes from HBM once.
__device__ __forceinline__ void decode_dense(const Params &p, int tile, Tile &t)
{
    const int band = p.group_m * p.n_tiles;
    const int bid = tile / band;
    const int first_m = bid * p.group_m;
    const int gsize = min(p.m_tiles - first_m, p.group_m);
    const int rr = tile - bid * band;
    t.tile = tile;
    t.tile_m = first_m + rr % gsize;
    t.tile_n = rr / gsize;
    t.kst0 = 0;
    t.kst1 = p.kstages;
    t.expert = 0;
    t.row0 = 0;
    t.row_end = 0;
    t.row_lo = 0;
}

// Grouped: first row of expert e's first tile.  Gathered rows start at the
// expert's first row; contiguous rows start at the 128-row boundary at or
// below it, so every tile lines up with the activations' 128-row scale
// atoms and loads like a dense tile (the rows before the expert's first one
// belong to the previous expert: computed, never stored).
__device__ __forceinline__ int64_t expert_tile_base(const Params &p, int64_t lo)
{
    return p.row_idx == nullptr ? (lo & ~(int64_t)(BM - 1)) : lo;
}

// Grouped: number of 128-row tiles of expert e's rows [lo, hi).
__device__ __forceinline__ int expert_tiles(const Params &p, int64_t lo, int64_t hi)
{
    return hi > lo ? (int)((hi - expert_tile_base(p, lo) + BM - 1) / BM) : 0;
}

// Expert e's output rows [lo, hi), with the device offsets clamped to
// [0, total_rows] and made non-decreasing so a malformed list cannot address
// memory outside the index list or the output.
__device__ __forceinline__ void expert_rows(const Params &p, int e, int64_t &lo, int64_t &hi)
{
    if (!in_span(NV4_SITE(0), p.sp_offsets, p.offsets + e, 16)) {
        lo = hi = 0;
        return;
    }
    lo = min(max(p.offsets[e], (int64_t)0), p.total_rows);
    hi = min(max(p.offsets[e + 1], lo), p.total_rows);
}

// Grouped: prefix[e] = number of 128-row tiles of experts 0..e-1, and from
// prefix + MAX_EXPERTS + 1 on, elo[e] = offsets[e] clamped to [0,
// total_rows] (e = 0..E), so expert e's rows are [elo[e], max(elo[e + 1],
// elo[e])): expert_rows without a global load.
__device__ __forceinline__ void decode_grouped(const Params &p, const int *prefix, int item, Tile &t)
{
    const int tile_idx = item / p.n_tiles;
    int lo = 0, hi = p.E; // find e with prefix[e] <= tile_idx < prefix[e+1]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (prefix[mid] <= tile_idx)
            lo = mid;
        else
            hi = mid;
    }
    const int e = lo;
    const int mt_e = prefix[e + 1] - prefix[e];
    const int local = item - prefix[e] * p.n_tiles;
    t.tile = item;
    t.expert = e;
    t.tile_n = local / mt_e;
    const int mt = local - t.tile_n * mt_e;
    t.tile_m = mt;
    const int *elo = prefix + MAX_EXPERTS + 1;
    const int64_t r_lo = elo[e], r_hi = max(elo[e + 1], elo[e]);
    t.row0 = expert_tile_base(p, r_lo) + (int64_t)mt * BM;
    t.row_end = r_hi;
    t.row_lo = r_lo;
    t.kst0 = 0;
    t.kst1 = p.kstages;
}

// The sequence of work segments of one CTA, identical for all its roles.
// Static mode: whole tiles blockIdx.x, blockIdx.x + gridDim.x, ...
// Stream-K mode: the contiguous range [b*T/G, (b+1)*T/G) of the flattened
// (tile, K-stage) space, cut at tile boundaries.  A CTA's range starts
// inside at most one tile (its first), so one partial slot per CTA suffices.
struct WorkIter {
    int64_t g, g_end;
    int item;
};

__device__ __forceinline__ void work_begin(const Params &p, int total_items, WorkIter &w)
{
    if (p.streamk) {
        const int64_t T = (int64_t)total_items * p.kstages;
        w.g = (int64_t)blockIdx.x * T / gridDim.x;
        w.g_end = (int64_t)(blockIdx.x + 1) * T / gridDim.x;
    }
    w.item = blockIdx.x;
}

template <bool GROUPED>
__device__ __forceinline__ bool work_next(const Params &p, const int *prefix, int total_items, WorkIter &w, Tile &t)
{
    if (!GROUPED && p.streamk) {
        if (w.g >= w.g_end)
            return false;
        const int tile = (int)(w.g / p.kstages);
        const int k0 = (int)(w.g - (int64_t)tile * p.kstages);
        const int64_t rem = w.g_end - w.g;
        const int k1 = rem < (int64_t)(p.kstages - k0) ? k0 + (int)rem : p.kstages;
        decode_dense(p, tile, t);
        t.kst0 = k0;
        t.kst1 = k1;
        w.g += k1 - k0;
        return true;
    }
    if (w.item >= total_items)
        return false;
    if (GROUPED)
        decode_grouped(p, prefix, w.item, t);
    else
        decode_dense(p, w.item, t);
    w.item += gridDim.x;
    return true;
}

// The same sequence for roles that need only the number of K stages of each
// work item (the MMA and scale warps): grouped items always run every K
// stage, so their expert rows (global offsets) are not loaded.
template <bool GROUPED>
__device__ __forceinline__ bool work_next_light(const Params &p, const int *prefix, int total_items, WorkIter &w,
                                                Tile &t)
{
    if (!GROUPED)
        return work_next<false>(p, prefix, total_items, w, t);
    if (w.item >= total_items)
        return false;
    t.tile = w.item;
    t.kst0 = 0;
    t.kst1 = p.kstages;
    w.item += gridDim.x;
    return true;
}

// Grouped: source activation row of tile rows lane + 32q, in two steps so
// the index loads of the next work item stay in flight while the current
// one runs: tile_rows_load issues them (raw[q]: the index, or NO_ROW for
// rows past the expert), tile_rows_use validates (row 0 for rows past the
// expert or out-of-range indices, whose results are unspecified).
constexpr int NO_ROW = -2147483647 - 1;
__device__ __forceinline__ void tile_rows_load(const Params &p, bool indexed, const Tile &t, int lane,
                                               int (&raw)[4])
{
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int64_t g = t.row0 + lane + 32 * q;
        int r = NO_ROW;
        if (g < t.row_end) {
            if (!indexed)
                r = (int)g;
            else if (in_span(NV4_SITE(0), p.sp_row_idx, p.row_idx + g, 4))
                r = p.row_idx[g];
            else
                r = 0;
        }
        raw[q] = r;
    }
}

__device__ __forceinline__ void tile_rows_use(const Params &p, const int (&raw)[4], int (&src_row)[4],
                                              bool (&row_ok)[4])
{
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        row_ok[q] = raw[q] != NO_ROW;
        int r = raw[q];
        if (r < 0 || r >= p.a_rows)
            r = 0;
        src_row[q] = r;
    }
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

__device__ __forceinline__ void record_timeout(const Params &p, volatile int *abort_flag)
{
    *abort_flag = 1;
    atomicOr(p.status, ST_TIMEOUT);
}

__device__ __forceinline__ void st_release_gpu(uint32_t *addr, uint32_t v)
{
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *addr)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(addr) : "memory");
    return v;
}

// Bounded wait for another CTA's ready flag (true once it reads non-zero).
__device__ __forceinline__ bool wait_flag(const uint32_t *f, uint64_t timeout_ns, const volatile int *abort_flag)
{
    const uint64_t t0 = globaltimer_ns();
    while (ld_acquire_gpu(f) == 0u) {
        if (*abort_flag || globaltimer_ns() - t0 > timeout_ns)
            return false;
        __nanosleep(64);
    }
    return true;
}

__device__ __forceinline__ OutDesc out_desc(const Params &p)
{
    return OutDesc{p.out, p.ld_i, p.ld_j, p.out_dtype, p.vec_ok, p.sp_out};
}

__device__ __forceinline__ QSpans q_spans(const Params &p)
{
    return QSpans{p.sp_yq_codes, p.sp_yq_scales};
}

// Row i of the NVFP4 output: its code row and the base of its scale slots.
__device__ __forceinline__ void q_row(const Params &p, int64_t i, uint8_t *&crow, uint8_t *&srow)
{
    q_row_addr(i, p.yq_n, p.yq_codes, p.yq_scales, crow, srow);
}

template <int BN, bool GROUPED, int AR>
__global__ void __launch_bounds__(THREADS, 1) w4a4_kernel(const __grid_constant__ Params p)
{
    using C = Cfg<BN, AR>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::STAGES * C::STAGE_BYTES);
    uint64_t *empty = full + C::STAGES;
    uint64_t *sf_ready = empty + C::STAGES;
    uint64_t *sf_full = sf_ready + C::STAGES;
    uint64_t *acc_full = sf_full + C::STAGES;
    uint64_t *acc_empty = acc_full + C::ACC_BUFS;
    uint64_t *drain = acc_empty + C::ACC_BUFS;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    __shared__ int prefix[GROUPED ? 2 * (MAX_EXPERTS + 1) : 1];
    __shared__ int total_items_s;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    constexpr unsigned FULLMASK = 0xFFFFFFFFu;

    const bool indexed = GROUPED && p.row_idx != nullptr;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            // codes: the bulk copies (one arrival), plus one cp.async
            // arrival per producer lane for gathered rows; scales likewise
            // (grouped: the activation scales are gathered by cp.async)
            mbar_init(&full[s], indexed ? 33 : 1);
            mbar_init(&sf_full[s], indexed ? 33 : 1);
            mbar_init(&empty[s], 1);
            mbar_init(&sf_ready[s], 1);
        }
        for (int b = 0; b < C::ACC_BUFS; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], EPI_WARPS);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    if (GROUPED) {
        if (warp == 2) {
            pdl_wait(); // the expert offsets may come from the previous grid
            // tiles per expert, prefix-summed by one warp: lane l owns a
            // contiguous run of experts; a shuffle scan joins the runs
            const int per = (p.E + 31) / 32;
            const int e0 = min(lane * per, p.E), e1 = min(e0 + per, p.E);
            int run = 0;
            for (int e = e0; e < e1; ++e) {
                int64_t lo, hi;
                expert_rows(p, e, lo, hi);
                run += expert_tiles(p, lo, hi);
            }
            int incl = run;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(FULLMASK, incl, o);
                if (lane >= o)
                    incl += v;
            }
            int acc = incl - run;
            int *elo = prefix + MAX_EXPERTS + 1;
            if (lane == 0)
                prefix[0] = 0;
            for (int e = e0; e < e1; ++e) {
                int64_t lo, hi;
                expert_rows(p, e, lo, hi);
                acc += expert_tiles(p, lo, hi);
                prefix[e + 1] = acc;
                elo[e] = (int)lo; // < 2^31: total_rows is bounded by the host checks
            }
            if (lane == 31) {
                total_items_s = incl * p.n_tiles;
                // offsets[E] clamped to [0, total_rows], as expert_rows clamps it
                elo[p.E] = (int)(in_span(NV4_SITE(0), p.sp_offsets, p.offsets + p.E, 8)
                                     ? min(max(p.offsets[p.E], (int64_t)0), p.total_rows)
                                     : 0);
            }
        }
    } else if (threadIdx.x == 0) {
        total_items_s = p.m_tiles * p.n_tiles;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int total_items = total_items_s;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        int stage = 0;
        uint32_t phase = 0;
        int issued = 0;
        bool ok = true;
        WorkIter wi;
        work_begin(p, total_items, wi);
        Tile t;
        // Copies of one stage (one per lane: copies issued by one thread
        // are served one after another, copies from different threads
        // overlap; lanes 8r..8r+4 serve stages r, r+4, ... so each thread has
        // at most one copy of four consecutive stages outstanding).
        // op 0: A codes, 1: B codes, 2: A scales, 3..3+NB-1: B scales.  Codes
        // and scales land on separate barriers, so the scale warp starts on a
        // stage's (small) scale copies while its codes are still in flight.
        auto issue = [&](const Tile &tt, int kb, int st, int idx, bool expect, bool part_b, bool part_a) {
            const int nk = min(4, p.k64 - 4 * kb);
            uint8_t *sA = smem + st * C::STAGE_BYTES;
            uint8_t *sB = sA + C::A_BYTES;
            uint8_t *sSFA = sB + C::B_BYTES;
            uint8_t *sSFB = sSFA + C::SFA_BYTES;
            const int brow0 = GROUPED ? tt.expert * (int)p.b_rows + tt.tile_n * BN : tt.tile_n * BN;
            const int bt0 = brow0 / 128;
            if (expect) {
                const uint32_t code_bytes =
                    C::B_BYTES + (indexed ? 0u : (uint32_t)p.a_box_rows * STAGE_K_BYTES);
                // A's atoms of the stage's K blocks; B's box is always whole
                // (atoms past K or past the weight rows read as zero)
                const uint32_t sf_bytes = (indexed ? 0u : (uint32_t)nk * 512u) + (uint32_t)C::SFB_BYTES;
                if (lane == 0)
                    mbar_arrive_expect_tx(&full[st], code_bytes);
                else if (lane == 1)
                    mbar_arrive_expect_tx(&sf_full[st], sf_bytes);
                __syncwarp();
            }
            const int op = lane - 8 * (idx & 3);
            if (GROUPED && op == 1 && part_b) {
                // the experts' weights are read once: evict them first, so
                // the activation rows the gathers read again stay in L2
                tma_load_2d_hint(sB, &p.tmap_b, kb * STAGE_K_BYTES, brow0, &full[st], (uint32_t)C::B_BYTES,
                                 l2_policy_evict_first());
            } else if ((op == 1 && part_b) || (op == 0 && !indexed && part_a)) {
                const int arow = GROUPED ? (int)tt.row0 : tt.tile_m * BM;
                tma_load_2d(op == 0 ? sA : sB, op == 0 ? &p.tmap_a : &p.tmap_b, kb * STAGE_K_BYTES,
                            op == 0 ? arow : brow0, &full[st],
                            op == 0 ? (uint32_t)p.a_box_rows * STAGE_K_BYTES : (uint32_t)C::B_BYTES);
            } else if (op == 2 && !indexed && part_a) {
                const int64_t a_atom_row = GROUPED ? tt.row0 / BM : tt.tile_m;
                const uint8_t *src = p.sfa + ((size_t)a_atom_row * p.k64 + 4 * kb) * 512;
                if (in_span(NV4_SITE(0), p.sp_sfa, src, nk * 512))
                    bulk_load(sSFA, src, nk * 512, &sf_full[st]);
            } else if (op == 3 && part_b) {
                // both 128-row groups' atoms of the stage in one copy
                tma_load_4d(sSFB, &p.tmap_sfb, 0, 0, 4 * kb, bt0, &sf_full[st], (uint32_t)C::SFB_BYTES);
            }
        };
        // Before waiting for the previous grid (programmatic dependent
        // launch): fetch the tensor maps.  When the previous grid is the
        // activation quantiser of the same call (it signals only after its
        // own wait, so every grid before it has completed and the weights
        // are final), the weight copies of the first ring stages go out now
        // as well; their activation copies follow the wait.
        if (lane == 0) {
            prefetch_tmap(&p.tmap_a);
            prefetch_tmap(&p.tmap_b);
            prefetch_tmap(&p.tmap_sfb);
        }
        int n_early = 0;
        if (!GROUPED && p.b_early) {
            WorkIter pw;
            work_begin(p, total_items, pw);
            Tile pt;
            while (n_early < C::STAGES && work_next<GROUPED>(p, prefix, total_items, pw, pt))
                for (int kb = pt.kst0; kb < pt.kst1 && n_early < C::STAGES; ++kb, ++n_early)
                    issue(pt, kb, n_early, n_early, true, true, false);
        }
        pdl_wait();
        // (grouped: the activation rows and scales are gathered by the
        // gather warp; this warp issues the bulk copies only)
        while (ok && work_next<GROUPED>(p, prefix, total_items, wi, t)) {
            for (int kb = t.kst0; kb < t.kst1; ++kb) {
                const bool got = mbar_wait(&empty[stage], phase ^ 1u, p.timeout_ns, abort_flag);
                if (!__all_sync(FULLMASK, got)) {
                    if (lane == 0)
                        record_timeout(p, abort_flag);
                    ok = false;
                    break;
                }
                // stages issued early (ring slots still fresh) already have
                // their barriers armed and weight copies in flight
                const bool early = issued < n_early;
                issue(t, kb, stage, issued, !early, !early, true);
                ++issued;
                if (++stage == C::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        // every load is issued: the next grid in the stream may start its
        // set-up (it waits for this grid's completion before touching memory)
        pdl_trigger();
        // drain: wait (bounded) until every copy this warp issued has landed
        if (lane == 0) {
            const int n = min(issued, C::STAGES);
            int s = stage;
            uint32_t ph = phase;
            for (int q = 0; q < n; ++q) {
                if (--s < 0) {
                    s = C::STAGES - 1;
                    ph ^= 1u;
                }
                mbar_wait(&full[s], ph, p.timeout_ns, nullptr);
                mbar_wait(&sf_full[s], ph, p.timeout_ns, nullptr);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        pdl_wait(); // bounded waits below start after the previous grid
        if (lane == 0) {
            const uint32_t idesc = idesc_mxf4nvf4(BN);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            WorkIter wi;
            work_begin(p, total_items, wi);
            Tile t;
            while (ok && work_next_light<GROUPED>(p, prefix, total_items, wi, t)) {
                if (!mbar_wait(&acc_empty[acc], acc_phase ^ 1u, p.timeout_ns, abort_flag)) {
                    record_timeout(p, abort_flag);
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem + acc * BN;
                uint32_t accumulate = 0;
                for (int kb = t.kst0; kb < t.kst1; ++kb) {
                    if (!mbar_wait(&full[stage], phase, p.timeout_ns, abort_flag) ||
                        !mbar_wait(&sf_ready[stage], phase, p.timeout_ns, abort_flag)) {
                        record_timeout(p, abort_flag);
                        ok = false;
                        break;
                    }
                    if (indexed) // gathered code rows were written by cp.async
                        fence_proxy_async_smem();
                    tc_fence_after();
                    const int nk = min(4, p.k64 - 4 * kb);
                    const uint8_t *sA = smem + stage * C::STAGE_BYTES;
                    const uint8_t *sB = sA + C::A_BYTES;
                    const uint32_t sf_col = tmem + C::SF_BASE + stage * C::SF_COLS;
                    const uint64_t adesc = sdesc_sw128(smem_u32(sA));
                    const uint64_t bdesc = sdesc_sw128(smem_u32(sB));
                    for (int kk = 0; kk < nk; ++kk) {
                        // A atom kk: 4 columns at 4 kk; B atom (kk, h): 4 columns
                        // at 16 + 4 kk (one 128-row group) or 16 + 8 kk + 4 h
                        const uint32_t sfa = sf_col + 4 * kk;
                        const uint32_t sfb = sf_col + 16 + (C::NB == 1 ? 4 * kk : 8 * kk);
                        // +32 bytes (64 FP4) inside the swizzled 128-byte row
                        mma_mxf4nvf4(d_tmem, adesc + (uint64_t)(kk * 2), bdesc + (uint64_t)(kk * 2), idesc, sfa,
                                     sfb, accumulate);
                        accumulate = 1;
                    }
                    tc_commit(&empty[stage]);
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok)
                    break;
                tc_commit(&acc_full[acc]);
                if (++acc == C::ACC_BUFS) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            // every MMA of this thread completes before TMEM is freed
            tc_commit(drain);
            mbar_wait(drain, 0, p.timeout_ns, nullptr);
        }
        __syncwarp();
    } else if (warp == 2) {
        // ------------------------------------------------------------ scale warp
        pdl_wait(); // bounded waits below start after the previous grid
        int stage = 0;
        uint32_t phase = 0;
        int issued = 0;
        bool ok = true;
        WorkIter wi;
        work_begin(p, total_items, wi);
        Tile t;
        while (ok && work_next_light<GROUPED>(p, prefix, total_items, wi, t)) {
            for (int kb = t.kst0; kb < t.kst1; ++kb) {
                const bool got = mbar_wait(&sf_full[stage], phase, p.timeout_ns, abort_flag);
                if (!__all_sync(FULLMASK, got)) {
                    if (lane == 0)
                        record_timeout(p, abort_flag);
                    ok = false;
                    break;
                }
                if (indexed) // gathered activation scales were written by cp.async
                    fence_proxy_async_smem();
                if (lane == 0) {
                    // atoms of B row groups past the weight rows read as zero
                    // bytes; they only feed output columns that are never stored
                    const int nk = min(4, p.k64 - 4 * kb);
                    const uint8_t *sSFA = smem + stage * C::STAGE_BYTES + C::A_BYTES + C::B_BYTES;
                    const uint8_t *sSFB = sSFA + C::SFA_BYTES;
                    const uint32_t sf_col = tmem + C::SF_BASE + stage * C::SF_COLS;
                    for (int kk = 0; kk < nk; ++kk) {
                        tc_cp_32x128b_warpx4(sf_col + 4 * kk, sdesc_sf(smem_u32(sSFA + kk * 512)));
                        if (C::NB == 1) {
                            tc_cp_32x128b_warpx4(sf_col + 16 + 4 * kk, sdesc_sf(smem_u32(sSFB + kk * 512)));
                        } else {
#pragma unroll
                            for (int h = 0; h < C::NB; ++h)
                                tc_cp_32x128b_warpx4(sf_col + 16 + 8 * kk + 4 * h,
                                                     sdesc_sf(smem_u32(sSFB + h * 2048 + kk * 512)));
                        }
                    }
                    tc_commit(&sf_ready[stage]);
                }
                __syncwarp();
                ++issued;
                if (++stage == C::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        // the copies this warp issued complete before TMEM is freed
        if (lane == 0) {
            const int n = min(issued, C::STAGES);
            int s_ = stage;
            uint32_t ph = phase;
            for (int q = 0; q < n; ++q) {
                if (--s_ < 0) {
                    s_ = C::STAGES - 1;
                    ph ^= 1u;
                }
                mbar_wait(&sf_ready[s_], ph, p.timeout_ns, nullptr);
            }
        }
        __syncwarp();
    } else if (warp < GATHER_WARP) {
        // ------------------------------------------------------------ epilogue
        const int ew = warp - EPI_FIRST_WARP;    // 0..7
        const int q = warp & 3;                  // the TMEM lane quarter this warp may access
        const int cbase = (ew >> 2) * C::EPI_COLS;
        const int row_in_tile = q * 32 + lane;
        int acc = 0;
        uint32_t acc_phase = 0;
        pdl_wait(); // activation scale, output and workspace follow the previous grid
        const float a_s = *p.a_second;
        WorkIter wi;
        work_begin(p, total_items, wi);
        Tile t;
        while (work_next<GROUPED>(p, prefix, total_items, wi, t)) {
            const bool got = mbar_wait(&acc_full[acc], acc_phase, p.timeout_ns, abort_flag);
            if (!epi_bar_all(got)) {
                if (threadIdx.x == 32 * EPI_FIRST_WARP)
                    record_timeout(p, abort_flag);
                break;
            }
            tc_fence_after();
            constexpr int NCH = C::EPI_COLS / 32;
            // the whole accumulator slice of this warp into registers, then
            // the accumulator goes back to the MMA warp (before any output
            // work, so the next tile's MMAs overlap this epilogue)
            uint32_t v[NCH][32];
            const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + acc * BN;
            // SwiGLU (BN == 256): the stacked weights interleave 128-row gate
            // and up blocks, so accumulator columns 0..127 hold the gate and
            // 128..255 the up products of the tile's 128 intermediate
            // columns; this warp takes 64 of them: gate chunks first, then
            // the matching up chunks
            const bool swiglu = GROUPED && p.epi == EPI_SWIGLU;
            const int h0 = (ew >> 2) * (BN / 4);
#pragma unroll
            for (int c = 0; c < NCH; ++c) {
                const int col = swiglu ? (c >= NCH / 2 ? BN / 2 : 0) + h0 + 32 * (c % (NCH / 2)) : cbase + 32 * c;
                tc_ld_32x32b_x32(tbase + col, v[c]);
            }
            tc_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&acc_empty[acc]);
            if (++acc == C::ACC_BUFS) {
                acc = 0;
                acc_phase ^= 1u;
            }
            const int b_idx = GROUPED ? t.expert : 0;
            const float alpha =
                a_s * (in_span(NV4_SITE(0), p.sp_b_second, p.b_second + b_idx, 4) ? p.b_second[b_idx] : 0.0f);
            int64_t i, i_end;
            if (GROUPED) {
                i = t.row0 + row_in_tile;
                // rows before the expert's first one (an aligned contiguous
                // tile) are the previous expert's: not stored
                i_end = i < t.row_lo ? i : t.row_end;
            } else {
                i = (int64_t)t.tile_m * BM + row_in_tile;
                i_end = p.a_rows;
            }
            const int64_t j_base = (int64_t)t.tile_n * BN + cbase;
            const int64_t j_end = p.b_rows;
            if (GROUPED && p.epi != EPI_PLAIN) {
                float m = 0.0f;
                if (p.epi == EPI_SWIGLU) {
                    const float s = p.out_q ? *p.yq_scale : 0.0f;
#pragma unroll
                    for (int c = 0; c < NCH / 2; ++c) {
                        // SiLU(g) * u into the gate chunk's registers
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            const float gv = __fmul_rn(alpha, __uint_as_float(v[c][e]));
                            const float uv = __fmul_rn(alpha, __uint_as_float(v[c + NCH / 2][e]));
                            // fast exponential and division: their relative
                            // error (~2^-21) is far inside the output
                            // tolerance, and they keep this epilogue shorter
                            // than the next tile's main loop
                            v[c][e] = __float_as_uint(__fmul_rn(__fdividef(gv, 1.0f + __expf(-gv)), uv));
                        }
                        const int64_t j = (int64_t)t.tile_n * (BN / 2) + h0 + 32 * c;
                        if (i < i_end) {
                            if (p.out_q) {
                                uint8_t *crow, *srow;
                                q_row(p, i, crow, srow);
                                m = fmaxf(m, encode_store_q(v[c], crow, srow, (int)j, s, q_spans(p)));
                            } else
                                store_chunk32(out_desc(p), v[c], i, j, 1.0f, i_end, p.yq_n);
                        }
                    }
                } else {
                    // gate-weighted combine: row i's products, times its
                    // routing weight, added to its token's output row (rows
                    // whose token index is out of range add nothing)
                    const bool row_in = i < i_end && in_span(NV4_SITE(0), p.sp_comb_idx, p.comb_idx + i, 4) &&
                                        in_span(NV4_SITE(0), p.sp_comb_w, p.comb_w + i, 4);
                    const int64_t tok = row_in ? (int64_t)p.comb_idx[i] : -1;
                    if (tok >= 0 && tok < p.comb_rows) {
                        const float gw = p.comb_w[i];
#pragma unroll
                        for (int c = 0; c < NCH; ++c) {
                            float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.out) + tok * p.ld_i +
                                                                     j_base + 32 * c);
                            if (!in_span(NV4_SITE(0), p.sp_out, dst, 128))
                                continue;
#pragma unroll
                            for (int e = 0; e < 32; e += 4)
                                atomicAdd(dst + e / 4, make_float4(gw * (alpha * __uint_as_float(v[c][e])),
                                                                   gw * (alpha * __uint_as_float(v[c][e + 1])),
                                                                   gw * (alpha * __uint_as_float(v[c][e + 2])),
                                                                   gw * (alpha * __uint_as_float(v[c][e + 3]))));
                        }
                    }
                }
                if (p.out_q && p.yq_amax != nullptr) {
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1)
                        m = fmaxf(m, __shfl_xor_sync(FULLMASK, m, o));
                    if (lane == 0)
                        atomicMax(p.yq_amax, __float_as_uint(m)); // |y| >= 0: bit order = value order
                }
                continue;
            }
            if (!GROUPED && p.out_q) {
                // NVFP4 output (whole tiles only; N is a multiple of 64)
                float m = 0.0f;
                uint8_t *crow, *srow;
                q_row(p, i, crow, srow);
                if (i < i_end) {
                    const float s = *p.yq_scale;
#pragma unroll
                    for (int c = 0; c < NCH; ++c) {
                        if (j_base + c * 32 >= j_end)
                            continue;
#pragma unroll
                        for (int e = 0; e < 32; ++e) // y = alpha * acc, as the FP32 output path forms it
                            v[c][e] = __float_as_uint(__fmul_rn(alpha, __uint_as_float(v[c][e])));
                        m = fmaxf(m, encode_store_q(v[c], crow, srow, (int)(j_base + c * 32), s, q_spans(p)));
                    }
                } else {
                    // padding rows of the last M tile (the tile's rows all
                    // exist in the scale layout): zero scales, as the
                    // quantisers leave them
                    for (int c = 0; c < NCH; ++c) {
                        const int j = (int)(j_base + c * 32);
                        if (j < j_end)
                            zero_pad_scales32(srow, j, q_spans(p));
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
                    m = fmaxf(m, __shfl_xor_sync(FULLMASK, m, o));
                if (p.yq_amax != nullptr && lane == 0)
                    atomicMax(p.yq_amax, __float_as_uint(m)); // |y| >= 0: bit order = value order
                continue;
            }
            const bool partial = !GROUPED && p.streamk && !(t.kst0 == 0 && t.kst1 == p.kstages);
            if (partial && t.kst0 != 0) {
                // contributor: this is the CTA's first tile and its range
                // starts inside it; park the raw partial and raise the flag
                float *slot = p.slots + (size_t)blockIdx.x * p.slot_stride + (size_t)row_in_tile * BN + cbase;
                if (i < i_end) {
#pragma unroll
                    for (int c = 0; c < NCH; ++c)
#pragma unroll
                        for (int u = 0; u < 32; u += 4)
                            if (in_span(NV4_SITE(0), p.sp_slots, slot + c * 32 + u, 16))
                                __stcg(reinterpret_cast<float4 *>(slot + c * 32 + u),
                                       make_float4(__uint_as_float(v[c][u]), __uint_as_float(v[c][u + 1]),
                                                   __uint_as_float(v[c][u + 2]), __uint_as_float(v[c][u + 3])));
                }
                epi_bar_sync();
                // (diag_skip_flag: a test names one CTA that never raises its
                // flag, so the owner's bounded wait runs out)
                if (threadIdx.x == 32 * EPI_FIRST_WARP && (int)blockIdx.x != p.diag_skip_flag &&
                    in_span(NV4_SITE(0), p.sp_flags, p.flags + blockIdx.x, 4)) {
                    __threadfence();
                    st_release_gpu(p.flags + blockIdx.x, 1u);
                }
                continue;
            }
            if (partial) {
                // owner: it holds the tile's first K stages, and since its
                // range ends inside the tile this is its last work item: every
                // load and MMA of the CTA has completed, so the ring's shared
                // memory is free.  The accumulator goes there (row stride
                // BN + 4 floats), then all epilogue threads add the partials
                // of the CTAs after this one whose ranges start inside the tile
                // (they wait on nothing, so the bounded wait is normally
                // already satisfied) and store the tile, coalesced.
                constexpr int RS = BN + 4;
                float *tile_s = reinterpret_cast<float *>(smem);
                fence_proxy_async_smem(); // the ring was last written by TMA
                if (i < i_end) {
#pragma unroll
                    for (int c = 0; c < NCH; ++c)
#pragma unroll
                        for (int u = 0; u < 32; u += 4)
                            if (in_dyn_smem(NV4_SITE(0), smem_u32(tile_s + row_in_tile * RS + cbase + c * 32 + u), 16))
                                *reinterpret_cast<float4 *>(tile_s + row_in_tile * RS + cbase + c * 32 + u) =
                                make_float4(__uint_as_float(v[c][u]), __uint_as_float(v[c][u + 1]),
                                            __uint_as_float(v[c][u + 2]), __uint_as_float(v[c][u + 3]));
                }
                const int64_t T = (int64_t)total_items * p.kstages;
                const int64_t tile_end = (int64_t)(t.tile + 1) * p.kstages;
                int n_contrib = 0;
                while (blockIdx.x + 1 + n_contrib < (int)gridDim.x &&
                       (int64_t)(blockIdx.x + 1 + n_contrib) * T / gridDim.x < tile_end)
                    ++n_contrib;
                bool got = true;
                if (threadIdx.x == 32 * EPI_FIRST_WARP)
                    for (int c = 1; c <= n_contrib && got; ++c)
                        got = in_span(NV4_SITE(0), p.sp_flags, p.flags + blockIdx.x + c, 4) &&
                              wait_flag(p.flags + blockIdx.x + c, p.timeout_ns, abort_flag);
                if (!epi_bar_all(got)) {
                    if (threadIdx.x == 32 * EPI_FIRST_WARP)
                        record_timeout(p, abort_flag);
                    break;
                }
                const int et = threadIdx.x - 32 * EPI_FIRST_WARP;
                const int64_t r0 = (int64_t)t.tile_m * BM; // dense: i_end = a_rows
                const int rows = (int)(i_end - r0 < BM ? i_end - r0 : BM);
                const int64_t c0 = (int64_t)t.tile_n * BN;
                const int cols = (int)(j_end - c0 < BN ? j_end - c0 : BN);
                // 4 consecutive columns per thread and position; UB positions
                // per round, the slot loads of CB contributors in flight
                // together (the partials are added in contributor order)
                constexpr int UB = 4, CB = 4;
                constexpr int STEP = 4 * 32 * EPI_WARPS;
                const int total4 = rows * BN;
                for (int base = et * 4; base < total4; base += UB * STEP) {
                    float4 acc4[UB];
#pragma unroll
                    for (int u = 0; u < UB; ++u) {
                        const int e4 = base + u * STEP;
                        const int r = e4 / BN, cc = e4 - r * BN;
                        acc4[u] = e4 < total4 && in_dyn_smem(NV4_SITE(0), smem_u32(tile_s + r * RS + cc), 16)
                                      ? *reinterpret_cast<const float4 *>(tile_s + r * RS + cc)
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                    for (int c0 = 1; c0 <= n_contrib; c0 += CB) {
                        float4 w4[CB][UB];
#pragma unroll
                        for (int b = 0; b < CB; ++b) {
                            const float *slot = p.slots + (size_t)(blockIdx.x + c0 + b) * p.slot_stride;
#pragma unroll
                            for (int u = 0; u < UB; ++u) {
                                const int e4 = base + u * STEP;
                                w4[b][u] = c0 + b <= n_contrib && e4 < total4 &&
                                                   in_span(NV4_SITE(0), p.sp_slots, slot + e4, 16)
                                               ? __ldcg(reinterpret_cast<const float4 *>(slot + e4))
                                               : make_float4(0.f, 0.f, 0.f, 0.f);
                            }
                        }
#pragma unroll
                        for (int b = 0; b < CB; ++b)
#pragma unroll
                            for (int u = 0; u < UB; ++u) {
                                if (c0 + b > n_contrib)
                                    continue;
                                acc4[u].x += w4[b][u].x;
                                acc4[u].y += w4[b][u].y;
                                acc4[u].z += w4[b][u].z;
                                acc4[u].w += w4[b][u].w;
                            }
                    }
#pragma unroll
                    for (int u = 0; u < UB; ++u) {
                        const int e4 = base + u * STEP;
                        if (e4 >= total4)
                            continue;
                        const int r = e4 / BN, cc = e4 - r * BN;
                        const float y4[4] = {alpha * acc4[u].x, alpha * acc4[u].y, alpha * acc4[u].z,
                                             alpha * acc4[u].w};
                        const int64_t row = r0 + r;
                        if (p.vec_ok && cc + 4 <= cols) {
                            if (p.out_dtype == NVFP4_OUT_BF16) {
                                __nv_bfloat162 h0 = __floats2bfloat162_rn(y4[0], y4[1]);
                                __nv_bfloat162 h1 = __floats2bfloat162_rn(y4[2], y4[3]);
                                const uint2 w2 = make_uint2(*reinterpret_cast<uint32_t *>(&h0),
                                                            *reinterpret_cast<uint32_t *>(&h1));
                                __nv_bfloat16 *d = static_cast<__nv_bfloat16 *>(p.out) + row * p.ld_i + c0 + cc;
                                if (in_span(NV4_SITE(0), p.sp_out, d, 8))
                                    *reinterpret_cast<uint2 *>(d) = w2;
                            } else {
                                float *d = static_cast<float *>(p.out) + row * p.ld_i + c0 + cc;
                                if (in_span(NV4_SITE(0), p.sp_out, d, 16))
                                    *reinterpret_cast<float4 *>(d) = make_float4(y4[0], y4[1], y4[2], y4[3]);
                            }
                        } else {
#pragma unroll
                            for (int q4 = 0; q4 < 4; ++q4) {
                                if (cc + q4 < cols) {
                                    const int64_t off = row * p.ld_i + (c0 + cc + q4) * p.ld_j;
                                    if (p.out_dtype == NVFP4_OUT_BF16) {
                                        if (in_span(NV4_SITE(0), p.sp_out, static_cast<__nv_bfloat16 *>(p.out) + off, 2))
                                            static_cast<__nv_bfloat16 *>(p.out)[off] = __float2bfloat16_rn(y4[q4]);
                                    } else if (in_span(NV4_SITE(0), p.sp_out, static_cast<float *>(p.out) + off, 4)) {
                                        static_cast<float *>(p.out)[off] = y4[q4];
                                    }
                                }
                            }
                        }
                    }
                }
                // every thread has read the slots: clear the flags for the next call
                epi_bar_sync();
                if (threadIdx.x == 32 * EPI_FIRST_WARP)
                    for (int c = 1; c <= n_contrib; ++c)
                        if (in_span(NV4_SITE(0), p.sp_flags, p.flags + blockIdx.x + c, 4))
                            p.flags[blockIdx.x + c] = 0u;
                continue;
            }
            const int64_t r0 = i - lane; // the warp's first row
            const int64_t i_lo = GROUPED ? t.row_lo : 0, i_hi = GROUPED ? t.row_end : p.a_rows;
            if (p.out_dtype == NVFP4_OUT_BF16 && rows64_ok(out_desc(p), j_base, j_end - 32 * (NCH - 1))) {
                // BF16 with 32-byte aligned rows: the whole slice packed first
                // (half the registers), then the warp's 32 rows together as
                // whole 64-byte runs
                if (r0 < i_hi && r0 + 32 > i_lo) {
                    uint32_t w[NCH][16];
#pragma unroll
                    for (int c = 0; c < NCH; ++c)
                        pack_bf16x32(v[c], alpha, w[c]);
#pragma unroll
                    for (int c = 0; c < NCH; ++c)
                        store_rows64(w[c], reinterpret_cast<uint8_t *>(static_cast<__nv_bfloat16 *>(p.out) + j_base + c * 32),
                                     p.ld_i * 2, r0, i_lo, i_hi, p.sp_out, lane);
                }
            } else {
#pragma unroll
                for (int c = 0; c < NCH; ++c)
                    store_chunk32(out_desc(p), v[c], i, j_base + c * 32, alpha, i < i_lo ? i : i_hi, j_end);
            }
        }
    } else if (GROUPED && indexed) {
        // ------------------------------------------------------------ gather warp
        // Grouped: the activation code rows (gathered) and the activation
        // scales of each stage, by 16- and 4-byte cp.async into the stage
        // the producer arms.  Many small copies per stage would otherwise
        // hold up the producer's bulk copies; this warp waits for the same
        // free slots and completes the stage's barriers with one arrival per
        // lane.  Items are decoded one ahead: the expert offsets come from
        // shared memory and the next item's row-index loads are issued when
        // the current item starts, to be used only by the next item.
        pdl_wait(); // the activations may come from the previous grid
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        WorkIter wi;
        work_begin(p, total_items, wi);
        Tile t, t_next;
        bool have_next = work_next<GROUPED>(p, prefix, total_items, wi, t_next);
        int src_row[4] = {0, 0, 0, 0}, next_raw[4] = {NO_ROW, NO_ROW, NO_ROW, NO_ROW};
        bool row_ok[4] = {false, false, false, false};
        if (have_next)
            tile_rows_load(p, indexed, t_next, lane, next_raw);
        while (ok && have_next) {
            t = t_next;
            tile_rows_use(p, next_raw, src_row, row_ok);
            have_next = work_next<GROUPED>(p, prefix, total_items, wi, t_next);
            if (have_next)
                tile_rows_load(p, indexed, t_next, lane, next_raw);
            for (int kb = t.kst0; kb < t.kst1; ++kb) {
                const bool got = mbar_wait(&empty[stage], phase ^ 1u, p.timeout_ns, abort_flag);
                if (!__all_sync(FULLMASK, got)) {
                    if (lane == 0)
                        record_timeout(p, abort_flag);
                    ok = false;
                    break;
                }
                const int nk = min(4, p.k64 - 4 * kb);
                uint8_t *sA = smem + stage * C::STAGE_BYTES;
                uint8_t *sSFA = sA + C::A_BYTES + C::B_BYTES;
                if (GROUPED) {
                    if (indexed) {
                        // gathered code rows: 16-byte cp.async with the 128-byte
                        // swizzle (chunk c of row r lands in chunk c ^ (r & 7)).
                        // Eight lanes take the eight chunks of one row, so a
                        // warp instruction covers four whole rows (four cache
                        // lines, not 32); tile row r's source row is held by
                        // lane r % 32 in src_row[r / 32] (-1: no row)
                        const int row_bytes = p.k64 * 32;
                        const int kbytes = min(STAGE_K_BYTES, row_bytes - kb * STAGE_K_BYTES);
                        const int c = lane & 7;
                        const int cbytes = max(0, min(16, kbytes - c * 16));
                        const uint64_t keep = l2_policy_evict_last();
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const int mine = row_ok[q] ? src_row[q] : -1;
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                const int r = 32 * q + 4 * j + (lane >> 3);
                                const int srow = __shfl_sync(FULLMASK, mine, 4 * j + (lane >> 3));
                                const uint8_t *src =
                                    p.a_codes + (size_t)max(srow, 0) * row_bytes + kb * STAGE_K_BYTES + c * 16;
                                int n = srow >= 0 ? cbytes : 0;
                                if (n && !in_span(NV4_SITE(0), p.sp_a_codes, src, n))
                                    n = 0;
                                cp_async_16_hint(sA + r * STAGE_K_BYTES + ((c ^ (r & 7)) << 4), n ? src : p.a_codes, n,
                                                 keep);
                            }
                        }
                    }
                    // activation scales of the tile's rows: 4 bytes per row and
                    // 64-K chunk, gathered asynchronously (zero for rows past
                    // the expert and chunks past K)
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int r = src_row[q];
                        const size_t base =
                            ((size_t)(r >> 7) * p.k64 + 4 * kb) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const bool live = row_ok[q] && kk < nk &&
                                              in_span(NV4_SITE(0), p.sp_sfa, p.sfa + base + kk * 512, 4);
                            cp_async_4(sSFA + kk * 512 + lane * 16 + q * 4, p.sfa + (live ? base + kk * 512 : 0),
                                       live ? 4u : 0u);
                        }
                    }
                    // each lane's gathers complete the stage's barriers on
                    // their own; the consumers fence before the tensor core reads
                    cp_async_arrive_noinc(&sf_full[stage]);
                    if (indexed)
                        cp_async_arrive_noinc(&full[stage]);
                }
                if (++stage == C::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        // every gather of this warp lands before the CTA exits
        cp_async_wait_all();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <int BN, bool GROUPED, int AR = BM>
cudaError_t launch(const Params &p, int grid_units, cudaStream_t stream)
{
    using C = Cfg<BN, AR>;
    auto kern = w4a4_kernel<BN, GROUPED, AR>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess)
        return e;
    const int grid = std::max(1, std::min(grid_units, device_sm_count()));
    if (!GROUPED)
        return launch_pdl(kern, grid, THREADS, C::SMEM_BYTES, stream, p);
    kern<<<grid, THREADS, C::SMEM_BYTES, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t dispatch(int bn, bool grouped, const Params &p, int grid_units, cudaStream_t stream)
{
    if (grouped)
        return bn == 256 ? launch<256, true>(p, grid_units, stream) : launch<128, true>(p, grid_units, stream);
    if (p.a_box_rows <= 16)
        return bn == 256 ? launch<256, false, 16>(p, grid_units, stream)
                         : launch<128, false, 16>(p, grid_units, stream);
    return bn == 256 ? launch<256, false>(p, grid_units, stream) : launch<128, false>(p, grid_units, stream);
}

// Band of M-tiles that run together: every M-tile when the quantised
// activations fit comfortably in L2 (each weight tile then streams from HBM
// once), else 8.
int group_m_for(int64_t m_tiles, int64_t K)
{
    const int64_t a_bytes = m_tiles * 128 * (K / 2 + K / 16);
    if (a_bytes <= ((int64_t)48 << 20))
        return (int)std::max<int64_t>(1, m_tiles);
    return (int)std::min<int64_t>(8, m_tiles);
}

} // namespace

// N-side tile width: 256 when N fills it (every weight tile starts on a scale
// atom), 128 for narrow N.
int w4a4_dense_bn(int64_t b_rows)
{
    if (b_rows <= 128 || (b_rows % 256 != 0 && b_rows < 1024))
        return 128;
    return 256;
}

StreamKPlan w4a4_streamk_plan(int64_t M, int64_t N, int64_t K, int sms)
{
    StreamKPlan pl;
    if (M <= 0 || N <= 0 || K <= 0 || sms <= 0)
        return pl;
    const int bn = w4a4_dense_bn(N);
    const int64_t tiles = ceil_div(M, BM) * ceil_div(N, bn);
    const int64_t kstages = ceil_div(ceil_div(K, 64), 4);
    // M <= 128 is bound by streaming the weights.  Measured on B300 (M = 8 to
    // 128, K = 8192): 112 whole tiles of N = 28672 already keep HBM busy and
    // beat stream-K at every M (its partial reduction only adds a tail),
    // while 16 tiles (N = 4096) leave most SMs idle and stream-K is 1.5x
    // faster.  So stream-K only when the tiles cover under 60% of the SMs and
    // there is enough K to share.  Several M tiles (compute-bound) run whole
    // tiles: measured on [2048, 4096] x [4096, 4096] (256 tiles, 1.73 waves),
    // stream-K took 41 us against 33 us for whole tiles of the wider [2048,
    // 4352] x [4096, 4352] (272 tiles), its FP32 partial tiles (128 KB per
    // CTA) moving through L2 at ~30-60 GB/s per SM, far more than the part
    // of a wave it saves.
    if (M > BM || !(tiles * 10 < 6 * (int64_t)sms && tiles * kstages >= 2 * (int64_t)sms))
        return pl;
    pl.used = true;
    pl.grid = (int)std::min<int64_t>(tiles * kstages, sms);
    pl.slot_bytes = align_up((size_t)pl.grid * (size_t)std::min<int64_t>(M, BM) * (size_t)bn * 4, 256);
    pl.flag_bytes = align_up((size_t)pl.grid * 4, 256);
    return pl;
}

cudaError_t launch_w4a4_dense(const DenseGemmArgs &g, cudaStream_t stream)
{
    Params p{};
    const int64_t k64 = g.K / 64;
    const int sms = device_sm_count();
    const int bn = w4a4_dense_bn(g.b_rows);
    const int64_t m_tiles = ceil_div(g.a_rows, BM);
    const int64_t n_tiles = ceil_div(g.b_rows, bn);
    const int64_t kstages = ceil_div(k64, 4);
    p.m_tiles = (int)m_tiles;
    p.n_tiles = (int)n_tiles;
    p.k64 = (int)k64;
    p.kstages = (int)kstages;
    p.group_m = group_m_for(m_tiles, g.K);
    p.streamk = g.streamk ? 1 : 0;
    // a single M-tile of fewer than 128 rows loads only its rows (rounded
    // up to 16); the MMA still reads 128 rows, and the rows past the box
    // only feed output rows that are never stored
    p.a_box_rows = g.a_rows < BM ? (int)ceil_div(g.a_rows, 16) * 16 : BM;
    CUresult r = make_tmap_2d_u8(&p.tmap_a, g.a_codes, (uint64_t)(g.K / 2), (uint64_t)g.a_rows,
                                 (uint64_t)(g.K / 2), STAGE_K_BYTES, (uint32_t)p.a_box_rows, true);
    if (r != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    r = make_tmap_2d_u8(&p.tmap_b, g.b_codes, (uint64_t)(g.K / 2), (uint64_t)g.b_rows, (uint64_t)(g.K / 2),
                        STAGE_K_BYTES, (uint32_t)bn, true);
    if (r != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    r = make_tmap_scale_atoms(&p.tmap_sfb, g.b_scales, (uint64_t)ceil_div(g.b_rows, 128), (uint64_t)k64, 4,
                              (uint32_t)(bn / 128));
    if (r != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    p.a_codes = g.a_codes;
    p.sfa = g.a_scales;
    p.sfb = g.b_scales;
    p.a_second = g.a_second;
    p.b_second = g.b_second;
    p.out = g.out;
    p.ld_i = g.ld_i;
    p.ld_j = g.ld_j;
    p.a_rows = g.a_rows;
    p.b_rows = g.b_rows;
    p.out_dtype = g.out_dtype;
    p.b_early = g.b_early ? 1 : 0;
    p.diag_skip_flag = g.diag_skip_flag;
    p.out_q = g.yq_codes != nullptr ? 1 : 0;
    p.yq_codes = g.yq_codes;
    p.yq_scales = g.yq_scales;
    p.yq_scale = g.yq_scale;
    p.yq_amax = g.yq_amax;
    p.yq_n = g.b_rows;
    p.slots = g.slots;
    p.flags = g.flags;
    p.slot_stride = std::min<int64_t>(g.a_rows, BM) * bn; // rows of one M tile
    const int esz = g.out_dtype == NVFP4_OUT_BF16 ? 2 : 4;
    p.vec_ok = out_vec_level(g.out, g.ld_i, g.ld_j, esz);
    p.b_row_tiles = (int)ceil_div(g.b_rows, 128);
    p.offsets = nullptr;
    p.row_idx = nullptr;
    p.E = 0;
    p.status = g.status;
    p.timeout_ns = g.timeout_ns;
    const int tiles = p.m_tiles * p.n_tiles;
    // stream-K: one CTA per SM over all (tile, stage) units
    const int grid_units = g.streamk ? (int)std::min<int64_t>((int64_t)tiles * kstages, sms) : tiles;
    p.sp_a_codes = span_of(g.a_codes, (uint64_t)g.a_rows * (uint64_t)(g.K / 2));
    p.sp_sfa = span_of(g.a_scales, tiled_scale_bytes(g.a_rows, g.K));
    p.sp_sfb = span_of(g.b_scales, tiled_scale_bytes(g.b_rows, g.K));
    p.sp_b_second = span_of(g.b_second, 4);
    p.sp_out = span_of(g.out, g.a_rows > 0 && g.b_rows > 0
                                  ? (uint64_t)((g.a_rows - 1) * g.ld_i + (g.b_rows - 1) * g.ld_j + 1) * esz
                                  : 0u);
    if (g.streamk) {
        p.sp_slots = span_of(g.slots, (uint64_t)grid_units * (uint64_t)p.slot_stride * 4u);
        p.sp_flags = span_of(g.flags, (uint64_t)grid_units * 4u);
    }
    p.sp_yq_codes = span_of(g.yq_codes, (uint64_t)g.a_rows * (uint64_t)(g.b_rows / 2));
    p.sp_yq_scales = span_of(g.yq_scales, tiled_scale_bytes(g.a_rows, g.b_rows));
    return dispatch(bn, false, p, grid_units, stream);
}

cudaError_t launch_w4a4_grouped(const GroupedGemmArgs &g, cudaStream_t stream)
{
    Params p{};
    const int64_t k64 = g.K / 64;
    const int bn = (g.N % 256 == 0) ? 256 : 128;
    p.m_tiles = 0;
    p.n_tiles = (int)(g.N / bn);
    p.k64 = (int)k64;
    p.kstages = (int)ceil_div(k64, 4);
    p.streamk = 0;
    p.group_m = 1;
    p.a_box_rows = BM;
    CUresult r = make_tmap_2d_u8(&p.tmap_a, g.a_codes, (uint64_t)(g.K / 2), (uint64_t)g.a_rows,
                                 (uint64_t)(g.K / 2), STAGE_K_BYTES, BM, true);
    if (r != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    r = make_tmap_2d_u8(&p.tmap_b, g.w_codes, (uint64_t)(g.K / 2), (uint64_t)(g.E * g.N), (uint64_t)(g.K / 2),
                        STAGE_K_BYTES, (uint32_t)bn, true);
    if (r != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    r = make_tmap_scale_atoms(&p.tmap_sfb, g.w_scales, (uint64_t)ceil_div(g.E * g.N, 128), (uint64_t)k64, 4,
                              (uint32_t)(bn / 128));
    if (r != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    p.a_codes = g.a_codes;
    p.sfa = g.a_scales;
    p.sfb = g.w_scales;
    p.a_second = g.a_second;
    p.b_second = g.w_second;
    p.out = g.out;
    p.ld_i = g.ldy;
    p.ld_j = 1;
    p.a_rows = g.a_rows;
    p.b_rows = g.N;
    p.out_dtype = g.out_dtype;
    const int esz = g.out_dtype == NVFP4_OUT_BF16 ? 2 : 4;
    p.vec_ok = out_vec_level(g.out, g.ldy, 1, esz);
    p.b_row_tiles = (int)ceil_div(g.E * g.N, 128);
    p.diag_skip_flag = -1;
    p.epi = g.epi;
    p.comb_idx = g.comb_idx;
    p.comb_w = g.comb_w;
    p.comb_rows = g.comb_rows;
    p.out_q = g.yq_codes != nullptr ? 1 : 0;
    p.yq_codes = g.yq_codes;
    p.yq_scales = g.yq_scales;
    p.yq_scale = g.yq_scale;
    p.yq_amax = g.yq_amax;
    p.yq_n = g.N / 2; // SwiGLU output columns
    p.offsets = g.offsets;
    p.row_idx = g.row_idx;
    p.E = g.E;
    p.total_rows = g.total_rows;
    p.status = g.status;
    p.timeout_ns = g.timeout_ns;
    p.sp_a_codes = span_of(g.a_codes, (uint64_t)g.a_rows * (uint64_t)(g.K / 2));
    p.sp_sfa = span_of(g.a_scales, tiled_scale_bytes(g.a_rows, g.K));
    p.sp_sfb = span_of(g.w_scales, tiled_scale_bytes(g.E * g.N, g.K));
    p.sp_b_second = span_of(g.w_second, 4u * (uint64_t)g.E);
    const int64_t out_cols = g.epi == EPI_SWIGLU ? g.N / 2 : g.N;
    const int64_t out_rows = g.epi == EPI_COMBINE ? g.comb_rows : g.total_rows;
    p.sp_out = span_of(g.out, matrix_bytes(out_rows, out_cols, g.ldy, g.epi == EPI_COMBINE ? 4 : esz));
    p.sp_yq_codes = span_of(g.yq_codes, (uint64_t)g.total_rows * (uint64_t)(g.N / 4));
    p.sp_yq_scales = span_of(g.yq_scales, tiled_scale_bytes(g.total_rows, g.N / 2));
    p.sp_comb_idx = span_of(g.comb_idx, 4u * (uint64_t)g.total_rows);
    p.sp_comb_w = span_of(g.comb_w, 4u * (uint64_t)g.total_rows);
    p.sp_offsets = span_of(g.offsets, 8u * (uint64_t)(g.E + 1));
    p.sp_row_idx = span_of(g.row_idx, 4u * (uint64_t)g.total_rows);
    // upper bound of items: every expert's rows in tiles of 128, plus one partial tile per expert
    const int64_t max_tiles = ceil_div(g.total_rows, BM) + g.E;
    const int total = (int)std::min<int64_t>(max_tiles * p.n_tiles, 1 << 30);
    return dispatch(bn, true, p, total, stream);
}

} // namespace nv4
