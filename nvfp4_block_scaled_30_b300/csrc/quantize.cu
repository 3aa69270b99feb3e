// Quantisers on the NVFP4 hot path.
//
// NVFP4 encode follows "NVIDIA Ships TensorRT-LLM 0.16: Native FP4
// Quantization for Blackwell B200", section "The Mathematical Breakthrough of
// Microscopic FP4 Scaling", item 2 "Two-Level Block Scaling": one E4M3 scale
// per 16 consecutive elements and a second level that is either one FP32
// tensor scale (amax / (6 * 448)) or one FP16 macro-scale per 16 micro-vectors
// (256 elements).  Per-token FP8 encode serves the W4A8 route of "llama.cpp
// Put Precision Policy Inside the Model. That Matters More Than W4A4",
// section "One model can need more than one precision".
//
// All encode arithmetic is IEEE binary32 with explicit round-to-nearest
// intrinsics, in this order per 16-element block:
//   t = amax_b / 6, u = t / s, e = E4M3(u) (0 when s == 0), d = e * s,
//   r = 1 / d (0 when d == 0, at most FLT_MAX), code = E2M1(x * r).
//
// Memory: each thread owns 8 consecutive BF16 values per 16-byte load and
// keeps several loads in flight; a lane pair owns one 16-element block
// (absmax by one shfl.xor); the pair writes 8 packed code bytes (one 32-bit
// store each) and one scale byte.  Activations of up to 262144 values take a
// single-launch path on one thread-block cluster (amax exchanged through
// distributed shared memory); larger tensors take two streaming passes.
#include <cfloat>
#include <mutex>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace nv4 {

namespace {

constexpr int QT = 256; // threads per quantiser CTA
constexpr unsigned FULL = 0xFFFFFFFFu;

// The bytes a quantiser call's arguments grant each tensor (tested before
// each plain access in the bounds-checked build): x, codes (FP8 values for
// the per-token quantiser), scales (s_t), the second-level scale or macro
// scales, and the partial maxima.
struct QuantSpans {
    Span x, codes, scales, second, partial;
};

__device__ __forceinline__ void bf16x8(const uint16_t *p, float (&f)[8])
{
    uint4 v = __ldg(reinterpret_cast<const uint4 *>(p));
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ uint32_t block_max_u32(uint32_t v, uint32_t *red)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = max(v, __shfl_xor_sync(FULL, v, o));
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0)
        red[w] = v;
    __syncthreads();
    uint32_t r = 0;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i)
        r = max(r, red[i]);
    __syncthreads();
    return r;
}



// 8 values times r -> 4 packed E2M1 bytes (element 0 in the lowest nibble).
__device__ __forceinline__ uint32_t pack8(const float (&f)[8], float r)
{
    return e2m1x8(__fmul_rn(f[0], r), __fmul_rn(f[1], r), __fmul_rn(f[2], r), __fmul_rn(f[3], r),
                  __fmul_rn(f[4], r), __fmul_rn(f[5], r), __fmul_rn(f[6], r), __fmul_rn(f[7], r));
}

__device__ __forceinline__ size_t scale_offset(int64_t row, int64_t blk, int64_t K, bool tiled)
{
    if (!tiled)
        return (size_t)(row * (K / 16) + blk);
    int64_t r = row & 127;
    return (size_t)(((row >> 7) * (K / 64) + (blk >> 2)) * 512 + (r & 31) * 16 + (r >> 5) * 4 + (blk & 3));
}

// Loads in flight per thread in the streaming passes.
constexpr int QU = 4;

// Position (row, chunk) in a rows x cpr grid of 8-value chunks, advanced by
// a fixed flat step without dividing: step = q * cpr + r with r < cpr.
struct Cursor {
    int64_t row, j;
};

__device__ __forceinline__ void cursor_advance(Cursor &c, int64_t q, int64_t r, int64_t cpr)
{
    c.j += r;
    c.row += q;
    if (c.j >= cpr) {
        c.j -= cpr;
        ++c.row;
    }
}

__device__ __forceinline__ void bf16x8_of(const uint4 v, float (&f)[8])
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ void absmax_bits(const uint4 v, uint32_t &m, uint32_t &bad)
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t lo = w[i] & 0x7FFFu, hi = (w[i] >> 16) & 0x7FFFu;
        bad |= (lo >= 0x7F80u) | (hi >= 0x7F80u);
        m = max(m, max(lo, hi));
    }
}

// Zero scales of the tiled layout's padding rows rows..rows_pad: one 32-bit
// word = one row's 4 scales of a 64-element chunk.
__device__ __forceinline__ void zero_pad_scales(uint8_t *scales, int64_t rows, int64_t rows_pad, int64_t K,
                                                int64_t first, int64_t stride, const QuantSpans &sp)
{
    // fewer than 128 padding rows: 32-bit index arithmetic suffices
    const uint32_t k64 = (uint32_t)(K / 64);
    const uint32_t pad = (uint32_t)(rows_pad - rows) * k64;
    const int64_t tile0 = rows >> 7; // the padding rows all lie in the last 128-row tile
    for (int64_t i = first; i < (int64_t)pad; i += stride) {
        const uint32_t q = (uint32_t)i / k64, c = (uint32_t)i - q * k64;
        const uint32_t r = (uint32_t)(rows & 127) + q;
        const size_t off = ((size_t)tile0 * k64 + c) * 512 + (r & 31) * 16 + (r >> 5) * 4;
        if (in_span(NV4_SITE(0), sp.scales, scales + off, 4))
            *reinterpret_cast<uint32_t *>(scales + off) = 0u;
    }
}

// One 16-element block (a lane pair, both lanes live) of tensor-scale encode:
// codes and scale of chunk (row, j) of f under second-level scale sg.
template <bool TILED>
__device__ __forceinline__ void encode_chunk(const float (&f)[8], bool real, int64_t row, int64_t j, int64_t K,
                                             float sg, uint8_t *codes, uint8_t *scales, const QuantSpans &sp)
{
    float am = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        am = fmaxf(am, fabsf(f[i]));
    const float amb = fmaxf(am, __shfl_xor_sync(FULL, am, 1));
    const uint32_t e = real ? block_scale_code(amb, sg) : 0u;
    const float r = recip_step(__fmul_rn(e4m3_value(e), sg));
    if (real) {
        const uint32_t pk = pack8(f, r);
        if (in_span(NV4_SITE(0), sp.codes, codes + row * (K / 2) + j * 4, 4))
            *reinterpret_cast<uint32_t *>(codes + row * (K / 2) + j * 4) = pk;
        if ((threadIdx.x & 1) == 0 && in_span(NV4_SITE(0), sp.scales, scales + scale_offset(row, j >> 1, K, TILED), 1))
            scales[scale_offset(row, j >> 1, K, TILED)] = (uint8_t)e;
    }
}

// Blocks in flight per thread in the two-pass encode.
constexpr int QB = 2;

// One whole 16-element block (16 BF16 values in 8 words) by one thread: the
// block maximum from the magnitude bits (exact, equal to the float maximum
// of finite values), the same scale and code arithmetic as encode_chunk, and
// one 8-byte code store plus one scale byte.
template <bool TILED>
__device__ __forceinline__ void encode_block16(const uint32_t (&w)[8], int64_t row, int64_t blk, int64_t K, float sg,
                                               uint8_t *codes, uint8_t *scales, const QuantSpans &sp)
{
    uint32_t pk[2];
    const uint32_t e = encode_bf16_block(w, sg, pk);
    if (in_span(NV4_SITE(0), sp.codes, codes + row * (K / 2) + blk * 8, 8))
        *reinterpret_cast<uint2 *>(codes + row * (K / 2) + blk * 8) = make_uint2(pk[0], pk[1]);
    if (in_span(NV4_SITE(0), sp.scales, scales + scale_offset(row, blk, K, TILED), 1))
        scales[scale_offset(row, blk, K, TILED)] = (uint8_t)e;
}

// One 16-value block (32 bytes) of x.  With V8 the block is 32-byte aligned
// and comes in one 256-bit load; KEEP asks L2 to keep it (the amax pass:
// the encode pass reads x again) and !KEEP marks its last use.  Without V8
// two 16-byte loads.
template <bool V8, bool KEEP>
__device__ __forceinline__ void load_block16(const uint16_t *p, uint32_t (&w)[8])
{
    if (V8) {
        if (KEEP)
            asm volatile("ld.global.nc.L1::no_allocate.L2::evict_last.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                         : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]),
                           "=r"(w[7])
                         : "l"(p));
        else
            asm volatile("ld.global.nc.L1::no_allocate.L2::evict_first.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                         : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]),
                           "=r"(w[7])
                         : "l"(p));
    } else {
        const uint4 a = __ldg(reinterpret_cast<const uint4 *>(p));
        const uint4 b = __ldg(reinterpret_cast<const uint4 *>(p) + 1);
        w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
        w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
    }
}

// Pass 1: per-CTA maximum of |x| (as BF16 magnitude bits) and a non-finite
// flag.  The rows x K/16 blocks of 16 values are one flat index space, so
// small row counts still spread over many CTAs; each thread keeps QU block
// loads in flight and walks the index space with a cursor (no division per
// block).  Loads ask L2 to keep x for the encode pass.
template <bool V8>
__global__ void __launch_bounds__(QT) amax_partial_kernel(const uint16_t *__restrict__ x, int64_t rows, int64_t K,
                                                          int64_t ldx, uint32_t *__restrict__ partial,
                                                          uint32_t *__restrict__ status, const QuantSpans sp)
{
    __shared__ uint32_t red[QT / 32];
    // launched as a programmatic dependent: wait for the previous grid (it
    // may still read the buffers this pass and the next one write)
    pdl_wait();
    pdl_trigger();
    const int64_t bpr = K / 16;
    const int64_t total = rows * bpr;
    const int64_t base0 = (int64_t)blockIdx.x * QT * QU + threadIdx.x;
    const int64_t stride = (int64_t)gridDim.x * QT * QU;
    Cursor cur{base0 / bpr, base0 % bpr};
    const int64_t qs = QT / bpr, rs = QT % bpr, qi = stride / bpr, ri = stride % bpr;
    uint32_t m2 = 0, bad = 0; // m2: two 16-bit magnitude maxima
    for (int64_t base = base0; base < total; base += stride) {
        uint32_t w[QU][8];
        Cursor c = cur;
#pragma unroll
        for (int u = 0; u < QU; ++u) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                w[u][i] = 0u;
            if (base + (int64_t)u * QT < total && in_span(NV4_SITE(0), sp.x, x + c.row * ldx + c.j * 16, 32))
                load_block16<V8, true>(x + c.row * ldx + c.j * 16, w[u]);
            cursor_advance(c, qs, rs, bpr);
        }
#pragma unroll
        for (int u = 0; u < QU; ++u)
#pragma unroll
            for (int i = 0; i < 8; ++i)
                m2 = __vmaxu2(m2, w[u][i] & 0x7FFF7FFFu);
        cursor_advance(cur, qi, ri, bpr);
    }
    const uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
    // a non-finite value has the largest magnitude bits (>= 0x7F80)
    bad = __any_sync(FULL, m >= 0x7F80u);
    uint32_t bm = block_max_u32(m, red);
    if (threadIdx.x == 0 && in_span(NV4_SITE(0), sp.partial, partial + blockIdx.x, 4))
        partial[blockIdx.x] = bm;
    if (bad && (threadIdx.x & 31) == 0)
        atomicOr(status, ST_NONFINITE);
}

// Pass 2, tensor-scale mode.  Every CTA reduces the partial maxima itself,
// so no extra launch or host synchronisation is needed.  The real rows' chunks
// form one flat index space (a lane pair = one 16-element block, never split
// across rows since K/8 is even); the padding rows rows..rows_pad of the tiled
// layout only get zero scales, written by a separate loop.
template <bool TILED, bool V8>
__global__ void __launch_bounds__(QT) nvfp4_encode_kernel(const uint16_t *__restrict__ x, int64_t rows,
                                                          int64_t rows_pad, int64_t K, int64_t ldx,
                                                          uint8_t *__restrict__ codes, uint8_t *__restrict__ scales,
                                                          float *__restrict__ sg_out,
                                                          const uint32_t *__restrict__ partial, int n_partial,
                                                          int zero_pad, const QuantSpans sp)
{
    __shared__ uint32_t red[QT / 32];
    pdl_wait(); // the partial maxima of pass 1
    pdl_trigger();
    uint32_t m = 0;
    for (int i = threadIdx.x; i < n_partial; i += QT)
        if (in_span(NV4_SITE(0), sp.partial, partial + i, 4))
            m = max(m, partial[i]);
    const float amax = __uint_as_float(block_max_u32(m, red) << 16);
    const float sg = __fdiv_rn(amax, 2688.0f);
    if (blockIdx.x == 0 && threadIdx.x == 0 && in_span(NV4_SITE(0), sp.second, sg_out, 4))
        *sg_out = sg;

    // one thread per 16-element block (two 16-byte loads), QB blocks in
    // flight per thread; blocks of all real rows form one flat index space
    const int64_t bpr = K / 16;
    const int64_t total = rows * bpr;
    const int64_t base0 = (int64_t)blockIdx.x * QT * QB + threadIdx.x;
    const int64_t stride = (int64_t)gridDim.x * QT * QB;
    Cursor cur{base0 / bpr, base0 % bpr};
    const int64_t qs = QT / bpr, rs = QT % bpr, qi = stride / bpr, ri = stride % bpr;
    for (int64_t base = base0; base < total; base += stride) {
        uint32_t v[QB][8];
        Cursor c[QB];
        c[0] = cur;
#pragma unroll
        for (int u = 0; u < QB; ++u) {
            if (u > 0) {
                c[u] = c[u - 1];
                cursor_advance(c[u], qs, rs, bpr);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i)
                v[u][i] = 0u;
            if (base + (int64_t)u * QT < total && in_span(NV4_SITE(0), sp.x, x + c[u].row * ldx + c[u].j * 16, 32))
                load_block16<V8, false>(x + c[u].row * ldx + c[u].j * 16, v[u]);
        }
#pragma unroll
        for (int u = 0; u < QB; ++u) {
            if (base + (int64_t)u * QT >= total)
                continue;
            encode_block16<TILED>(v[u], c[u].row, c[u].j, K, sg, codes, scales, sp);
        }
        cursor_advance(cur, qi, ri, bpr);
    }
    if (TILED && zero_pad)
        zero_pad_scales(scales, rows, rows_pad, K, (int64_t)blockIdx.x * QT + threadIdx.x, (int64_t)gridDim.x * QT,
                        sp);
}

// ---- staged streaming passes (contiguous x) ----------------------------------
// x (ldx == K) is one flat run of 16-element blocks cut into units of SU_BLOCKS
// blocks (SU_BYTES bytes).  One producer thread brings each unit into a
// SU_STAGES-deep shared-memory ring with a single bulk copy carrying an L2
// hint (pass 1 asks L2 to keep x, pass 2 marks its last use); 8 consumer
// warps work from the ring, so the bytes in flight per SM are the ring's,
// independent of the consumers' arithmetic.
constexpr int SU_CONSUMERS = 256;
constexpr int SU_BPT = 2;                          // blocks per consumer thread and unit
constexpr int SU_BLOCKS = SU_CONSUMERS * SU_BPT;   // 512 blocks
constexpr int SU_BYTES = SU_BLOCKS * 32;           // 16 KB
constexpr int SU_THREADS = SU_CONSUMERS + 32;      // + the producer warp
// pass 1 streams x from HBM: a deep ring, 3 CTAs per SM; pass 2 normally
// finds x in L2 and is arithmetic-heavy: a short ring, and one wave of the
// 4 CTAs per SM its registers allow (measured: a grid of 6 per SM ran as
// 1.5 waves and was 2 % slower; capping registers for 5 per SM, 8 % slower)
constexpr int SU_STAGES_1 = 4, SU_CTAS_1 = 3;
constexpr int SU_STAGES_2 = 2, SU_CTAS_2 = 4;
constexpr int su_smem(int stages) { return stages * SU_BYTES + 2 * stages * 8 + 16; }

__device__ __forceinline__ void bulk_load_hint(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                               uint64_t policy)
{
    if (!(in_dyn_smem(NV4_SITE(0), smem_u32(dst), bytes) && aligned_to(NV4_SITE(0), smem_u32(dst), 16) &&
          aligned_to(NV4_SITE(0), reinterpret_cast<uint64_t>(src), 16) && aligned_to(NV4_SITE(0), bytes, 16)))
        return;
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, "
                 "[%3], %4;" ::"r"(smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
                 : "memory");
}

template <bool KEEP>
__device__ __forceinline__ uint64_t l2_policy()
{
    uint64_t pol;
    if (KEEP)
        asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    else
        asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Named barrier 1 over the consumer warps only.
__device__ __forceinline__ void consumers_sync()
{
    asm volatile("bar.sync 1, %0;" ::"n"(SU_CONSUMERS) : "memory");
}

__device__ __forceinline__ uint32_t consumers_max(uint32_t v, uint32_t *red)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = max(v, __shfl_xor_sync(FULL, v, o));
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = v;
    consumers_sync();
    uint32_t r = 0;
#pragma unroll
    for (int i = 0; i < SU_CONSUMERS / 32; ++i)
        r = max(r, red[i]);
    consumers_sync();
    return r;
}

// The block scale code of a block whose |x| maximum has BF16 magnitude bits
// mb, from a per-CTA table: for amax = (1 + i/128) * 2^k the quantisers'
// u = RN(RN(amax / 6) / s) equals U[i] * 2^k with U[i] = RN(RN((1 + i/128)
// / 6) / s) whenever RN(amax / 6) and u are normal binary32 numbers (round to
// nearest commutes with exact power-of-two scaling), and any u below the
// normal range gives code 0 either way, as an overflow gives 448 either way.
// So when s lies in [2^-100, 2^100] (U normal) and amax >= 2^-123 (amax / 6
// normal) the code is e4m3(U[i] * 2^k), bit-identical to block_scale_code;
// other blocks take block_scale_code itself.
__device__ __forceinline__ uint32_t scale_code_tab(uint32_t mb, float sg, bool fast, const float *tab_u)
{
    const uint32_t eb = mb >> 7;
    if (fast && eb >= 4u)
        return e4m3(__fmul_rn(tab_u[mb & 127u], __uint_as_float(eb << 23)));
    return block_scale_code(__uint_as_float(mb << 16), sg);
}

// PASS 1: per-CTA maximum of |x| magnitude bits into partial[blockIdx.x] and
// the non-finite flag.  PASS 2: tensor scale from the partial maxima, then
// the block encode of every block (and zero scales for the tiled padding
// rows when zero_pad).  Units go to CTAs round robin.
template <int PASS, bool TILED, int SU_STAGES>
__global__ void __launch_bounds__(SU_THREADS) stream_quant_kernel(const uint16_t *__restrict__ x, int64_t rows,
                                                                  int64_t rows_pad, int64_t K,
                                                                  uint8_t *__restrict__ codes,
                                                                  uint8_t *__restrict__ scales,
                                                                  float *__restrict__ sg_out,
                                                                  uint32_t *__restrict__ partial, int n_partial,
                                                                  int zero_pad, uint32_t *__restrict__ status,
                                                                  uint64_t timeout_ns, const QuantSpans sp)
{
    extern __shared__ __align__(128) uint8_t sq[];
    uint64_t *full = reinterpret_cast<uint64_t *>(sq + SU_STAGES * SU_BYTES);
    uint64_t *empty = full + SU_STAGES;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + SU_STAGES);
    __shared__ uint32_t red[SU_CONSUMERS / 32];
    __shared__ float tab_u[PASS == 2 ? 128 : 1]; // scale_code_tab's U
    __shared__ float tab_r[PASS == 2 ? 128 : 1]; // reciprocal step of every scale code
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < SU_STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], SU_CONSUMERS / 32);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    // a programmatic dependent: wait for the previous grid before touching
    // memory it may use (pass 2: the partial maxima of pass 1)
    pdl_wait();
    pdl_trigger();
    const int64_t bpr = K / 16;
    const int64_t total = rows * bpr;
    const int64_t units = (total + SU_BLOCKS - 1) / SU_BLOCKS;

    if (warp == SU_CONSUMERS / 32) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            const uint64_t pol = l2_policy<PASS == 1>();
            int s = 0, issued = 0;
            uint32_t ph = 0;
            for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
                if (!mbar_wait(&empty[s], ph ^ 1u, timeout_ns, abort_flag)) {
                    *abort_flag = 1;
                    atomicOr(status, ST_TIMEOUT);
                    break;
                }
                const int64_t nb = min((int64_t)SU_BLOCKS, total - u * SU_BLOCKS);
                mbar_arrive_expect_tx(&full[s], (uint32_t)(nb * 32));
                if (in_span(NV4_SITE(0), sp.x, x + u * SU_BLOCKS * 16, (uint64_t)(nb * 32)))
                    bulk_load_hint(sq + s * SU_BYTES, x + u * SU_BLOCKS * 16, (uint32_t)(nb * 32), &full[s], pol);
                ++issued;
                if (++s == SU_STAGES) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            // every copy issued lands before the CTA exits
            for (int q = 0; q < min(issued, SU_STAGES); ++q) {
                if (--s < 0) {
                    s = SU_STAGES - 1;
                    ph ^= 1u;
                }
                mbar_wait(&full[s], ph, timeout_ns, nullptr);
            }
        }
        return;
    }

    // -------------------------------------------------------------- consumers
    const int t = threadIdx.x;
    float sg = 0.0f;
    bool fast = false;
    if (PASS == 2) {
        uint32_t m = 0;
        for (int i = t; i < n_partial; i += SU_CONSUMERS)
            if (in_span(NV4_SITE(0), sp.partial, partial + i, 4))
                m = max(m, partial[i]);
        const float amax = __uint_as_float(consumers_max(m, red) << 16);
        sg = __fdiv_rn(amax, 2688.0f);
        if (blockIdx.x == 0 && t == 0 && in_span(NV4_SITE(0), sp.second, sg_out, 4))
            *sg_out = sg;
        fast = sg >= 0x1p-100f && sg <= 0x1p100f;
        if (t < 128) {
            if (fast)
                tab_u[t] = __fdiv_rn(__fdiv_rn(1.0f + (float)t * 0.0078125f, 6.0f), sg);
            // codes 0x00..0x7E are all a non-negative saturating conversion gives
            tab_r[t] = recip_step(__fmul_rn(e4m3_value(t < 127 ? (uint32_t)t : 0u), sg));
        }
        consumers_sync();
    }
    // block b = u * SU_BLOCKS + k * SU_CONSUMERS + t of unit u, k < SU_BPT:
    // (row, block-in-row) cursors advanced by the round-robin unit step
    Cursor cur[SU_BPT];
#pragma unroll
    for (int k = 0; k < SU_BPT; ++k) {
        const int64_t b0 = (int64_t)blockIdx.x * SU_BLOCKS + k * SU_CONSUMERS + t;
        cur[k] = Cursor{b0 / bpr, b0 % bpr};
    }
    const int64_t step = (int64_t)gridDim.x * SU_BLOCKS;
    const int64_t qi = step / bpr, ri = step % bpr;
    uint32_t m2 = 0;
    int s = 0;
    uint32_t ph = 0;
    for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
        const bool got = mbar_wait(&full[s], ph, timeout_ns, abort_flag);
        if (!__all_sync(FULL, got)) {
            if (lane == 0) {
                *abort_flag = 1;
                atomicOr(status, ST_TIMEOUT);
            }
            break;
        }
        const uint8_t *src = sq + s * SU_BYTES;
#pragma unroll
        for (int k = 0; k < SU_BPT; ++k) {
            const int slot = k * SU_CONSUMERS + t;
            if (u * SU_BLOCKS + slot < total) {
                const uint4 a = *reinterpret_cast<const uint4 *>(src + slot * 32);
                const uint4 b = *reinterpret_cast<const uint4 *>(src + slot * 32 + 16);
                const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
                if (PASS == 1) {
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        m2 = __vmaxu2(m2, w[i] & 0x7FFF7FFFu);
                } else {
                    uint32_t mb2 = 0;
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        mb2 = __vmaxu2(mb2, w[i] & 0x7FFF7FFFu);
                    const uint32_t e = scale_code_tab(max(mb2 & 0xFFFFu, mb2 >> 16), sg, fast, tab_u);
                    const float r = tab_r[e];
                    uint32_t pk[2];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        float q[8];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const uint32_t ww = w[4 * h + i];
                            mul2_rn(__uint_as_float(ww << 16), __uint_as_float(ww & 0xFFFF0000u), r, q[2 * i],
                                    q[2 * i + 1]);
                        }
                        pk[h] = e2m1x8(q[0], q[1], q[2], q[3], q[4], q[5], q[6], q[7]);
                    }
                    // codes are contiguous: block b's 8 bytes sit at 8 b
                    const int64_t b = u * SU_BLOCKS + slot;
                    if (in_span(NV4_SITE(0), sp.codes, codes + b * 8, 8))
                        *reinterpret_cast<uint2 *>(codes + b * 8) = make_uint2(pk[0], pk[1]);
                    const size_t so = TILED ? scale_offset(cur[k].row, cur[k].j, K, true) : (size_t)b;
                    if (in_span(NV4_SITE(0), sp.scales, scales + so, 1))
                        scales[so] = (uint8_t)e;
                }
            }
            cursor_advance(cur[k], qi, ri, bpr);
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&empty[s]);
        if (++s == SU_STAGES) {
            s = 0;
            ph ^= 1u;
        }
    }
    if (PASS == 1) {
        const uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
        const bool bad = __any_sync(FULL, m >= 0x7F80u);
        const uint32_t bm = consumers_max(m, red);
        if (t == 0 && in_span(NV4_SITE(0), sp.partial, partial + blockIdx.x, 4))
            partial[blockIdx.x] = bm;
        if (bad && lane == 0)
            atomicOr(status, ST_NONFINITE);
    } else if (TILED && zero_pad) {
        zero_pad_scales(scales, rows, rows_pad, K, (int64_t)blockIdx.x * SU_CONSUMERS + t,
                        (int64_t)gridDim.x * SU_CONSUMERS, sp);
    }
}

// Small activations (decode): one kernel on one thread-block cluster of FC
// CTAs.  Each thread holds up to FQ chunks of x in registers (a warp stops at
// its last real chunk); every CTA pushes its absolute maximum into all CTAs'
// shared memory, one cluster barrier publishes them, and each CTA encodes
// from its registers, so x is read once and there is no second launch.
// A cluster of 16 CTAs (a non-portable size; one chunk per thread at 8 x 8192)
// measured 0.7-1.1 us faster per decode step than 8; 8 is kept for devices
// that cannot hold a 16-CTA cluster.
constexpr int FT = 512;  // threads per CTA
constexpr int64_t FUSED_MAX_CHUNKS = 32768;

template <bool TILED, int FC>
__global__ void __launch_bounds__(FT) nvfp4_encode_small_kernel(const uint16_t *__restrict__ x, int64_t rows,
                                                                int64_t rows_pad, int64_t K, int64_t ldx,
                                                                uint8_t *__restrict__ codes,
                                                                uint8_t *__restrict__ scales,
                                                                float *__restrict__ sg_out,
                                                                uint32_t *__restrict__ status, int zero_pad,
                                                                const QuantSpans sp)
{
    constexpr int FQ = (int)(FUSED_MAX_CHUNKS / (FC * FT)); // chunks per thread
    static_assert(FQ * FC * FT == FUSED_MAX_CHUNKS, "cluster shape");
    __shared__ uint32_t red[FT / 32];
    __shared__ uint32_t cta_max[FC];
    // this CTA is running: peers may write its shared memory once they have
    // waited on this phase
    cluster_arrive_relaxed();
    pdl_wait(); // x may come from the previous grid
    pdl_trigger();
    const uint32_t rank = cluster_ctarank();
    const int cpr = (int)(K / 8);
    const int total = (int)(rows * (K / 8)); // at most FUSED_MAX_CHUNKS
    const int first = (int)rank * FT + (int)threadIdx.x;
    const int wfirst = first - (int)(threadIdx.x & 31);
    constexpr int STEP = FC * FT;
    uint4 v[FQ];
    uint32_t m = 0, bad = 0;
#pragma unroll
    for (int k = 0; k < FQ; ++k) {
        v[k] = make_uint4(0, 0, 0, 0);
        const int idx = first + k * STEP;
        if (idx < total) {
            const int row = idx / cpr, j = idx - row * cpr;
            if (in_span(NV4_SITE(0), sp.x, x + (int64_t)row * ldx + j * 8, 16))
                v[k] = __ldg(reinterpret_cast<const uint4 *>(x + (int64_t)row * ldx + j * 8));
        }
    }
#pragma unroll
    for (int k = 0; k < FQ; ++k)
        absmax_bits(v[k], m, bad);
    if (__any_sync(FULL, bad) && (threadIdx.x & 31) == 0)
        atomicOr(status, ST_NONFINITE);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        m = max(m, __shfl_xor_sync(FULL, m, o));
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = m;
    __syncthreads();
    cluster_wait(); // every CTA of the cluster is running
    if (threadIdx.x < FC) {
        // this CTA's maximum into slot `rank` of every CTA of the cluster
        uint32_t bb = red[0];
#pragma unroll
        for (int w = 1; w < FT / 32; ++w)
            bb = max(bb, red[w]);
        st_dsmem_u32(&cta_max[rank], threadIdx.x, bb);
    }
    cluster_sync_all(); // all maxima are in every CTA; no remote access follows
    uint32_t g = 0;
#pragma unroll
    for (int c = 0; c < FC; ++c)
        g = max(g, cta_max[c]);
    const float amax = __uint_as_float(g << 16);
    const float sg = __fdiv_rn(amax, 2688.0f);
    if (rank == 0 && threadIdx.x == 0 && in_span(NV4_SITE(0), sp.second, sg_out, 4))
        *sg_out = sg;
#pragma unroll
    for (int k = 0; k < FQ; ++k) {
        if (wfirst + k * STEP >= total) // warp-uniform: nothing left for this warp
            break;
        const int idx = first + k * STEP;
        const bool real = idx < total;
        const int row = real ? idx / cpr : 0, j = real ? idx - row * cpr : 0;
        float f[8];
        bf16x8_of(v[k], f);
        encode_chunk<TILED>(f, real, row, j, K, sg, codes, scales, sp);
    }
    if (TILED && zero_pad)
        zero_pad_scales(scales, rows, rows_pad, K, first, STEP, sp);
}

// Macro mode: one warp covers 32 chunks = 256 elements = one macro group (K is
// a multiple of 256 and the chunk loop advances in whole CTAs of 8 warps).
template <bool TILED>
__global__ void __launch_bounds__(QT) nvfp4_encode_macro_kernel(const uint16_t *__restrict__ x, int64_t rows,
                                                                int64_t rows_pad, int64_t K, int64_t ldx,
                                                                uint8_t *__restrict__ codes,
                                                                uint8_t *__restrict__ scales,
                                                                uint16_t *__restrict__ macro,
                                                                uint32_t *__restrict__ status, const QuantSpans sp)
{
    const int64_t cpr = K / 8;
    uint32_t bad = 0;
    for (int64_t row = blockIdx.x; row < rows_pad; row += gridDim.x) {
        const bool real_row = row < rows;
        for (int64_t j0 = 0; j0 < cpr; j0 += QT) {
            const int64_t j = j0 + threadIdx.x;
            const bool valid = j < cpr;
            const bool real = valid && real_row;
            float f[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            if (real && in_span(NV4_SITE(0), sp.x, x + row * ldx + j * 8, 16)) {
                bf16x8(x + row * ldx + j * 8, f);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    bad |= (__float_as_uint(f[i]) & 0x7F800000u) == 0x7F800000u;
            }
            float am = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i)
                am = fmaxf(am, fabsf(f[i]));
            const float amb = fmaxf(am, __shfl_xor_sync(FULL, am, 1));
            float ag = amb;
#pragma unroll
            for (int o = 2; o < 32; o <<= 1)
                ag = fmaxf(ag, __shfl_xor_sync(FULL, ag, o));
            float q = __fdiv_rn(ag, 2688.0f);
            q = fminf(q, 65504.0f);
            const __half h = __float2half_rn(q);
            const float S = __half2float(h);
            const uint32_t e = real ? block_scale_code(amb, S) : 0u;
            const float r = recip_step(__fmul_rn(e4m3_value(e), S));
            if (real) {
                const uint32_t pk = pack8(f, r);
                if (in_span(NV4_SITE(0), sp.codes, codes + row * (K / 2) + j * 4, 4))
                    *reinterpret_cast<uint32_t *>(codes + row * (K / 2) + j * 4) = pk;
                if ((threadIdx.x & 31) == 0 && in_span(NV4_SITE(0), sp.second, macro + row * (K / 256) + (j >> 5), 2))
                    macro[row * (K / 256) + (j >> 5)] = __half_as_ushort(h);
            }
            if (valid && (threadIdx.x & 1) == 0 &&
                in_span(NV4_SITE(0), sp.scales, scales + scale_offset(row, j >> 1, K, TILED), 1))
                scales[scale_offset(row, j >> 1, K, TILED)] = (uint8_t)e;
        }
    }
    if (__any_sync(FULL, bad) && (threadIdx.x & 31) == 0)
        atomicOr(status, ST_NONFINITE);
}

__device__ __forceinline__ uint32_t e4m3_signed(float v)
{
    return (e4m3(v) & 0x7Fu) | ((__float_as_uint(v) >> 31) << 7);
}

// Per-token FP8: one CTA per row (grid-stride); pass 1 finds the row maximum,
// pass 2 (re-reading the row from L1/L2) encodes 8 elements per thread.
__global__ void __launch_bounds__(QT) fp8_token_kernel(const uint16_t *__restrict__ x, int64_t rows, int64_t K,
                                                       int64_t ldx, uint8_t *__restrict__ a,
                                                       float *__restrict__ s_t, uint32_t *__restrict__ status,
                                                       const QuantSpans sp)
{
    __shared__ uint32_t red[QT / 32];
    const int64_t cpr = K / 8;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const uint16_t *xr = x + row * ldx;
        uint32_t m = 0, bad = 0;
        for (int64_t j = threadIdx.x; j < cpr; j += QT) {
            const uint4 v = in_span(NV4_SITE(0), sp.x, xr + j * 8, 16) ? __ldg(reinterpret_cast<const uint4 *>(xr + j * 8))
                                                                       : make_uint4(0u, 0u, 0u, 0u);
            uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint32_t lo = w[i] & 0x7FFFu, hi = (w[i] >> 16) & 0x7FFFu;
                bad |= (lo >= 0x7F80u) | (hi >= 0x7F80u);
                m = max(m, max(lo, hi));
            }
        }
        if (__any_sync(FULL, bad) && (threadIdx.x & 31) == 0)
            atomicOr(status, ST_NONFINITE);
        const float amax = __uint_as_float(block_max_u32(m, red) << 16);
        const float s = __fdiv_rn(amax, 448.0f);
        const float r = recip_step(s);
        if (threadIdx.x == 0 && in_span(NV4_SITE(0), sp.scales, s_t + row, 4))
            s_t[row] = s;
        for (int64_t j = threadIdx.x; j < cpr; j += QT) {
            float f[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            if (in_span(NV4_SITE(0), sp.x, xr + j * 8, 16))
                bf16x8(xr + j * 8, f);
            uint32_t lo = 0, hi = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                lo |= e4m3_signed(__fmul_rn(f[i], r)) << (8 * i);
                hi |= e4m3_signed(__fmul_rn(f[4 + i], r)) << (8 * i);
            }
            if (in_span(NV4_SITE(0), sp.codes, a + row * K + j * 8, 8))
                *reinterpret_cast<uint2 *>(a + row * K + j * 8) = make_uint2(lo, hi);
        }
    }
}

__global__ void probe_convert_kernel(const float *__restrict__ in, int64_t n, uint8_t *__restrict__ o2,
                                     uint8_t *__restrict__ o3, const QuantSpans sp)
{
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        if (!(in_span(NV4_SITE(0), sp.x, in + i, 4) && in_span(NV4_SITE(0), sp.codes, o2 + i, 1) &&
              in_span(NV4_SITE(0), sp.scales, o3 + i, 1)))
            continue;
        const float v = in[i];
        o2[i] = (uint8_t)(e2m1x2(v, 0.0f) & 0xFu);
        o3[i] = (uint8_t)e4m3_signed(v);
    }
}

// Split-K epilogue for BF16 outputs: y = bf16_rn(acc).
__global__ void finalize_bf16_kernel(const float *__restrict__ acc, int64_t rows, int64_t cols, int64_t ld_acc,
                                     uint16_t *__restrict__ y, int64_t ldy, const QuantSpans sp)
{
    const int64_t total = rows * cols;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / cols, c = i - r * cols;
        if (in_span(NV4_SITE(0), sp.x, acc + r * ld_acc + c, 4) && in_span(NV4_SITE(0), sp.codes, y + r * ldy + c, 2))
            y[r * ldy + c] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[r * ld_acc + c]));
    }
}

// Cluster size of the small-activation quantiser: 16 CTAs where the device
// can hold such a cluster (decided once, by an occupancy query: no launch,
// so it is also safe while a stream is being captured), else 8.
int small_cluster_size()
{
    static std::once_flag once;
    static int fc = 8;
    std::call_once(once, [] {
        if (cudaFuncSetAttribute(nvfp4_encode_small_kernel<true, 16>, cudaFuncAttributeNonPortableClusterSizeAllowed,
                                 1) != cudaSuccess ||
            cudaFuncSetAttribute(nvfp4_encode_small_kernel<false, 16>, cudaFuncAttributeNonPortableClusterSizeAllowed,
                                 1) != cudaSuccess) {
            cudaGetLastError();
            return;
        }
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(16);
        cfg.blockDim = dim3(FT);
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 16;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, nvfp4_encode_small_kernel<true, 16>, &cfg) == cudaSuccess &&
            clusters > 0)
            fc = 16;
        cudaGetLastError();
    });
    return fc;
}

} // namespace

cudaError_t launch_nvfp4_quantize(const uint16_t *x, int64_t rows, int64_t K, int64_t ldx, uint8_t *codes,
                                  uint8_t *scales, void *second, int mode, int layout, uint32_t *amax_partial,
                                  uint32_t *status, cudaStream_t stream, bool zero_pad)
{
    const int zp = zero_pad ? 1 : 0;
    const bool tiled = layout == NVFP4_LAYOUT_MMA_TILED;
    const int64_t rows_pad = tiled ? ceil_div(rows, 128) * 128 : rows;
    QuantSpans sp;
    sp.x = span_of(x, matrix_bytes(rows, K, ldx, 2));
    sp.codes = span_of(codes, (uint64_t)rows * (uint64_t)(K / 2));
    sp.scales = span_of(scales, tiled ? tiled_scale_bytes(rows, K) : (uint64_t)rows * (uint64_t)(K / 16));
    sp.second = span_of(second, mode == NVFP4_SCALE_MACRO_FP16 ? 2u * (uint64_t)rows * (uint64_t)(K / 256) : 4u);
    sp.partial = span_of(amax_partial, WS_AMAX_BYTES);
    const int sms = device_sm_count();
    if (rows_pad == 0)
        return cudaSuccess;
    const int grid2 = (int)std::min<int64_t>(rows_pad, (int64_t)sms * 8);
    if (mode == NVFP4_SCALE_TENSOR_FP32 && rows * (K / 8) <= FUSED_MAX_CHUNKS) {
        // small activations: one cluster, one launch
        const int fc = small_cluster_size();
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(fc);
        cfg.blockDim = dim3(FT);
        cfg.stream = stream;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = fc;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        float *sg = static_cast<float *>(second);
        if (fc == 16)
            return tiled ? cudaLaunchKernelEx(&cfg, nvfp4_encode_small_kernel<true, 16>, x, rows, rows_pad, K, ldx,
                                              codes, scales, sg, status, zp, sp)
                         : cudaLaunchKernelEx(&cfg, nvfp4_encode_small_kernel<false, 16>, x, rows, rows_pad, K, ldx,
                                              codes, scales, sg, status, zp, sp);
        return tiled ? cudaLaunchKernelEx(&cfg, nvfp4_encode_small_kernel<true, 8>, x, rows, rows_pad, K, ldx, codes,
                                          scales, sg, status, zp, sp)
                     : cudaLaunchKernelEx(&cfg, nvfp4_encode_small_kernel<false, 8>, x, rows, rows_pad, K, ldx, codes,
                                          scales, sg, status, zp, sp);
    }
    if (mode == NVFP4_SCALE_TENSOR_FP32 && ldx == K) {
        // contiguous x: the staged streaming passes (3 and 4 CTAs per SM)
        const int64_t units = ceil_div(std::max<int64_t>(rows * (K / 16), 1), (int64_t)SU_BLOCKS);
        const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(units, std::min(AMAX_MAX_CTAS, sms * SU_CTAS_1)));
        const uint64_t tmo = 2000000000ull;
        float *sg = static_cast<float *>(second);
        const int grid2 = (int)std::max<int64_t>(1, std::min<int64_t>(units, (int64_t)sms * SU_CTAS_2));
        auto k1 = stream_quant_kernel<1, false, SU_STAGES_1>;
        auto k2 = tiled ? stream_quant_kernel<2, true, SU_STAGES_2> : stream_quant_kernel<2, false, SU_STAGES_2>;
        cudaError_t e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, su_smem(SU_STAGES_1));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, su_smem(SU_STAGES_2));
        if (e == cudaSuccess)
            e = launch_pdl(k1, grid, SU_THREADS, su_smem(SU_STAGES_1), stream, x, rows, rows_pad, K, codes, scales,
                           sg, amax_partial, 0, zp, status, tmo, sp);
        if (e == cudaSuccess)
            e = launch_pdl(k2, grid2, SU_THREADS, su_smem(SU_STAGES_2), stream, x, rows, rows_pad, K, codes, scales,
                           sg, amax_partial, grid, zp, status, tmo, sp);
        if (e != cudaSuccess)
            return e;
    } else if (mode == NVFP4_SCALE_TENSOR_FP32) {
        // strided x: flat passes with register loads; enough CTAs for one
        // sweep of QU loads per thread, at most a few waves
        const int64_t blocks1 = std::max<int64_t>(rows * (K / 16), 1);
        const int64_t per_cta = (int64_t)QT * QU;
        const int grid1 = (int)std::min<int64_t>(ceil_div(blocks1, per_cta), std::min(AMAX_MAX_CTAS, sms * 4));
        const int64_t pad_words = tiled ? (rows_pad - rows) * (K / 64) : 0;
        const int64_t blocks = std::max<int64_t>(rows * (K / 16), 1);
        const int grid_e = (int)std::max<int64_t>(
            1, std::min<int64_t>(std::max(ceil_div(blocks, (int64_t)QT * QB), ceil_div(pad_words, (int64_t)QT * 8)),
                                 (int64_t)sms * 8));
        // 32-byte block loads when x and its row stride allow them
        const bool v8 = (reinterpret_cast<uintptr_t>(x) % 32) == 0 && (ldx % 16) == 0;
        cudaError_t e = v8 ? launch_pdl(amax_partial_kernel<true>, grid1, QT, 0, stream, x, rows, K, ldx,
                                        amax_partial, status, sp)
                           : launch_pdl(amax_partial_kernel<false>, grid1, QT, 0, stream, x, rows, K, ldx,
                                        amax_partial, status, sp);
        if (e != cudaSuccess)
            return e;
        float *sg = static_cast<float *>(second);
        const uint32_t *part = amax_partial;
        if (tiled)
            e = v8 ? launch_pdl(nvfp4_encode_kernel<true, true>, grid_e, QT, 0, stream, x, rows, rows_pad, K, ldx,
                                codes, scales, sg, part, grid1, zp, sp)
                   : launch_pdl(nvfp4_encode_kernel<true, false>, grid_e, QT, 0, stream, x, rows, rows_pad, K, ldx,
                                codes, scales, sg, part, grid1, zp, sp);
        else
            e = v8 ? launch_pdl(nvfp4_encode_kernel<false, true>, grid_e, QT, 0, stream, x, rows, rows_pad, K, ldx,
                                codes, scales, sg, part, grid1, zp, sp)
                   : launch_pdl(nvfp4_encode_kernel<false, false>, grid_e, QT, 0, stream, x, rows, rows_pad, K, ldx,
                                codes, scales, sg, part, grid1, zp, sp);
        if (e != cudaSuccess)
            return e;
    } else {
        if (tiled)
            nvfp4_encode_macro_kernel<true><<<grid2, QT, 0, stream>>>(x, rows, rows_pad, K, ldx, codes, scales,
                                                                        static_cast<uint16_t *>(second), status, sp);
        else
            nvfp4_encode_macro_kernel<false><<<grid2, QT, 0, stream>>>(x, rows, rows_pad, K, ldx, codes, scales,
                                                                         static_cast<uint16_t *>(second), status, sp);
    }
    return cudaGetLastError();
}

cudaError_t launch_fp8_quantize(const uint16_t *x, int64_t rows, int64_t K, int64_t ldx, uint8_t *a, float *s_t,
                                uint32_t *status, cudaStream_t stream)
{
    if (rows == 0)
        return cudaSuccess;
    const int grid = (int)std::min<int64_t>(rows, (int64_t)device_sm_count() * 8);
    QuantSpans sp;
    sp.x = span_of(x, matrix_bytes(rows, K, ldx, 2));
    sp.codes = span_of(a, (uint64_t)rows * (uint64_t)K);
    sp.scales = span_of(s_t, 4u * (uint64_t)rows);
    fp8_token_kernel<<<grid, QT, 0, stream>>>(x, rows, K, ldx, a, s_t, status, sp);
    return cudaGetLastError();
}

cudaError_t launch_probe_convert(const float *in, int64_t n, uint8_t *o2, uint8_t *o3, cudaStream_t stream)
{
    if (n == 0)
        return cudaSuccess;
    const int grid = (int)std::min<int64_t>(ceil_div(n, 256), (int64_t)device_sm_count() * 16);
    QuantSpans sp;
    sp.x = span_of(in, 4u * (uint64_t)n);
    sp.codes = span_of(o2, (uint64_t)n);
    sp.scales = span_of(o3, (uint64_t)n);
    probe_convert_kernel<<<grid, 256, 0, stream>>>(in, n, o2, o3, sp);
    return cudaGetLastError();
}

cudaError_t launch_finalize_bf16(const float *acc, int64_t rows, int64_t cols, int64_t ld_acc, uint16_t *y,
                                 int64_t ldy, cudaStream_t stream)
{
    const int64_t total = rows * cols;
    if (total == 0)
        return cudaSuccess;
    const int grid = (int)std::min<int64_t>(ceil_div(total, 256), (int64_t)device_sm_count() * 8);
    QuantSpans sp;
    sp.x = span_of(acc, matrix_bytes(rows, cols, ld_acc, 4));
    sp.codes = span_of(y, matrix_bytes(rows, cols, ldy, 2));
    finalize_bf16_kernel<<<grid, 256, 0, stream>>>(acc, rows, cols, ld_acc, y, ldy, sp);
    return cudaGetLastError();
}

} // namespace nv4
