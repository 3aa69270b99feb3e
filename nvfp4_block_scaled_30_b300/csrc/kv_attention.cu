// NVFP4 paged KV cache: append of one token per sequence and decode attention.
//
// "The FP4 Inflection: Rethinking AI Inference Architecture" (section "What
// does this mean for model serving engines?") stores the KV cache in FP4 and
// names paged attention as its consumer; the engine-build listing of "NVIDIA
// Ships TensorRT-LLM 0.16" pages the cache in blocks of 64 tokens.  Cached key
// and value head vectors use the activation block encoder (16 elements along
// head_dim, E4M3 block scales) under a static FP32 tensor scale per cache
// tensor; attention is scaled dot-product attention of one query token over
// the cached tokens, the query heads of a group sharing one KV head.
//
// Page block layout (head_dim D = 128, 64 tokens per page): one contiguous
// 9216-byte block per page and KV head, made of two 4608-byte halves of 32
// tokens each; half h (at byte 4608 h) holds, for its tokens:
//   [0, 2048)     K codes  [4 dim chunks][32 key slots][16 bytes] (chunk q:
//                 dims 32 q .. 32 q + 31, element 2j in the low nibble of
//                 byte j); key slot kpos4(token) holds the token
//   [2048, 2304)  K scales [32 key slots][8]
//   [2304, 4352)  V codes  [128 dims][16 bytes]  (dim-major: byte j of row d
//                 holds tokens 2j (low nibble) and 2j+1 of dim d)
//   [4352, 4608)  V scales [8 blocks][32 tokens]
// so that every tensor-core operand fragment of the attention comes straight
// from code bytes (K rows feed the B operand of S = Q K^T, V rows (dims) the
// A operand of O^T = V^T P^T, both through ldmatrix, each 8x16-byte matrix
// one contiguous 128 bytes: no bank conflicts), and a half page, the unit
// the attention streams, is ONE bulk copy (measured on B300: an SM serves
// bulk copies this small at a roughly fixed cost per copy).
//
// Decode attention, one CTA per (sequence, KV head, split of the context),
// 4 warps; each warp streams its own half pages through a 2-stage per-warp
// ring (4.5 KB units for NVFP4, small enough for 4 CTAs = 16 warps per SM;
// 8 KB units for FP8, 3 CTAs): the kernels are bound by instruction latency
// at these occupancies, not by tensor or memory throughput.  Products by mma.sync m16n8k16 (FP16 operands, FP32
// accumulation): S = Q K^T with the group's query heads (<= 16) as M, then
// O^T = V^T P^T with 16 value dimensions as M and the heads as N; these
// contractions have 8-16 rows on one side, far below the 64/128 rows of a
// tcgen05 MMA.  Online softmax in FP32 (base 2); warps merge through shared
// memory; splits merge in a second kernel.
#include <algorithm>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace nv4 {

namespace {

constexpr int KV_D = 128;           // head_dim
constexpr int KV_P = 64;            // tokens per page
constexpr int KV_H = KV_P / 2;      // tokens per half page, the unit of the attention
constexpr int KS4_OFF = KV_H * KV_D / 2;              // 2048: K scales of a half page
constexpr int VC4_OFF = KS4_OFF + KV_H * KV_D / 16;   // 2304: V codes
constexpr int VS4_OFF = VC4_OFF + KV_H * KV_D / 2;    // 4352: V scales
constexpr int HALF4_BYTES = VS4_OFF + KV_H * KV_D / 16; // 4608
constexpr int PAGE_BYTES = 2 * HALF4_BYTES;           // 9216
constexpr int KC8_BYTES = KV_P * KV_D;              // FP8 codes of one page and head, 8192
constexpr int HALF8_BYTES = KC8_BYTES / 2;          // one 32-token half (keys or values)
constexpr int PAGE8_BYTES = 2 * KC8_BYTES;          // FP8 page block: [2 halves][K 4096 | V 4096]
constexpr int ATT_WARPS = 4;
constexpr int ATT_STAGES = 2;

// Key slot of token k (0..31) of a half page.  The attention reads the keys
// of one score n-tile (8 keys, chunk_key / chunk_key8 below) as 8
// consecutive 16-byte rows: n-tile j column n sits in slot 8 j + n.  NVFP4:
// the 2-bit fields k[4:3] and k[2:1] trade places; FP8: k[1] moves to bit 3
// and k[3:2] to bits 2:1.
__host__ __device__ __forceinline__ int kpos4(int k) { return 8 * ((k >> 1) & 3) + 2 * (k >> 3) + (k & 1); }
__host__ __device__ __forceinline__ int kpos8(int k) { return (k & 16) | ((k & 2) << 2) | ((k >> 1) & 6) | (k & 1); }

__device__ __forceinline__ uint32_t h2_e2m1x2(uint32_t byte)
{
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(r) : "r"(byte));
    return r;
}

// f16x2 of two E4M3 bytes (lo in bits 0..7, hi in bits 8..15).
__device__ __forceinline__ uint32_t h2_e4m3x2(uint32_t two)
{
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"((uint16_t)two));
    return r;
}

__device__ __forceinline__ uint32_t hmul2u(uint32_t a, uint32_t b)
{
    __half2 r = __hmul2(*reinterpret_cast<__half2 *>(&a), *reinterpret_cast<__half2 *>(&b));
    return *reinterpret_cast<uint32_t *>(&r);
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi)
{
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// 2^x (the approximate hardware exponential: relative error ~2^-22, far
// inside the attention tolerance)
__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void ldsm_x4(const void *row_addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(row_addr)));
}

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
                 "{%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ---- append ------------------------------------------------------------------------
// One thread per 16-element block of one new key or value vector.
__global__ void kv_append_kernel(KvAppendArgs a)
{
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int nblk = KV_D / 16;
    const int64_t total = (int64_t)a.B * a.H_kv * 2 * nblk;
    if (tid >= total)
        return;
    const int blk = (int)(tid % nblk);
    const int which = (int)((tid / nblk) % 2); // 0 key, 1 value
    const int hk = (int)((tid / (2 * nblk)) % a.H_kv);
    const int b = (int)(tid / (2 * nblk * a.H_kv));
    if (!in_span(NV4_SITE(0), a.sp_positions, a.positions + b, 4))
        return;
    const int pos = a.positions[b];
    if (pos < 0 || pos / KV_P >= a.max_pages)
        return;
    if (!in_span(NV4_SITE(0), a.sp_block_table, a.block_table + (int64_t)b * a.max_pages + pos / KV_P, 4))
        return;
    const int page = a.block_table[(int64_t)b * a.max_pages + pos / KV_P];
    if (page < 0 || page >= a.num_pages)
        return;
    const int slot = pos % KV_P;
    const uint16_t *src = (which ? a.v_new : a.k_new) + ((int64_t)b * a.H_kv + hk) * KV_D + blk * 16;
    if (!in_span(NV4_SITE(0), which ? a.sp_v_new : a.sp_k_new, src, 32) ||
        !in_span(NV4_SITE(0), which ? a.sp_v_scale : a.sp_k_scale, which ? a.v_scale : a.k_scale, 4))
        return;
    float x[16];
    float amb = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        x[i] = __uint_as_float((uint32_t)src[i] << 16);
        amb = fmaxf(amb, fabsf(x[i]));
    }
    const float s = *(which ? a.v_scale : a.k_scale);
    if (a.fmt == KV_FMT_FP8) {
        // E4M3(x * 1/s) per element; per 32-token half, keys [8 dim chunks]
        // [32 key slots][16], values [2 token groups][128 dims][16]
        const float r8 = recip_step(s);
        uint8_t *blk8 = a.pages + ((int64_t)page * a.H_kv + hk) * PAGE8_BYTES + (slot / 32) * (2 * HALF8_BYTES);
        uint32_t c[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
            c[i] = e4m3(__fmul_rn(x[i], r8)) | (x[i] < 0.0f || (x[i] == 0.0f && signbit(x[i])) ? 0x80u : 0u);
        if (!which) {
            uint32_t wds[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                wds[q] = c[4 * q] | (c[4 * q + 1] << 8) | (c[4 * q + 2] << 16) | (c[4 * q + 3] << 24);
            uint8_t *dk = blk8 + (blk * 32 + kpos8(slot % 32)) * 16;
            if (in_span(NV4_SITE(0), a.sp_pages, dk, 16))
                *reinterpret_cast<uint4 *>(dk) = make_uint4(wds[0], wds[1], wds[2], wds[3]);
        } else {
            const int sl = slot % 32;
            uint8_t *vc = blk8 + HALF8_BYTES + (sl >> 4) * (KV_D * 16) + (sl & 15);
#pragma unroll
            for (int i = 0; i < 16; ++i)
                if (in_span(NV4_SITE(0), a.sp_pages, vc + (blk * 16 + i) * 16, 1))
                    vc[(blk * 16 + i) * 16] = (uint8_t)c[i];
        }
        return;
    }
    const uint32_t e = block_scale_code(amb, s);
    const float r = recip_step(__fmul_rn(e4m3_value(e), s));
    // the half page of this slot, and the slot's token within it
    uint8_t *pb = a.pages + ((int64_t)page * a.H_kv + hk) * PAGE_BYTES + (slot / KV_H) * HALF4_BYTES;
    const int sl = slot % KV_H;
    if (!which) {
        uint32_t pk[2] = {0u, 0u};
#pragma unroll
        for (int i = 0; i < 8; ++i)
            pk[i >> 2] |= e2m1x2(__fmul_rn(x[2 * i], r), __fmul_rn(x[2 * i + 1], r)) << (8 * (i & 3));
        const int kp = kpos4(sl);
        uint8_t *dk = pb + ((blk >> 1) * KV_H + kp) * 16 + (blk & 1) * 8;
        if (in_span(NV4_SITE(0), a.sp_pages, dk, 8))
            *reinterpret_cast<uint2 *>(dk) = make_uint2(pk[0], pk[1]);
        if (in_span(NV4_SITE(0), a.sp_pages, pb + KS4_OFF + kp * (KV_D / 16) + blk, 1))
            pb[KS4_OFF + kp * (KV_D / 16) + blk] = (uint8_t)e;
    } else {
        uint8_t *vc = pb + VC4_OFF;
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
            const uint32_t two = e2m1x2(__fmul_rn(x[i], r), __fmul_rn(x[i + 1], r));
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t c = (two >> (4 * h)) & 15u;
                uint8_t *p = vc + (blk * 16 + i + h) * (KV_H / 2) + sl / 2;
                if (!in_span(NV4_SITE(0), a.sp_pages, p, 1))
                    continue;
                *p = (sl & 1) ? (uint8_t)((*p & 0x0Fu) | (c << 4)) : (uint8_t)((*p & 0xF0u) | c);
            }
        }
        if (in_span(NV4_SITE(0), a.sp_pages, pb + VS4_OFF + blk * KV_H + sl, 1))
            pb[VS4_OFF + blk * KV_H + sl] = (uint8_t)e;
    }
}

// ---- decode attention ------------------------------------------------------------------

// The unit ring is dead once every warp has left its loop, so the warps'
// partial outputs reuse it for the merge.
struct AttMerge {
    float o[ATT_WARPS][16][KV_D];
    float m[ATT_WARPS][16];
    float l[ATT_WARPS][16];
};
template <int UNIT>
struct AttSmem {
    union {
        uint8_t unit[ATT_WARPS][ATT_STAGES][UNIT]; // per warp: the half pages in flight
        AttMerge merge;
    };
    uint64_t full[ATT_WARPS][ATT_STAGES];
};
static_assert(sizeof(AttMerge) <= ATT_WARPS * ATT_STAGES * HALF4_BYTES, "merge buffer fits in the ring");
using AttSmem4 = AttSmem<HALF4_BYTES>;
using AttSmem8 = AttSmem<2 * HALF8_BYTES>;

// Merge of the 4 warps' running softmax states (row sums over the 4 lanes
// of a group, then through shared memory: the page ring, idle in every warp
// by now) and the store of the output, or of this split's partial.
// The output accumulators hold O^T: o[mt][nt][i] is dimension 16 mt + g +
// 8 (i >> 1) of head 8 nt + 2t + (i & 1).
template <int NT>
__device__ __forceinline__ void kv_merge_and_store(const KvAttnArgs &a, AttMerge &mg, const float (&o)[8][NT][4],
                                                   const float (&m_run)[2], float (&l_run)[2], int warp, int g,
                                                   int t, int G, int b, int hk, int split, float s_v)
{
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        l_run[rr] += __shfl_xor_sync(0xFFFFFFFFu, l_run[rr], 1);
        l_run[rr] += __shfl_xor_sync(0xFFFFFFFFu, l_run[rr], 2);
    }
    __syncthreads();
    if (t == 0) {
        mg.m[warp][g] = m_run[0];
        mg.m[warp][g + 8] = m_run[1];
        mg.l[warp][g] = l_run[0];
        mg.l[warp][g + 8] = l_run[1];
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i)
                mg.o[warp][8 * nt + 2 * t + (i & 1)][16 * mt + g + 8 * (i >> 1)] = o[mt][nt][i];
    __syncthreads();
    for (int idx = threadIdx.x; idx < G * KV_D; idx += 32 * ATT_WARPS) {
        const int head = idx / KV_D, d = idx % KV_D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < ATT_WARPS; ++w)
            M = fmaxf(M, mg.m[w][head]);
        float L = 0.0f, O = 0.0f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < ATT_WARPS; ++w) {
                const float f = mg.m[w][head] == -INFINITY ? 0.0f : ex2(mg.m[w][head] - M);
                L += f * mg.l[w][head];
                O += f * mg.o[w][head][d];
            }
        }
        const int64_t hq = (int64_t)b * a.H + hk * G + head;
        if (a.n_splits == 1) {
            const float y = L > 0.0f ? O * s_v / L : 0.0f;
            if (a.out_dtype == NVFP4_OUT_BF16) {
                if (in_span(NV4_SITE(0), a.sp_out, static_cast<__nv_bfloat16 *>(a.out) + hq * KV_D + d, 2))
                    static_cast<__nv_bfloat16 *>(a.out)[hq * KV_D + d] = __float2bfloat16_rn(y);
            } else if (in_span(NV4_SITE(0), a.sp_out, static_cast<float *>(a.out) + hq * KV_D + d, 4)) {
                static_cast<float *>(a.out)[hq * KV_D + d] = y;
            }
        } else {
            float *part = a.partial + (hq * a.n_splits + split) * (KV_D + 2);
            if (in_span(NV4_SITE(0), a.sp_partial, part, (KV_D + 2) * 4)) {
                part[d] = O;
                if (d == 0) {
                    part[KV_D] = M;
                    part[KV_D + 1] = L;
                }
            }
        }
    }
}

// Online softmax update of one 32-key chunk's scores (base 2, already
// scaled): masks keys past `valid` (a partial chunk only), updates the running
// maxima and sums, and returns the P fragments of the chunk's two 16-key
// steps and whether any row maximum grew (warp-uniform), with the factors
// corr[] (rows g, g + 8) by which that row's accumulated output must be
// scaled.  Key of sc[j][i] is key_of(j, 2t + (i & 1)); rows g (i < 2), g + 8
// (i >= 2, skipped when the group has at most 8 query heads: those rows are
// padding and get P = 0).  P of 16-key step s, n-tile (heads) nt: the B
// operand pair (pf[s][nt], pf[s][2 + nt]) of O^T += V^T P^T.
template <typename KeyOf>
__device__ __forceinline__ bool kv_softmax_chunk(float (&sc)[4][4], int valid, int t, KeyOf key_of, bool hi_rows,
                                                 float (&m_run)[2], float (&l_run)[2], float (&corr)[2],
                                                 uint32_t (&pf)[2][4])
{
    if (valid < 32) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int i = 0; i < 4; ++i)
                sc[j][i] = key_of(j, 2 * t + (i & 1)) < valid ? sc[j][i] : -INFINITY;
    }
    float cmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int i = 0; i < 4; ++i)
            cmax[i >> 1] = fmaxf(cmax[i >> 1], sc[j][i]);
    const int nrows = hi_rows ? 2 : 1;
    bool grew = false;
    corr[0] = corr[1] = 1.0f;
    for (int rr = 0; rr < nrows; ++rr) {
        cmax[rr] = fmaxf(cmax[rr], __shfl_xor_sync(0xFFFFFFFFu, cmax[rr], 1));
        cmax[rr] = fmaxf(cmax[rr], __shfl_xor_sync(0xFFFFFFFFu, cmax[rr], 2));
        if (cmax[rr] > m_run[rr]) {
            corr[rr] = m_run[rr] == -INFINITY ? 0.0f : ex2(m_run[rr] - cmax[rr]);
            m_run[rr] = cmax[rr];
            l_run[rr] *= corr[rr];
            grew = true;
        }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float pv[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (i >= 2 && !hi_rows)
                continue;
            const float mm = m_run[i >> 1];
            pv[i] = mm == -INFINITY ? 0.0f : ex2(sc[j][i] - mm);
            l_run[i >> 1] += pv[i];
        }
        // n-tile j -> step j / 2; even j: k slots 2t, 2t+1; odd j: 2t+8, 2t+9
        pf[j >> 1][(j & 1) * 2 + 0] = pack_h2(pv[0], pv[1]);
        pf[j >> 1][(j & 1) * 2 + 1] = pack_h2(pv[2], pv[3]);
    }
    return __any_sync(0xFFFFFFFFu, grew);
}

// Rescale of the O^T accumulators by the factors of their heads (column
// 2t, 2t+1 of n-tile nt = head rows held by lanes 4 (2t) and 4 (2t+1)).
template <int NT>
__device__ __forceinline__ void kv_rescale(float (&o)[8][NT][4], const float (&corr)[2], int t)
{
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const float c0 = __shfl_sync(0xFFFFFFFFu, corr[nt], 8 * t);
        const float c1 = __shfl_sync(0xFFFFFFFFu, corr[nt], 8 * t + 4);
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            o[mt][nt][0] *= c0;
            o[mt][nt][1] *= c1;
            o[mt][nt][2] *= c0;
            o[mt][nt][3] *= c1;
        }
    }
}

// Key order inside a 32-key chunk: QK n-tile j (8 keys) column n holds key
// 8 (n / 2) + (n % 2) + 2 j, so that the S fragment of n-tiles 0, 1 (2, 3)
// is exactly the P^T operand (B) of the first (second) 16-key step of
// O^T = V^T P^T, whose k slots 2t, 2t+1, 2t+8, 2t+9 hold keys 8t .. 8t+3
// (8t+4 .. 8t+7): the keys of V code byte 4t .. 4t+1 (4t+2 .. 4t+3) that
// ldmatrix hands lane t.  That key sits in slot kpos4 = 8 j + n.
__device__ __forceinline__ int chunk_key(int j, int n) { return 8 * (n >> 1) + (n & 1) + 2 * j; }

// Occupancy: at most 128 registers a thread for one n-tile, so that 4 CTAs
// fit on an SM (the ring takes 36 KB of shared memory per CTA); 3 for two.
template <int NT>
__global__ void __launch_bounds__(32 * ATT_WARPS, NT == 1 ? 4 : 3) kv_decode_kernel(const KvAttnArgs a)
{
    extern __shared__ __align__(128) uint8_t att_raw[];
    AttSmem4 &sm = *reinterpret_cast<AttSmem4 *>(att_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int split = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
    const int G = a.H / a.H_kv;
    const int ctx_b = in_span(NV4_SITE(0), a.sp_ctx_lens, a.ctx_lens + b, 4) ? a.ctx_lens[b] : 0;
    const int ctx = max(0, min(min(ctx_b, a.max_ctx), a.max_pages * KV_P));
    const int k_begin = split * a.keys_per_split;
    const int k_end = min(ctx, k_begin + a.keys_per_split);
    const int n_chunks = k_end > k_begin ? (k_end - k_begin + KV_H - 1) / KV_H : 0;

    if (lane == 0) {
        for (int s = 0; s < ATT_STAGES; ++s)
            mbar_init(&sm.full[warp][s], 1);
        fence_mbar_init();
    }
    __syncwarp();

    // query fragments (A operand of S = Q K^T): rows = the group's heads (row
    // g and g + 8), k slots of 16-dim step 2c + u hold dims 32 c + 8 t + 4 u
    // + {0, 1} (slots 2t, 2t+1) and + {2, 3} (slots 2t+8, 2t+9), matching
    // the dims ldmatrix hands lane t from a 16-byte chunk of a key row.
    // Scores in base 2: q is pre-multiplied by sm_scale * log2(e).
    uint32_t qf[8][4];
    {
        const float qs = a.sm_scale * 1.4426950408889634f;
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int d0 = 32 * c + 8 * t + 4 * u;
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    const int head = g + 8 * rr;
                    float v[4] = {0.f, 0.f, 0.f, 0.f};
                    if (head < G) {
                        const uint16_t *q = a.q + ((int64_t)b * a.H + hk * G + head) * KV_D + d0;
                        if (in_span(NV4_SITE(0), a.sp_q, q, 8)) {
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                v[i] = __uint_as_float((uint32_t)q[i] << 16) * qs;
                        }
                    }
                    qf[2 * c + u][rr] = pack_h2(v[0], v[1]);
                    qf[2 * c + u][2 + rr] = pack_h2(v[2], v[3]);
                }
            }
    }
    const float s_k = in_span(NV4_SITE(0), a.sp_k_scale, a.k_scale, 4) ? *a.k_scale : 0.0f;
    const float s_v = in_span(NV4_SITE(0), a.sp_v_scale, a.v_scale, 4) ? *a.v_scale : 0.0f;

    // O^T accumulators: 8 m-tiles of 16 dimensions x NT n-tiles of 8 heads
    float o[8][NT][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i)
                o[mt][nt][i] = 0.0f;
    float m_run[2] = {-INFINITY, -INFINITY}; // rows g, g + 8 (base-2 scores of unit K)
    float l_run[2] = {0.0f, 0.0f};           // this lane's share of the row sums

    // chunk c of this CTA's range: keys k_begin + 32 c .. + 31 = half
    // ((k_begin / 32 + c) % 2) of page (k_begin + 32 c) / 64; chunks of this
    // warp: c = warp, warp + 4, ...; page ids of its first 32, one per lane
    int my_pg = 0;
    if (warp + ATT_WARPS * lane < n_chunks)
    {
        const int32_t *bt = a.block_table + (int64_t)b * a.max_pages + (k_begin + KV_H * (warp + ATT_WARPS * lane)) / KV_P;
        my_pg = in_span(NV4_SITE(0), a.sp_block_table, bt, 4) ? *bt : 0;
    }
    // warp-collective (the page id comes from a shuffle); one copy per half page
    auto issue = [&](int c, int s) {
        const int i = (c - warp) / ATT_WARPS;
        const int tok = k_begin + KV_H * c;
        int page = __shfl_sync(0xFFFFFFFFu, my_pg, i & 31);
        if (i >= 32)
            page = in_span(NV4_SITE(0), a.sp_block_table, a.block_table + (int64_t)b * a.max_pages + tok / KV_P, 4)
                       ? a.block_table[(int64_t)b * a.max_pages + tok / KV_P]
                       : 0;
        const int64_t ph = (int64_t)min(max(page, 0), a.num_pages - 1) * a.H_kv + hk;
        const int half = (tok / KV_H) & 1;
        if (lane == 0) {
            mbar_arrive_expect_tx(&sm.full[warp][s], HALF4_BYTES);
            if (in_span(NV4_SITE(0), a.sp_pages, a.pages + ph * PAGE_BYTES + half * HALF4_BYTES, HALF4_BYTES))
                bulk_load(sm.unit[warp][s], a.pages + ph * PAGE_BYTES + half * HALF4_BYTES, HALF4_BYTES,
                          &sm.full[warp][s]);
        }
    };
    for (int i = 0; i < ATT_STAGES && warp + i * ATT_WARPS < n_chunks; ++i)
        issue(warp + i * ATT_WARPS, i);
    bool ok = true;
    int it = 0;
    for (int c = warp; c < n_chunks; c += ATT_WARPS, ++it) {
        const int s = it % ATT_STAGES;
        const uint32_t par = (uint32_t)(it / ATT_STAGES) & 1u;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&sm.full[warp][s], par, a.timeout_ns, nullptr))) {
            if (lane == 0)
                atomicOr(a.status, ST_TIMEOUT);
            ok = false;
            break;
        }
        const uint8_t *kc = sm.unit[warp][s];
        const uint8_t *ks = kc + KS4_OFF;
        const uint8_t *vc = kc + VC4_OFF;
        const uint8_t *vs = kc + VS4_OFF;
        const int valid = min(KV_H, k_end - (k_begin + KV_H * c)); // keys of this chunk in the context
        {
            // ---- S = Q K^T over 32 keys: 4 n-tiles x 8 k-steps
            float sc[4][4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                // ldmatrix matrix i = dims 32 i .. 32 i + 31 of the n-tile's
                // 8 keys (slots 8 j .. 8 j + 7); lane (g, t) receives key
                // chunk_key(j, g), dims 32 i + 8 t .. + 7
                uint32_t kr[4];
                ldsm_x4(kc + ((lane >> 3) * KV_H + 8 * j + (lane & 7)) * 16, kr);
                const uint2 sc8 = *reinterpret_cast<const uint2 *>(ks + (8 * j + g) * (KV_D / 16));
                const uint32_t sb[2] = {sc8.x, sc8.y}; // block scales of this lane's key, 8 bytes
                sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.0f;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    // dims 32 c + 8 t .. + 7 lie in block 2 c + t / 2
                    const uint32_t e = (sb[c >> 1] >> (8 * (2 * (c & 1) + (t >> 1)))) & 0xFFu;
                    const uint32_t e2 = h2_e4m3x2(e * 0x0101u);
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const uint32_t b0 = hmul2u(h2_e2m1x2((kr[c] >> (16 * u)) & 0xFFu), e2);
                        const uint32_t b1 = hmul2u(h2_e2m1x2((kr[c] >> (16 * u + 8)) & 0xFFu), e2);
                        mma16816(sc[j], qf[2 * c + u], b0, b1);
                    }
                }
            }
            // ---- online softmax (base 2: the queries carry sm_scale * log2 e)
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    sc[j][i] *= s_k;
            uint32_t pf[2][4]; // P fragments of the two 16-key steps
            float corr[2];
            if (kv_softmax_chunk(sc, valid, t, chunk_key, NT == 2, m_run, l_run, corr, pf))
                kv_rescale<NT>(o, corr, t);
            // ---- O^T += V^T P^T: A = value rows (8 m-tiles of 16 dims), B = P^T
            // (N = the group's heads: no padding rows); keys 8t .. 8t+7 of
            // this chunk are valid up to `valid`
            const bool full_chunk = valid >= 32;
            const int nv = min(8, max(0, valid - 8 * t));
#pragma unroll
            for (int mp = 0; mp < 4; ++mp) {
                // matrix i: value rows (dims) 32 mp + 8 i + 0..7; lane l supplies dim 32 mp + l
                uint32_t vr[4];
                ldsm_x4(vc + (32 * mp + lane) * (KV_H / 2), vr);
#pragma unroll
                for (int hm = 0; hm < 2; ++hm) {
                    // m-tile mt: dims 16 mt + g (vr[2 hm]) and + g + 8 (vr[2 hm + 1]), scale block mt
                    const int mt = 2 * mp + hm;
                    const uint2 e8 = *reinterpret_cast<const uint2 *>(vs + mt * KV_H + 8 * t);
                    uint32_t e2[4];
#pragma unroll
                    for (int y = 0; y < 4; ++y)
                        e2[y] = h2_e4m3x2(((y < 2 ? e8.x : e8.y) >> (16 * (y & 1))) & 0xFFFFu);
                    uint32_t av[2][4];
#pragma unroll
                    for (int r2 = 0; r2 < 2; ++r2)
#pragma unroll
                        for (int y = 0; y < 4; ++y) {          // byte y: keys 8t+2y, 8t+2y+1
                            uint32_t val = hmul2u(h2_e2m1x2((vr[2 * hm + r2] >> (8 * y)) & 0xFFu), e2[y]);
                            if (!full_chunk) {
                                if (2 * y >= nv)
                                    val = 0u;
                                else if (2 * y + 1 >= nv)
                                    val &= 0x0000FFFFu;
                            }
                            av[r2][y] = val;
                        }
#pragma unroll
                    for (int st = 0; st < 2; ++st) {
                        const uint32_t afr[4] = {av[0][2 * st], av[1][2 * st], av[0][2 * st + 1], av[1][2 * st + 1]};
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
                            mma16816(o[mt][nt], afr, pf[st][nt], pf[st][2 + nt]);
                    }
                }
            }
        }
        // the stage is free again: this warp's next half page goes into it
        __syncwarp();
        if (c + ATT_STAGES * ATT_WARPS < n_chunks) {
            fence_proxy_async_smem();
            issue(c + ATT_STAGES * ATT_WARPS, s);
        }
    }
    // drain: every copy this warp issued lands before the CTA moves on
    if (lane == 0 && !ok) {
        const int mine = n_chunks > warp ? (n_chunks - warp + ATT_WARPS - 1) / ATT_WARPS : 0;
        for (int i = it; i < mine && i < it + ATT_STAGES; ++i)
            mbar_wait(&sm.full[warp][i % ATT_STAGES], (uint32_t)(i / ATT_STAGES) & 1u, a.timeout_ns, nullptr);
    }

    kv_merge_and_store(a, sm.merge, o, m_run, l_run, warp, g, t, G, b, hk, split, s_v);
}

// FP8 cache (E4M3 codes, one static scale per tensor): the same structure
// with 32-token half pages as the unit (keys [8 dim chunks][32 key slots]
// [16] then values [2 token groups][128 dims][16], 8 KB contiguous in the
// FP8 page block, one bulk copy).  A 16-byte ldmatrix row holds 16 FP8
// elements, so lane t receives elements 4t .. 4t+3 of its row: for keys,
// dims 16 kk + 4t + {0,1} / {2,3} fill k slots 2t, 2t+1 / 2t+8, 2t+9 of k-step
// kk; for values, keys 16 s + 4t + ... of step s.  QK n-tile j column n holds
// key chunk_key8(j, n) (slot kpos8 = 8 j + n), matching those P slots.  One
// conversion per two elements, no per-element scale.
__device__ __forceinline__ int chunk_key8(int j, int n) { return 16 * (j >> 1) + 4 * (n >> 1) + (n & 1) + 2 * (j & 1); }

template <int NT>
__global__ void __launch_bounds__(32 * ATT_WARPS) kv_decode_fp8_kernel(const KvAttnArgs a)
{
    extern __shared__ __align__(128) uint8_t att_raw[];
    AttSmem8 &sm = *reinterpret_cast<AttSmem8 *>(att_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int split = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
    const int G = a.H / a.H_kv;
    const int ctx_b = in_span(NV4_SITE(0), a.sp_ctx_lens, a.ctx_lens + b, 4) ? a.ctx_lens[b] : 0;
    const int ctx = max(0, min(min(ctx_b, a.max_ctx), a.max_pages * KV_P));
    const int k_begin = split * a.keys_per_split;
    const int k_end = min(ctx, k_begin + a.keys_per_split);
    const int n_chunks = k_end > k_begin ? (k_end - k_begin + 31) / 32 : 0;

    if (lane == 0) {
        for (int s = 0; s < ATT_STAGES; ++s)
            mbar_init(&sm.full[warp][s], 1);
        fence_mbar_init();
    }
    __syncwarp();

    uint32_t qf[8][4];
    {
        const float qs = a.sm_scale * 1.4426950408889634f;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const int head = g + 8 * rr;
                float v[4] = {0.f, 0.f, 0.f, 0.f};
                if (head < G) {
                    const uint16_t *q = a.q + ((int64_t)b * a.H + hk * G + head) * KV_D + 16 * kk + 4 * t;
                    if (in_span(NV4_SITE(0), a.sp_q, q, 8)) {
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            v[i] = __uint_as_float((uint32_t)q[i] << 16) * qs;
                    }
                }
                qf[kk][rr] = pack_h2(v[0], v[1]);
                qf[kk][2 + rr] = pack_h2(v[2], v[3]);
            }
    }
    const float s_k = in_span(NV4_SITE(0), a.sp_k_scale, a.k_scale, 4) ? *a.k_scale : 0.0f;
    const float s_v = in_span(NV4_SITE(0), a.sp_v_scale, a.v_scale, 4) ? *a.v_scale : 0.0f;
    // O^T accumulators: 8 m-tiles of 16 dimensions x NT n-tiles of 8 heads
    float o[8][NT][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i)
                o[mt][nt][i] = 0.0f;
    float m_run[2] = {-INFINITY, -INFINITY};
    float l_run[2] = {0.0f, 0.0f};

    // chunk c of this CTA's range: keys k_begin + 32 c .. + 31 = half
    // ((k_begin / 32 + c) % 2) of page (k_begin / 64 + c / 2)
    // page ids of this warp's first 32 chunks, one per lane, read once
    int my_pg = 0;
    if (warp + ATT_WARPS * lane < n_chunks)
    {
        const int32_t *bt = a.block_table + (int64_t)b * a.max_pages + (k_begin + 32 * (warp + ATT_WARPS * lane)) / KV_P;
        my_pg = in_span(NV4_SITE(0), a.sp_block_table, bt, 4) ? *bt : 0;
    }
    // warp-collective (the page id comes from a shuffle); one copy per half page
    auto issue = [&](int c, int s) {
        const int i = (c - warp) / ATT_WARPS;
        const int tok = k_begin + 32 * c;
        int page = __shfl_sync(0xFFFFFFFFu, my_pg, i & 31);
        if (i >= 32)
            page = in_span(NV4_SITE(0), a.sp_block_table, a.block_table + (int64_t)b * a.max_pages + tok / KV_P, 4)
                       ? a.block_table[(int64_t)b * a.max_pages + tok / KV_P]
                       : 0;
        const int64_t ph = (int64_t)min(max(page, 0), a.num_pages - 1) * a.H_kv + hk;
        const int half = (tok / 32) & 1;
        if (lane == 0) {
            mbar_arrive_expect_tx(&sm.full[warp][s], 2 * HALF8_BYTES);
            if (in_span(NV4_SITE(0), a.sp_pages, a.pages + ph * PAGE8_BYTES + half * (2 * HALF8_BYTES),
                        2 * HALF8_BYTES))
                bulk_load(sm.unit[warp][s], a.pages + ph * PAGE8_BYTES + half * (2 * HALF8_BYTES), 2 * HALF8_BYTES,
                          &sm.full[warp][s]);
        }
    };
    for (int i = 0; i < ATT_STAGES && warp + i * ATT_WARPS < n_chunks; ++i)
        issue(warp + i * ATT_WARPS, i);
    bool ok = true;
    int it = 0;
    for (int c = warp; c < n_chunks; c += ATT_WARPS, ++it) {
        const int s = it % ATT_STAGES;
        const uint32_t par = (uint32_t)(it / ATT_STAGES) & 1u;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&sm.full[warp][s], par, a.timeout_ns, nullptr))) {
            if (lane == 0)
                atomicOr(a.status, ST_TIMEOUT);
            ok = false;
            break;
        }
        const uint8_t *kc = sm.unit[warp][s];      // [8 dim chunks][32 key slots][16]
        const uint8_t *vc = kc + HALF8_BYTES;      // [2 token groups][128 dims][16]
        const int valid = min(32, k_end - (k_begin + 32 * c));
        // ---- S = Q K^T over 32 keys
        float sc[4][4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            // matrix i of the two loads: dim chunk i (4 + i) of slots 8 j .. 8 j + 7
            const uint8_t *krow = kc + ((lane >> 3) * 32 + 8 * j + (lane & 7)) * 16;
            uint32_t kr[8];
            ldsm_x4(krow, *reinterpret_cast<uint32_t(*)[4]>(&kr[0]));
            ldsm_x4(krow + 4 * 32 * 16, *reinterpret_cast<uint32_t(*)[4]>(&kr[4]));
            sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.0f;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma16816(sc[j], qf[kk], h2_e4m3x2(kr[kk] & 0xFFFFu), h2_e4m3x2(kr[kk] >> 16));
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int i = 0; i < 4; ++i)
                sc[j][i] *= s_k;
        uint32_t pf[2][4];
        float corr[2];
        if (kv_softmax_chunk(sc, valid, t, chunk_key8, NT == 2, m_run, l_run, corr, pf))
            kv_rescale<NT>(o, corr, t);
        // ---- O^T += V^T P^T: A = value rows (8 m-tiles of 16 dims), B = P^T
        const bool full_chunk = valid >= 32;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            // matrix i: dims 16 mt + 8 (i & 1) + 0..7, keys 16 (i >> 1) .. + 15
            uint32_t vr[4];
            ldsm_x4(vc + ((lane >> 4) * KV_D + 16 * mt + 8 * ((lane >> 3) & 1) + (lane & 7)) * 16, vr);
#pragma unroll
            for (int st = 0; st < 2; ++st) {
                // rows g (vr[2 st]) and g + 8 (vr[2 st + 1]): keys 16 st + 4t + {0,1} / {2,3}
                uint32_t afr[4] = {h2_e4m3x2(vr[2 * st] & 0xFFFFu), h2_e4m3x2(vr[2 * st + 1] & 0xFFFFu),
                                   h2_e4m3x2(vr[2 * st] >> 16), h2_e4m3x2(vr[2 * st + 1] >> 16)};
                if (!full_chunk) {
                    const int nv = min(4, max(0, valid - 16 * st - 4 * t));
#pragma unroll
                    for (int r2 = 0; r2 < 2; ++r2) {
                        afr[r2] = nv >= 2 ? afr[r2] : (nv == 1 ? (afr[r2] & 0x0000FFFFu) : 0u);
                        afr[2 + r2] = nv >= 4 ? afr[2 + r2] : (nv == 3 ? (afr[2 + r2] & 0x0000FFFFu) : 0u);
                    }
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    mma16816(o[mt][nt], afr, pf[st][nt], pf[st][2 + nt]);
            }
        }
        __syncwarp();
        if (c + ATT_STAGES * ATT_WARPS < n_chunks) {
            fence_proxy_async_smem();
            issue(c + ATT_STAGES * ATT_WARPS, s);
        }
    }
    if (lane == 0 && !ok) {
        const int mine = n_chunks > warp ? (n_chunks - warp + ATT_WARPS - 1) / ATT_WARPS : 0;
        for (int i = it; i < mine && i < it + ATT_STAGES; ++i)
            mbar_wait(&sm.full[warp][i % ATT_STAGES], (uint32_t)(i / ATT_STAGES) & 1u, a.timeout_ns, nullptr);
    }
    kv_merge_and_store(a, sm.merge, o, m_run, l_run, warp, g, t, G, b, hk, split, s_v);
}

// Merge of the splits: o = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s.
__global__ void kv_combine_kernel(const KvAttnArgs a)
{
    const int64_t hq = blockIdx.x; // b * H + h
    const int d = threadIdx.x;
    const float *part = a.partial + hq * a.n_splits * (KV_D + 2);
    if (!in_span(NV4_SITE(0), a.sp_partial, part, (uint64_t)a.n_splits * (KV_D + 2) * 4) ||
        !in_span(NV4_SITE(0), a.sp_v_scale, a.v_scale, 4))
        return;
    float M = -INFINITY;
    for (int s = 0; s < a.n_splits; ++s)
        M = fmaxf(M, part[s * (KV_D + 2) + KV_D]);
    float L = 0.0f, O = 0.0f;
    if (M != -INFINITY)
        for (int s = 0; s < a.n_splits; ++s) {
            const float ms = part[s * (KV_D + 2) + KV_D];
            const float f = ms == -INFINITY ? 0.0f : exp2f(ms - M);
            L += f * part[s * (KV_D + 2) + KV_D + 1];
            O += f * part[s * (KV_D + 2) + d];
        }
    const float y = L > 0.0f ? O * *a.v_scale / L : 0.0f;
    if (a.out_dtype == NVFP4_OUT_BF16) {
        if (in_span(NV4_SITE(0), a.sp_out, static_cast<__nv_bfloat16 *>(a.out) + hq * KV_D + d, 2))
            static_cast<__nv_bfloat16 *>(a.out)[hq * KV_D + d] = __float2bfloat16_rn(y);
    } else if (in_span(NV4_SITE(0), a.sp_out, static_cast<float *>(a.out) + hq * KV_D + d, 4)) {
        static_cast<float *>(a.out)[hq * KV_D + d] = y;
    }
}

} // namespace

cudaError_t launch_kv_append(const KvAppendArgs &args, cudaStream_t stream)
{
    const int64_t threads = (int64_t)args.B * args.H_kv * 2 * (KV_D / 16);
    if (threads == 0)
        return cudaSuccess;
    KvAppendArgs a = args;
    const uint64_t page_bytes = a.fmt == KV_FMT_FP8 ? PAGE8_BYTES : PAGE_BYTES;
    a.sp_k_new = span_of(a.k_new, 2u * (uint64_t)a.B * a.H_kv * KV_D);
    a.sp_v_new = span_of(a.v_new, 2u * (uint64_t)a.B * a.H_kv * KV_D);
    a.sp_positions = span_of(a.positions, 4u * (uint64_t)a.B);
    a.sp_block_table = span_of(a.block_table, 4u * (uint64_t)a.B * a.max_pages);
    a.sp_pages = span_of(a.pages, page_bytes * (uint64_t)a.num_pages * a.H_kv);
    a.sp_k_scale = span_of(a.k_scale, 4);
    a.sp_v_scale = span_of(a.v_scale, 4);
    kv_append_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, stream>>>(a);
    return cudaGetLastError();
}

int kv_ctas_per_sm(int fmt, int64_t group)
{
    // NVFP4, one n-tile: 36 KB of ring and <= 128 registers a thread; FP8
    // (64 KB of ring) and two n-tiles (more registers): 3
    return fmt == KV_FMT_NVFP4 && group <= 8 ? 4 : 3;
}

void kv_attn_splits(int64_t B, int64_t H_kv, int64_t max_ctx, int sms, int ctas_per_sm, int &n_splits,
                    int &keys_per_split)
{
    // as many splits as keep every (sequence, KV head) CTA of the grid in one
    // wave of ctas_per_sm CTAs per SM
    const int64_t units = std::max<int64_t>(1, B * H_kv);
    int64_t ns = std::max<int64_t>(1, (int64_t)ctas_per_sm * sms / units);
    ns = std::min<int64_t>(ns, std::max<int64_t>(1, (max_ctx + 255) / 256));
    int64_t kps = (std::max<int64_t>(max_ctx, 1) + ns - 1) / ns;
    kps = (kps + KV_P - 1) / KV_P * KV_P;
    n_splits = (int)std::max<int64_t>(1, (max_ctx + kps - 1) / kps);
    keys_per_split = (int)kps;
}

size_t kv_attn_partial_bytes(int B, int H, int n_splits)
{
    return n_splits > 1 ? (size_t)B * H * n_splits * (KV_D + 2) * sizeof(float) : 0;
}

cudaError_t launch_kv_decode(const KvAttnArgs &args, cudaStream_t stream)
{
    KvAttnArgs a = args;
    const uint64_t page_bytes = a.fmt == KV_FMT_FP8 ? PAGE8_BYTES : PAGE_BYTES;
    a.sp_q = span_of(a.q, 2u * (uint64_t)a.B * a.H * KV_D);
    a.sp_ctx_lens = span_of(a.ctx_lens, 4u * (uint64_t)a.B);
    a.sp_block_table = span_of(a.block_table, 4u * (uint64_t)a.B * a.max_pages);
    a.sp_pages = span_of(a.pages, page_bytes * (uint64_t)a.num_pages * a.H_kv);
    a.sp_k_scale = span_of(a.k_scale, 4);
    a.sp_v_scale = span_of(a.v_scale, 4);
    a.sp_out = span_of(a.out, (a.out_dtype == NVFP4_OUT_BF16 ? 2u : 4u) * (uint64_t)a.B * a.H * KV_D);
    a.sp_partial = span_of(a.partial, kv_attn_partial_bytes(a.B, a.H, a.n_splits));
    const size_t smem = a.fmt == KV_FMT_FP8 ? sizeof(AttSmem8) : sizeof(AttSmem4);
    cudaError_t e;
    // one n-tile of 8 heads when a group has at most 8 query heads, else two
    const bool two = a.H / a.H_kv > 8;
    auto kern = a.fmt == KV_FMT_FP8 ? (two ? kv_decode_fp8_kernel<2> : kv_decode_fp8_kernel<1>)
                                    : (two ? kv_decode_kernel<2> : kv_decode_kernel<1>);
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
        return e;
    dim3 grid((unsigned)a.n_splits, (unsigned)a.H_kv, (unsigned)a.B);
    kern<<<grid, 32 * ATT_WARPS, smem, stream>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess || a.n_splits == 1)
        return e;
    kv_combine_kernel<<<(unsigned)(a.B * a.H), KV_D, 0, stream>>>(a);
    return cudaGetLastError();
}

} // namespace nv4
