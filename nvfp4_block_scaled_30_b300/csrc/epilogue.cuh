// Output stores shared by the W4A4 GEMM epilogues: 32 consecutive
// accumulator columns of one row as BF16/FP32 (alpha-scaled), and the NVFP4
// encode of such a run (the fused next-layer quantiser).
#pragma once
#include <cstdint>
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace nv4 {

// Where element (i, j) of the output goes: out[i * ld_i + j * ld_j]; vec_ok
// 1 when ld_j == 1 and 16-byte vector stores of a row are aligned, 2 when
// 32-byte ones are too; span: the output's bytes (tested in the
// bounds-checked build).
struct OutDesc {
    void *out;
    int64_t ld_i, ld_j;
    int32_t out_dtype, vec_ok;
    Span span;
};

// Host: OutDesc.vec_ok of an output at `out` with strides (ld_i, ld_j) in
// elements of esz bytes.
inline int32_t out_vec_level(const void *out, int64_t ld_i, int64_t ld_j, int esz)
{
    if (ld_j != 1)
        return 0;
    const uintptr_t a = reinterpret_cast<uintptr_t>(out);
    if ((ld_i * esz) % 32 == 0 && a % 32 == 0)
        return 2;
    return ((ld_i * esz) % 16 == 0 && a % 16 == 0) ? 1 : 0;
}

// Spans of an NVFP4 output's codes and tiled scales.
struct QSpans {
    Span codes, scales;
};

// Row i, columns j0 .. j0 + 31 (bits of the FP32 accumulator in v) times
// alpha; rows >= i_end and columns >= j_end are not stored.
__device__ __forceinline__ void store_chunk32(const OutDesc &o, const uint32_t (&v)[32], int64_t i, int64_t j0,
                                              float alpha, int64_t i_end, int64_t j_end)
{
    if (i >= i_end)
        return;
    if (o.ld_j == 1 && o.vec_ok && j0 + 32 <= j_end) {
        if (o.out_dtype == NVFP4_OUT_BF16) {
            uint4 *d = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(o.out) + i * o.ld_i + j0);
            if (!in_span(NV4_SITE(2), o.span, d, 64))
                return;
#pragma unroll
            for (int c = 0; c < 32; c += 8) {
                uint32_t w[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    __nv_bfloat162 h = __floats2bfloat162_rn(alpha * __uint_as_float(v[c + 2 * q]),
                                                             alpha * __uint_as_float(v[c + 2 * q + 1]));
                    w[q] = *reinterpret_cast<uint32_t *>(&h);
                }
                d[c / 8] = make_uint4(w[0], w[1], w[2], w[3]);
            }
        } else {
            float4 *d = reinterpret_cast<float4 *>(static_cast<float *>(o.out) + i * o.ld_i + j0);
            if (!in_span(NV4_SITE(2), o.span, d, 128))
                return;
#pragma unroll
            for (int c = 0; c < 32; c += 4)
                d[c / 4] = make_float4(alpha * __uint_as_float(v[c]), alpha * __uint_as_float(v[c + 1]),
                                       alpha * __uint_as_float(v[c + 2]), alpha * __uint_as_float(v[c + 3]));
        }
        return;
    }
#pragma unroll
    for (int c = 0; c < 32; ++c) {
        const int64_t j = j0 + c;
        if (j < j_end) {
            const float y = alpha * __uint_as_float(v[c]);
            const int64_t off = i * o.ld_i + j * o.ld_j;
            if (o.out_dtype == NVFP4_OUT_BF16) {
                if (in_span(NV4_SITE(2), o.span, static_cast<__nv_bfloat16 *>(o.out) + off, 2))
                    static_cast<__nv_bfloat16 *>(o.out)[off] = __float2bfloat16_rn(y);
            } else if (in_span(NV4_SITE(2), o.span, static_cast<float *>(o.out) + off, 4)) {
                static_cast<float *>(o.out)[off] = y;
            }
        }
    }
}

// 256-bit global store (sm_100 and later): one whole 32-byte sector.
__device__ __forceinline__ void st_global_v8(void *ptr, const uint32_t (&r)[8])
{
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(ptr), "r"(r[0]), "r"(r[1]),
                 "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}

// One warp's rows r0 .. r0 + 31 (lane l holds row r0 + l), a run of 64
// bytes per row in w (two 32-byte pieces of 8 words), stored so that each
// store instruction writes whole runs of 16 rows.  Lane l stores piece l % 2
// of row 16 s + l / 2 in instruction s; in exchange round a the lanes holding
// rows of instruction s = a ^ (l % 2) send, each source lane the piece its
// receiver stores, so every round moves 32 distinct words per word index (a
// transpose by shuffles, no shared memory).  Rows outside [i_lo, i_hi) are
// not stored; row i's run starts at base + i * row_bytes.  Every lane of the
// warp calls this.
__device__ __forceinline__ void store_rows64(const uint32_t (&w)[16], uint8_t *base, int64_t row_bytes, int64_t r0,
                                             int64_t i_lo, int64_t i_hi, const Span &span, int lane)
{
    const int piece = lane & 1;  // the piece this lane stores
    const int rsub = lane >> 1;  // its row within an instruction's 16 rows
    const int s_own = lane >> 4; // the instruction this lane's own row goes out in
    uint32_t o[2][8];
#pragma unroll
    for (int a = 0; a < 2; ++a) {
        const int src = 16 * (a ^ piece) + rsub;
        const bool give1 = (s_own ^ a) != 0; // the receiver stores piece 1
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint32_t got = __shfl_sync(0xFFFFFFFFu, give1 ? w[8 + k] : w[k], src);
            if ((a ^ piece) == 0)
                o[0][k] = got;
            else
                o[1][k] = got;
        }
    }
#pragma unroll
    for (int s = 0; s < 2; ++s) {
        const int64_t i = r0 + 16 * s + rsub;
        uint8_t *d = base + i * row_bytes + 32 * piece;
        if (i >= i_lo && i < i_hi && in_span(NV4_SITE(2), span, d, 32))
            st_global_v8(d, o[s]);
    }
}

// The BF16 words of 32 consecutive columns of one row: accumulator bits v
// times alpha, two columns per word.
__device__ __forceinline__ void pack_bf16x32(const uint32_t (&v)[32], float alpha, uint32_t (&w)[16])
{
#pragma unroll
    for (int q = 0; q < 16; ++q) {
        __nv_bfloat162 h =
            __floats2bfloat162_rn(alpha * __uint_as_float(v[2 * q]), alpha * __uint_as_float(v[2 * q + 1]));
        w[q] = *reinterpret_cast<uint32_t *>(&h);
    }
}

// Whether one warp's rows can go out through store_rows64 for the run of 32
// columns at j0: 32-byte aligned rows (vec_ok == 2), unit column stride and
// the whole run inside the output (warp-uniform).
__device__ __forceinline__ bool rows64_ok(const OutDesc &o, int64_t j0, int64_t j_end)
{
    return o.ld_j == 1 && o.vec_ok == 2 && j0 + 32 <= j_end;
}

// Rows r0 .. r0 + 31 of one warp (lane l: row r0 + l, accumulator bits of
// columns j0 .. j0 + 31 in v) times alpha (each lane its own), rows outside
// [i_lo, i_hi) and columns >= j_end not stored: by store_rows64 (BF16 as one
// 64-byte run per row, FP32 as two) when rows64_ok, else row by row through
// store_chunk32.  Every lane calls this.
__device__ __forceinline__ void store_chunk32_warp(const OutDesc &o, const uint32_t (&v)[32], int64_t r0,
                                                   int64_t i_lo, int64_t i_hi, int64_t j0, float alpha,
                                                   int64_t j_end, int lane)
{
    if (r0 >= i_hi || r0 + 32 <= i_lo) // no row of this warp is stored (warp-uniform)
        return;
    if (rows64_ok(o, j0, j_end)) {
        if (o.out_dtype == NVFP4_OUT_BF16) {
            uint32_t w[16];
            pack_bf16x32(v, alpha, w);
            store_rows64(w, reinterpret_cast<uint8_t *>(static_cast<__nv_bfloat16 *>(o.out) + j0), o.ld_i * 2, r0,
                         i_lo, i_hi, o.span, lane);
        } else {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t w[16];
#pragma unroll
                for (int q = 0; q < 16; ++q)
                    w[q] = __float_as_uint(alpha * __uint_as_float(v[16 * h + q]));
                store_rows64(w, reinterpret_cast<uint8_t *>(static_cast<float *>(o.out) + j0 + 16 * h), o.ld_i * 4,
                             r0, i_lo, i_hi, o.span, lane);
            }
        }
        return;
    }
    const int64_t i = r0 + lane;
    store_chunk32(o, v, i, j0, alpha, i >= i_lo ? i_hi : i, j_end);
}

// NVFP4 store of 32 consecutive outputs y (binary32 bits in v) of one row
// starting at column j0 (two 16-element blocks): the block encode of the
// quantisers under the given tensor scale s, 8 code bytes at crow + j0/2 and
// one scale byte per block in the row's MMA-tiled scale slots srow (see
// q_row_addr).  Returns the largest |y|.
__device__ __forceinline__ float encode_store_q(const uint32_t (&v)[32], uint8_t *crow, uint8_t *srow, int j0,
                                                float s, const QSpans &qs)
{
    float m = 0.0f;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        float amb = 0.0f;
#pragma unroll
        for (int t = 0; t < 16; ++t)
            amb = fmaxf(amb, fabsf(__uint_as_float(v[16 * h + t])));
        const uint32_t e = block_scale_code(amb, s);
        const float r = recip_step(__fmul_rn(e4m3_value(e), s));
        float q[16];
#pragma unroll
        for (int t = 0; t < 16; ++t)
            q[t] = __fmul_rn(__uint_as_float(v[16 * h + t]), r);
        const uint32_t pk[2] = {e2m1x8(q[0], q[1], q[2], q[3], q[4], q[5], q[6], q[7]),
                                e2m1x8(q[8], q[9], q[10], q[11], q[12], q[13], q[14], q[15])};
        const int j = j0 + 16 * h;
        if (in_span(NV4_SITE(2), qs.codes, crow + j / 2, 8))
            *reinterpret_cast<uint2 *>(crow + j / 2) = make_uint2(pk[0], pk[1]);
        const int blk = j / 16;
        if (in_span(NV4_SITE(2), qs.scales, srow + (blk >> 2) * 512 + (blk & 3), 1))
            srow[(blk >> 2) * 512 + (blk & 3)] = (uint8_t)e;
        m = fmaxf(m, amb);
    }
    return m;
}

// Row i of an NVFP4 output of n columns (codes [rows][n/2], MMA-tiled
// scales): its code row and the base of its scale slots (byte (i % 32) * 16
// + ((i % 128) / 32) * 4 + b % 4 of atom (i / 128) * (n / 64) + b / 4 holds
// block b).
__device__ __forceinline__ void q_row_addr(int64_t i, int64_t n, uint8_t *codes, uint8_t *scales, uint8_t *&crow,
                                           uint8_t *&srow)
{
    const int64_t r7 = i & 127;
    crow = codes + i * (n / 2);
    srow = scales + (i >> 7) * (n / 64) * 512 + (r7 & 31) * 16 + (r7 >> 5) * 4;
}

// Zero scale bytes of 32 columns from j in a padding row's scale slots (rows
// of the last 128-row tile past the real rows, as the quantisers leave them).
__device__ __forceinline__ void zero_pad_scales32(uint8_t *srow, int j, const QSpans &qs)
{
    uint8_t *b = srow + (j >> 6) * 512 + ((j >> 4) & 3);
    if (in_span(NV4_SITE(2), qs.scales, b, 2)) {
        b[0] = 0;
        b[1] = 0;
    }
}

} // namespace nv4
