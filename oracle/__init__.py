"""CPU oracle for the NVFP4 hot path (numpy front end over liboracle.so).

TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and
bench.py's CPU-baseline / reference legs may import this package.  It shares
no code with the CUDA path (nvfp4_block_scaled_30_b300), and neither imports
the other.  Every function follows a passage of the pages named in
nvfp4_oracle.c; the readings taken where the pages are silent are listed
there.

Layouts: activations/weights are BF16 bit patterns (uint16) [rows, K];
codes are uint8 [rows, K/2] with the even element in the low nibble; scales
are E4M3 bytes [rows, K/16] row-major; the second-level scale is one float32
(per-tensor mode) or binary16 bits [rows, K/256] (macro mode).
"""
import ctypes
import os

import numpy as np

from . import build as _build

_LIB = None

_u8 = np.ctypeslib.ndpointer(np.uint8, flags="C_CONTIGUOUS")
_u16 = np.ctypeslib.ndpointer(np.uint16, flags="C_CONTIGUOUS")
_i32 = np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS")
_i64 = np.ctypeslib.ndpointer(np.int64, flags="C_CONTIGUOUS")
_f32 = np.ctypeslib.ndpointer(np.float32, flags="C_CONTIGUOUS")
_f64 = np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")
_I64 = ctypes.c_int64
_F = ctypes.c_float
_VP = ctypes.c_void_p

ORC_OK, ORC_ERR_ARG, ORC_ERR_NONFINITE = 0, 1, 3


class OracleError(ValueError):
    pass


def lib():
    global _LIB
    if _LIB is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        L.orc_e2m1_value.restype = ctypes.c_double
        L.orc_e2m1_value.argtypes = [ctypes.c_uint32]
        L.orc_e2m1_encode.restype = ctypes.c_uint32
        L.orc_e2m1_encode.argtypes = [ctypes.c_float]
        L.orc_e4m3_value.restype = ctypes.c_double
        L.orc_e4m3_value.argtypes = [ctypes.c_uint32]
        L.orc_e4m3_encode.restype = ctypes.c_uint32
        L.orc_e4m3_encode.argtypes = [ctypes.c_float]
        L.orc_fp16_value.restype = ctypes.c_double
        L.orc_fp16_value.argtypes = [ctypes.c_uint32]
        L.orc_fp16_encode.restype = ctypes.c_uint32
        L.orc_fp16_encode.argtypes = [ctypes.c_float]
        L.orc_bf16_value.restype = ctypes.c_float
        L.orc_bf16_value.argtypes = [ctypes.c_uint32]
        L.orc_e2m1_encode_array.restype = None
        L.orc_e2m1_encode_array.argtypes = [_f32, _I64, _u8]
        L.orc_e4m3_encode_array.restype = None
        L.orc_e4m3_encode_array.argtypes = [_f32, _I64, _u8]
        L.orc_nvfp4_encode.restype = ctypes.c_int
        L.orc_nvfp4_encode.argtypes = [_u16, _I64, _I64, _I64, _u8, _u8, _f32]
        L.orc_nvfp4_encode_macro.restype = ctypes.c_int
        L.orc_nvfp4_encode_macro.argtypes = [_u16, _I64, _I64, _I64, _u8, _u8, _u16]
        L.orc_nvfp4_encode_f32_scaled.restype = ctypes.c_int
        L.orc_nvfp4_encode_f32_scaled.argtypes = [_f32, _I64, _I64, _I64, ctypes.c_float, _u8, _u8]
        L.orc_fp8_token_encode.restype = ctypes.c_int
        L.orc_fp8_token_encode.argtypes = [_u16, _I64, _I64, _I64, _u8, _f32]
        L.orc_nvfp4_dequant.restype = None
        L.orc_nvfp4_dequant.argtypes = [_u8, _u8, _F, _I64, _I64, _f64]
        L.orc_nvfp4_dequant_macro.restype = None
        L.orc_nvfp4_dequant_macro.argtypes = [_u8, _u8, _u16, _I64, _I64, _f64]
        L.orc_gemm_w4a4.restype = None
        L.orc_gemm_w4a4.argtypes = [_u8, _u8, _F, _u8, _u8, _F, _I64, _I64, _I64,
                                    _VP, _I64, _f64]
        L.orc_gemm_w4a4_macro.restype = None
        L.orc_gemm_w4a4_macro.argtypes = [_u8, _u8, _u16, _u8, _u8, _u16, _I64, _I64,
                                          _I64, _VP, _I64, _f64]
        L.orc_gemm_w4a8.restype = None
        L.orc_gemm_w4a8.argtypes = [_u8, _f32, _u8, _u8, _F, _I64, _I64, _I64, _VP,
                                    _I64, _f64]
        L.orc_gemm_grouped_w4a4.restype = None
        L.orc_gemm_grouped_w4a4.argtypes = [_u8, _u8, _F, _VP, _i64, _I64, _u8, _u8,
                                            _f32, _I64, _I64, _f64]
        _LIB = L
    return _LIB


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


def _check(rc):
    if rc == ORC_ERR_NONFINITE:
        raise OracleError("non-finite input")
    if rc != ORC_OK:
        raise OracleError(f"invalid argument (status {rc})")


# ---- element formats --------------------------------------------------------

def e2m1_value(code):
    return lib().orc_e2m1_value(int(code))


def e2m1_encode(q):
    return lib().orc_e2m1_encode(float(q))


def e4m3_value(code):
    return lib().orc_e4m3_value(int(code))


def e4m3_encode(u):
    return lib().orc_e4m3_encode(float(u))


def e2m1_encode_array(v):
    v = _c(v, np.float32).ravel()
    out = np.empty(v.size, np.uint8)
    lib().orc_e2m1_encode_array(v, v.size, out)
    return out


def e4m3_encode_array(v):
    v = _c(v, np.float32).ravel()
    out = np.empty(v.size, np.uint8)
    lib().orc_e4m3_encode_array(v, v.size, out)
    return out


def fp16_value(h):
    return lib().orc_fp16_value(int(h))


def fp16_encode(v):
    return lib().orc_fp16_encode(float(v))


def bf16_value(b):
    return lib().orc_bf16_value(int(b))


# ---- encoders -----------------------------------------------------------------

def bf16_round(y):
    """BF16 bits (uint16) of a layer output: y rounded to the nearest binary32
    value, then to BF16 with round-to-nearest-even on the 16 dropped bits (the
    output format of the W4A4 / W4A8 layers; finite inputs).  Used between
    the layers of the chained policy stack."""
    f = np.asarray(y, np.float64).astype(np.float32)
    if not np.isfinite(f).all():
        raise OracleError("bf16_round: non-finite value")
    b = f.view(np.uint32).astype(np.uint64)
    r = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def nvfp4_encode(x_bf16):
    """Per-tensor NVFP4 encode of a BF16-bit array [R, K].

    Returns (codes uint8 [R, K/2], scales uint8 [R, K/16], s_g float32)."""
    x = _c(x_bf16, np.uint16)
    R, K = x.shape
    codes = np.zeros((R, K // 2), np.uint8)
    scales = np.zeros((R, K // 16), np.uint8)
    sg = np.zeros(1, np.float32)
    _check(lib().orc_nvfp4_encode(x, R, K, K, codes, scales, sg))
    return codes, scales, np.float32(sg[0])


def nvfp4_encode_f32_scaled(x_f32, s_g):
    """Per-tensor NVFP4 encode of binary32 values [R, K] under a GIVEN tensor
    scale s_g (no amax pass).  Returns (codes [R, K/2], scales [R, K/16])."""
    x = _c(x_f32, np.float32)
    R, K = x.shape
    codes = np.zeros((R, K // 2), np.uint8)
    scales = np.zeros((R, K // 16), np.uint8)
    _check(lib().orc_nvfp4_encode_f32_scaled(x, R, K, K, np.float32(s_g), codes, scales))
    return codes, scales


def nvfp4_encode_macro(x_bf16):
    """Macro-mode NVFP4 encode: returns (codes, scales, macro fp16 bits [R, K/256])."""
    x = _c(x_bf16, np.uint16)
    R, K = x.shape
    codes = np.zeros((R, K // 2), np.uint8)
    scales = np.zeros((R, K // 16), np.uint8)
    macro = np.zeros((R, max(K // 256, 0)), np.uint16)
    _check(lib().orc_nvfp4_encode_macro(x, R, K, K, codes, scales, macro))
    return codes, scales, macro


def fp8_token_encode(x_bf16):
    """Per-token FP8 encode: returns (E4M3 bytes [R, K], s_t float32 [R])."""
    x = _c(x_bf16, np.uint16)
    R, K = x.shape
    a = np.zeros((R, K), np.uint8)
    st = np.zeros(R, np.float32)
    _check(lib().orc_fp8_token_encode(x, R, K, K, a, st))
    return a, st


def nvfp4_dequant(codes, scales, s_g):
    codes, scales = _c(codes, np.uint8), _c(scales, np.uint8)
    R, K = codes.shape[0], codes.shape[1] * 2
    out = np.zeros((R, K), np.float64)
    lib().orc_nvfp4_dequant(codes, scales, float(s_g), R, K, out)
    return out


def nvfp4_dequant_macro(codes, scales, macro):
    codes, scales, macro = _c(codes, np.uint8), _c(scales, np.uint8), _c(macro, np.uint16)
    R, K = codes.shape[0], codes.shape[1] * 2
    out = np.zeros((R, K), np.float64)
    lib().orc_nvfp4_dequant_macro(codes, scales, macro, R, K, out)
    return out


# ---- contractions -------------------------------------------------------------

def _rows(rows, M):
    if rows is None:
        return None, M
    r = _c(rows, np.int64)
    if r.size and (r.min() < 0 or r.max() >= M):
        raise OracleError("row index out of range")
    return r, r.size


def gemm_w4a4(a, w, rows=None):
    """a, w: (codes, scales, s_g) tuples.  Returns float64 Y [len(rows) or M, N]."""
    ac, as_, asg = _c(a[0], np.uint8), _c(a[1], np.uint8), float(a[2])
    wc, ws, wsg = _c(w[0], np.uint8), _c(w[1], np.uint8), float(w[2])
    M, N, K = ac.shape[0], wc.shape[0], ac.shape[1] * 2
    if wc.shape[1] * 2 != K:
        raise OracleError("K mismatch")
    r, nr = _rows(rows, M)
    Y = np.zeros((nr, N), np.float64)
    lib().orc_gemm_w4a4(ac, as_, asg, wc, ws, wsg, M, N, K,
                        None if r is None else r.ctypes.data, nr, Y)
    return Y


def gemm_w4a4_macro(a, w, rows=None):
    """a, w: (codes, scales, macro) tuples in macro mode."""
    ac, as_, am = _c(a[0], np.uint8), _c(a[1], np.uint8), _c(a[2], np.uint16)
    wc, ws, wm = _c(w[0], np.uint8), _c(w[1], np.uint8), _c(w[2], np.uint16)
    M, N, K = ac.shape[0], wc.shape[0], ac.shape[1] * 2
    r, nr = _rows(rows, M)
    Y = np.zeros((nr, N), np.float64)
    lib().orc_gemm_w4a4_macro(ac, as_, am, wc, ws, wm, M, N, K,
                              None if r is None else r.ctypes.data, nr, Y)
    return Y


def gemm_w4a8(a_fp8, s_t, w, rows=None):
    a, st = _c(a_fp8, np.uint8), _c(s_t, np.float32)
    wc, ws, wsg = _c(w[0], np.uint8), _c(w[1], np.uint8), float(w[2])
    M, K, N = a.shape[0], a.shape[1], wc.shape[0]
    r, nr = _rows(rows, M)
    Y = np.zeros((nr, N), np.float64)
    lib().orc_gemm_w4a8(a, st, wc, ws, wsg, M, N, K,
                        None if r is None else r.ctypes.data, nr, Y)
    return Y


def gemm_grouped_w4a4(a, row_idx, offsets, w_codes, w_scales, w_sg):
    """a: (codes, scales, s_g); row_idx int32 [T] or None; offsets int64 [E+1];
    w_codes uint8 [E, N, K/2]; w_scales uint8 [E, N, K/16]; w_sg float32 [E]."""
    ac, as_, asg = _c(a[0], np.uint8), _c(a[1], np.uint8), float(a[2])
    off = _c(offsets, np.int64)
    wc, ws, wsg = _c(w_codes, np.uint8), _c(w_scales, np.uint8), _c(w_sg, np.float32)
    E, N, K = wc.shape[0], wc.shape[1], wc.shape[2] * 2
    T = int(off[-1])
    ridx = None
    if row_idx is not None:
        ridx = _c(row_idx, np.int32)
        if ridx.size != T or (T and (ridx.min() < 0 or ridx.max() >= ac.shape[0])):
            raise OracleError("bad row_idx")
    elif T > ac.shape[0]:
        raise OracleError("offsets exceed activation rows")
    Y = np.zeros((T, N), np.float64)
    lib().orc_gemm_grouped_w4a4(ac, as_, asg, None if ridx is None else ridx.ctypes.data,
                                off, E, wc, ws, wsg, N, K, Y)
    return Y


def gemm_grouped_w4a8(a_fp8, s_t, row_idx, offsets, w_codes, w_scales, w_sg):
    """Grouped W4A8: the W4A8 contraction per expert over its routed rows
    (the W4A8 path covers MoE operations as well as dense ones: "llama.cpp
    Put Precision Policy Inside the Model", section "One model can need more
    than one precision").  a_fp8 uint8 [T, K] with per-token scales s_t
    float32 [T]; row_idx int32 [R] or None; offsets int64 [E+1]; weights as
    for gemm_grouped_w4a4.  Returns float64 [R, N]:
    Y[j] = s_t[row(j)] * s_w[e] * sum_k E4M3(a[row(j), k]) * w_e[n, k]."""
    off = _c(offsets, np.int64)
    wc, ws, wsg = _c(w_codes, np.uint8), _c(w_scales, np.uint8), _c(w_sg, np.float32)
    T = int(off[-1])
    Y = np.zeros((T, wc.shape[1]), np.float64)
    for e in range(wc.shape[0]):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi > lo:
            rows = np.arange(lo, hi) if row_idx is None else _c(row_idx, np.int32)[lo:hi].astype(np.int64)
            Y[lo:hi] = gemm_w4a8(a_fp8, s_t, (wc[e], ws[e], wsg[e]), rows=rows)
    return Y


# ---- mixture-of-experts feed-forward around the grouped contraction ------------
#
# The pages name MoE models (Qwen3 MoE variants) and MoE operations on the
# NVFP4/W4A8 paths ("llama.cpp Put Precision Policy Inside the Model",
# section "One model can need more than one precision"; "AdaLLM
# Breakthrough", model list) but print no expert formula.  Reading taken:
# the experts of those models are SwiGLU feed-forward blocks
#   h = SiLU(x W_gate^T) * (x W_up^T),   y_e(x) = h W_down^T,
# and a token's output is the gate-weighted sum of its routed experts'
# outputs, y(t) = sum_k g_k(t) y_{e_k(t)}(x_t).  Both products are the grouped
# W4A4 contraction above; the element-wise steps run in FP64.

def silu(x):
    """SiLU(x) = x * sigmoid(x) = x / (1 + exp(-x)) in FP64."""
    x = np.asarray(x, np.float64)
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(-x))


def moe_up_swiglu(a, row_idx, offsets, gate, up, w_sg):
    """SwiGLU expert up projection of the routed rows.

    a: (codes, scales, s_g) activations; row_idx int32 [R] (activation row of
    routed row j) or None; offsets int64 [E+1]; gate, up: (codes uint8
    [E, I, K/2], scales uint8 [E, I, K/16]) of each expert's gate and up
    weights, quantised together under the tensor scale w_sg[e].
    Returns h float64 [R, I] = SiLU(G) * U with G, U the grouped products."""
    G = gemm_grouped_w4a4(a, row_idx, offsets, gate[0], gate[1], w_sg)
    U = gemm_grouped_w4a4(a, row_idx, offsets, up[0], up[1], w_sg)
    return silu(G) * U


def moe_down_combine(h, offsets, w_codes, w_scales, w_sg, token_idx, gate_w, T, y0=None):
    """Expert down projection and gate-weighted combine.

    h: (codes, scales, s_g) of the routed rows [R, I]; offsets int64 [E+1];
    w_codes/w_scales/w_sg: the experts' down weights as for
    gemm_grouped_w4a4; token_idx int32 [R] (token of routed row j); gate_w
    float32 [R] (routing weight of routed row j); T tokens.
    Returns y float64 [T, N]: y0 (or zeros) plus, for every routed row j,
    gate_w[j] * (h[j] W_e(j)^T) added to row token_idx[j]."""
    D = gemm_grouped_w4a4(h, None, offsets, w_codes, w_scales, w_sg)
    R = D.shape[0]
    tok = _c(token_idx, np.int32)[:R].astype(np.int64)
    g = _c(gate_w, np.float32)[:R].astype(np.float64)
    if R and (tok.min() < 0 or tok.max() >= T):
        raise OracleError("token index out of range")
    y = np.zeros((T, D.shape[1]), np.float64) if y0 is None else np.array(y0, np.float64, copy=True)
    np.add.at(y, tok, g[:, None] * D)
    return y


# ---- NVFP4 KV cache and decode attention ---------------------------------------
#
# "The FP4 Inflection" (section "What does this mean for model serving
# engines?") stores the KV cache in FP4 and names paged attention as the
# consumer; the TensorRT-LLM page's engine-build listing pages the KV cache in
# blocks of 64 tokens; "AdaLLM Breakthrough" pairs a low-precision KV cache
# with its own decode kernel.  None prints the cache encoding or the attention
# formula.  Readings taken: every cached key and value vector of one KV head
# (head_dim D elements) is encoded by the same block encoder as the
# activations -- 16-element blocks along D, E4M3 block scales, under a static
# FP32 tensor scale per cache tensor fixed beforehand (as for the fused
# output quantiser) -- and decode attention is the standard scaled dot-product
# attention of one query token over the sequence's cached tokens, with the
# query heads of a group sharing one KV head.

def bf16_to_f32(bits):
    """Exact binary32 values of BF16 bit patterns (a format conversion)."""
    b = np.ascontiguousarray(bits, np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)


def kv_encode(x_bf16, s):
    """KV-cache encode of BF16 vectors [n, D] under the static tensor scale s:
    the given-scale block encode of their exact binary32 values.
    Returns (codes uint8 [n, D/2], scales uint8 [n, D/16])."""
    return nvfp4_encode_f32_scaled(bf16_to_f32(x_bf16), s)


def kv_encode_fp8(x_bf16, s):
    """FP8 KV-cache encode ("AdaLLM Breakthrough" keeps an FP8 key-value
    cache; the per-token FP8 quantiser's rule under a static tensor scale s):
    code = E4M3_rne_sat(x * r) in binary32, r = 1/s (0 when s = 0, at most
    FLT_MAX).  Returns uint8 [n, D]."""
    x = bf16_to_f32(x_bf16)
    s = np.float32(s)
    if s == 0:
        r = np.float32(0)
    else:
        with np.errstate(over="ignore"):
            r = np.float32(1) / s
        r = np.minimum(r, np.float32(np.finfo(np.float32).max))
    prod = (x * r).astype(np.float32)
    return e4m3_encode_array(prod).reshape(x.shape)


def kv_gather_fp8(codes_pages, s, block_table_row, n_tokens, head):
    """Decoded FP64 vectors [n_tokens, D] of one sequence and KV head of an
    FP8 cache (codes_pages [pages, H_kv, P, D]): E4M3 value times s."""
    P = codes_pages.shape[2]
    rows = [codes_pages[int(block_table_row[t // P]), head, t % P] for t in range(n_tokens)]
    if not rows:
        return np.zeros((0, codes_pages.shape[3]))
    table = np.array([e4m3_value(c & 0x7F) * (-1.0 if c & 0x80 else 1.0) for c in range(256)])
    return table[np.stack(rows)] * float(np.float32(s))


def kv_gather(codes_pages, scales_pages, s, block_table_row, n_tokens, head):
    """Dequantised FP64 vectors [n_tokens, D] of one sequence and KV head from
    paged storage: token t lives in page block_table_row[t // P] at slot
    t % P (P = tokens per page); codes_pages [pages, H_kv, P, D/2]."""
    P = codes_pages.shape[2]
    rows_c, rows_s = [], []
    for t in range(n_tokens):
        pg = int(block_table_row[t // P])
        rows_c.append(codes_pages[pg, head, t % P])
        rows_s.append(scales_pages[pg, head, t % P])
    if not rows_c:
        return np.zeros((0, codes_pages.shape[3] * 2))
    return nvfp4_dequant(np.stack(rows_c), np.stack(rows_s), s)


def decode_attention(q, k_cache, v_cache, s_k, s_v, block_table, ctx_lens, sm_scale, fmt="nvfp4"):
    """One decode step of scaled dot-product attention over an NVFP4 paged KV
    cache, in FP64.

    q: float [B, H, D] (the BF16 queries' exact values); k_cache / v_cache:
    (codes [pages, H_kv, P, D/2], scales [pages, H_kv, P, D/16]); block_table
    int [B, max_pages]; ctx_lens int [B]; query head h reads KV head
    h // (H / H_kv); fmt "fp8": k_cache / v_cache are E4M3 codes
    [pages, H_kv, P, D] alone.  Returns o [B, H, D]:
    o[b, h] = sum_t softmax_t(sm_scale * q[b, h] . k_t) v_t over the
    ctx_lens[b] cached tokens (o = 0 for an empty context)."""
    q = np.asarray(q, np.float64)
    B, H, D = q.shape
    H_kv = (k_cache if fmt == "fp8" else k_cache[0]).shape[1]
    G = H // H_kv
    o = np.zeros((B, H, D))
    for b in range(B):
        n = int(ctx_lens[b])
        if n == 0:
            continue
        for hk in range(H_kv):
            if fmt == "fp8":
                K = kv_gather_fp8(k_cache, s_k, block_table[b], n, hk)
                V = kv_gather_fp8(v_cache, s_v, block_table[b], n, hk)
            else:
                K = kv_gather(k_cache[0], k_cache[1], s_k, block_table[b], n, hk)
                V = kv_gather(v_cache[0], v_cache[1], s_v, block_table[b], n, hk)
            for g in range(G):
                h = hk * G + g
                sc = sm_scale * (K @ q[b, h])
                w = np.exp(sc - sc.max())
                o[b, h] = (w / w.sum()) @ V
    return o


_THREADS = None


def threads():
    """OpenMP threads the oracle's parallel loops use."""
    if _THREADS is not None:
        return _THREADS
    return int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))


def set_threads(n):
    """Threads of the oracle's parallel loops from now on (timing only)."""
    global _THREADS
    L = lib()
    L.orc_set_threads.restype = None
    L.orc_set_threads.argtypes = [ctypes.c_int]
    L.orc_set_threads(int(n))
    _THREADS = int(n)
