"""Test helpers: layout permutations of the ABI's tiled scale format, the
GEMM tolerance of the benchmark spec, and host/device moves.  No quantisation or
contraction arithmetic lives here."""
import numpy as np


def tile_scales(rowmajor: np.ndarray, rows: int, K: int) -> np.ndarray:
    """Row-major E4M3 scale bytes [rows, K/16] -> MMA-tiled bytes (rows padded
    to 128 with zeros): byte (r % 32) * 16 + ((r % 128) // 32) * 4 + b % 4 of
    atom (r // 128) * (K/64) + b // 4."""
    rt = -(-rows // 128)
    pad = np.zeros((rt * 128, K // 16), np.uint8)
    pad[:rows] = rowmajor
    t = pad.reshape(rt, 4, 32, K // 64, 4)            # [rt][sub][lane][kc][j]
    return np.ascontiguousarray(t.transpose(0, 3, 2, 1, 4)).reshape(-1)


def untile_scales(tiled: np.ndarray, rows: int, K: int) -> np.ndarray:
    t = np.asarray(tiled, np.uint8).reshape(-1, K // 64, 32, 4, 4)   # [rt][kc][lane][sub][j]
    return np.ascontiguousarray(t.transpose(0, 3, 2, 1, 4)).reshape(-1, K // 16)[:rows]


def interleave_gate_up(gate: np.ndarray, up: np.ndarray) -> np.ndarray:
    """Per-expert gate and up row arrays [E, I, X] -> the stacked [E, 2I, X]
    order of the SwiGLU up projection: 128-row gate and up blocks alternate
    (rows 256b .. 256b+127 = gate rows 128b.., the next 128 = up rows 128b..)."""
    E, I = gate.shape[:2]
    g = gate.reshape(E, I // 128, 128, -1)
    u = up.reshape(E, I // 128, 128, -1)
    return np.concatenate([g, u], axis=2).reshape(E, 2 * I, -1)


def kv_v_pages(codes_nat: np.ndarray, scales_nat: np.ndarray):
    """Value pages from the natural per-token layout (codes [..., 64 tokens,
    64 bytes], scales [..., 64, 8]) to the cache's dim-major layout (codes
    [..., 128 dims, 32 bytes]: byte j of row d = tokens 2j (low nibble),
    2j+1; scales [..., 8 blocks, 64 tokens]).  A pure relayout."""
    c = np.asarray(codes_nat, np.uint8)
    nib = np.empty(c.shape[:-1] + (c.shape[-1] * 2,), np.uint8)
    nib[..., 0::2] = c & 15
    nib[..., 1::2] = c >> 4                          # [..., token, dim]
    nt = np.swapaxes(nib, -1, -2)                    # [..., dim, token]
    v = (nt[..., 0::2] | (nt[..., 1::2] << 4)).astype(np.uint8)
    return np.ascontiguousarray(v), np.ascontiguousarray(np.swapaxes(np.asarray(scales_nat, np.uint8), -1, -2))


def kv_v_pages_natural(codes_dm: np.ndarray, scales_bm: np.ndarray):
    """Inverse of kv_v_pages."""
    c = np.asarray(codes_dm, np.uint8)
    nib = np.empty(c.shape[:-1] + (c.shape[-1] * 2,), np.uint8)
    nib[..., 0::2] = c & 15
    nib[..., 1::2] = c >> 4                          # [..., dim, token]
    nt = np.swapaxes(nib, -1, -2)                    # [..., token, dim]
    k = (nt[..., 0::2] | (nt[..., 1::2] << 4)).astype(np.uint8)
    return np.ascontiguousarray(k), np.ascontiguousarray(np.swapaxes(np.asarray(scales_bm, np.uint8), -1, -2))


def bf16_half_ulp(y: np.ndarray) -> np.ndarray:
    """Half the BF16 spacing at |y| (the largest error of rounding y to BF16)."""
    a = np.abs(np.asarray(y, np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(e - 8), 0.0)


def row_tolerance_ok(y_gpu: np.ndarray, y_ref: np.ndarray, rel: float = 1e-3, out_bf16: bool = False):
    """Per output row m: max_n |Y_gpu - Y_ref| <= rel * ||Y_ref[m, :]||_2
    (zero rows must be exactly zero).  For BF16 outputs each element may in
    addition carry the rounding of Y_ref to BF16 (half a BF16 ulp), since the
    output format alone cannot hold a dominant element of a row to 1e-3 of the
    row norm.  Returns (ok, worst ratio)."""
    y_gpu = np.asarray(y_gpu, np.float64)
    y_ref = np.asarray(y_ref, np.float64)
    diff = np.abs(y_gpu - y_ref)
    if out_bf16:
        diff = np.maximum(diff - bf16_half_ulp(y_ref), 0.0)
    err = diff.max(axis=1)
    norm = np.sqrt((y_ref ** 2).sum(axis=1))
    zero = norm == 0
    ratio = np.where(zero, np.where(err == 0, 0.0, np.inf), err / np.where(zero, 1, norm))
    return bool((ratio <= rel).all()), float(ratio.max(initial=0.0))
