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


def _kv_slots(fp8: bool) -> np.ndarray:
    """slot -> token of a 32-token half page's keys: the attention reads the
    8 keys of one score n-tile as 8 consecutive slots.  NVFP4 swaps the bit
    fields token[4:3] and token[2:1]; FP8 moves token bit 1 to bit 3 and
    token bits 3:2 to bits 2:1."""
    k = np.arange(32)
    if fp8:
        pos = (k & 16) | ((k & 2) << 2) | ((k >> 1) & 6) | (k & 1)
    else:
        pos = 8 * ((k >> 1) & 3) + 2 * (k >> 3) + (k & 1)
    tok = np.empty(32, np.int64)
    tok[pos] = k
    return tok


def kv_pack_nvfp4(k_c, k_s, v_c_nat, v_s_nat):
    """Natural per-token NVFP4 cache arrays ([..., 64, 64] codes, [..., 64, 8]
    scales, for keys and values) -> the cache's page blocks [..., 9216]: per
    32-token half, key codes [4 dim chunks][32 key slots][16], key scales
    [32 key slots][8], value codes dim-major [128][16], value scales
    block-major [8][32]."""
    lead = np.asarray(k_c).shape[:-2]
    tok = _kv_slots(False)
    parts = []
    for h in range(2):
        sl = slice(32 * h, 32 * h + 32)
        kc = np.asarray(k_c, np.uint8)[..., sl, :][..., tok, :]                  # [..., slot, 64]
        kc = np.swapaxes(kc.reshape(lead + (32, 4, 16)), -3, -2)                # [..., chunk, slot, 16]
        ks = np.asarray(k_s, np.uint8)[..., sl, :][..., tok, :]
        vdm, vsbm = kv_v_pages(np.asarray(v_c_nat)[..., sl, :], np.asarray(v_s_nat)[..., sl, :])
        parts += [kc, ks, vdm, vsbm]
    return np.ascontiguousarray(np.concatenate([x.reshape(lead + (-1,)) for x in parts], axis=-1))


def kv_unpack_nvfp4(blocks):
    """Inverse of kv_pack_nvfp4: (k_c, k_s, v_c natural, v_s natural)."""
    b = np.asarray(blocks, np.uint8)
    lead = b.shape[:-1]
    tok = _kv_slots(False)
    out = [[], [], [], []]
    for h in range(2):
        o = 4608 * h
        kc = np.swapaxes(b[..., o:o + 2048].reshape(lead + (4, 32, 16)), -3, -2).reshape(lead + (32, 64))
        ks = b[..., o + 2048:o + 2304].reshape(lead + (32, 8))
        kn, sn = np.empty_like(kc), np.empty_like(ks)
        kn[..., tok, :] = kc
        sn[..., tok, :] = ks
        out[0].append(kn)
        out[1].append(sn)
        v_c, v_s = kv_v_pages_natural(b[..., o + 2304:o + 4352].reshape(lead + (128, 16)),
                                      b[..., o + 4352:o + 4608].reshape(lead + (8, 32)))
        out[2].append(v_c)
        out[3].append(v_s)
    return tuple(np.ascontiguousarray(np.concatenate(x, axis=-2)) for x in out)


def kv_pack_fp8(k, v_nat):
    """Natural FP8 cache arrays ([..., 64 tokens, 128]) -> page blocks
    [..., 16384]: per 32-token half, keys [8 dim chunks][32 key slots][16]
    then values [2 token groups][128 dims][16] (byte j of group u = token
    16 u + j)."""
    k, v = np.asarray(k, np.uint8), np.asarray(v_nat, np.uint8)
    lead = k.shape[:-2]
    tok = _kv_slots(True)
    halves = []
    for h in range(2):
        kh = k[..., 32 * h:32 * h + 32, :][..., tok, :]                           # [..., slot, 128]
        halves.append(np.swapaxes(kh.reshape(lead + (32, 8, 16)), -3, -2).reshape(lead + (-1,)))
        vh = v[..., 32 * h:32 * h + 32, :].reshape(lead + (2, 16, 128))          # [..., group, token, dim]
        halves.append(np.swapaxes(vh, -1, -2).reshape(lead + (-1,)))
    return np.ascontiguousarray(np.concatenate(halves, axis=-1))


def kv_unpack_fp8(blocks):
    """Inverse of kv_pack_fp8: (keys, values) natural [..., 64, 128]."""
    b = np.asarray(blocks, np.uint8)
    lead = b.shape[:-1]
    tok = _kv_slots(True)
    ks, vs = [], []
    for h in range(2):
        base = 8192 * h
        kh = np.swapaxes(b[..., base:base + 4096].reshape(lead + (8, 32, 16)), -3, -2).reshape(lead + (32, 128))
        kn = np.empty_like(kh)
        kn[..., tok, :] = kh
        ks.append(kn)
        vh = b[..., base + 4096:base + 8192].reshape(lead + (2, 128, 16))
        vs.append(np.swapaxes(vh, -1, -2).reshape(lead + (32, 128)))
    return np.ascontiguousarray(np.concatenate(ks, axis=-2)), np.ascontiguousarray(np.concatenate(vs, axis=-2))


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
