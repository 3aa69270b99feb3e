"""Pins for the oracle's contractions (W4A4, macro W4A4, W4A8, grouped).

Pins: brute force over all 16x16 E2M1 code pairs at K = 16 with exact
rational arithmetic from the golden code table; every non-negative E4M3
scale; one-hot activation rows that read out single dequantised weights;
whole-block K permutations; numpy's float64 matmul of the dequantised
operands; and the reduction of the grouped product to per-expert dense ones.
"""
import os
from fractions import Fraction

import numpy as np
import torch

import synth
from conftest import GOLDEN

ONE = 0x38  # E4M3 code of 1.0


def _golden_e2m1():
    vals = {}
    with open(os.path.join(GOLDEN, "e2m1_codes.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                c, v = line.split()
                vals[int(c)] = Fraction(v)
    return vals


def pack(codes):
    codes = np.asarray(codes, np.uint8)
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)


def e4m3_values():
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()


def test_all_code_pairs_brute_force(orc):
    # A row i: codes (i + k) % 16; W row j: codes (j + 3k) % 16, K = 16, unit
    # scales, tensor scales 1 -> Y[i][j] = sum_k v(a_ik) v(w_jk) exactly.
    g = _golden_e2m1()
    ca = np.array([[(i + k) % 16 for k in range(16)] for i in range(16)], np.uint8)
    cw = np.array([[(j + 3 * k) % 16 for k in range(16)] for j in range(16)], np.uint8)
    sa = np.full((16, 1), ONE, np.uint8)
    Y = orc.gemm_w4a4((pack(ca), sa, 1.0), (pack(cw), sa.copy(), 1.0))
    for i in range(16):
        for j in range(16):
            want = sum(g[int(ca[i, k])] * g[int(cw[j, k])] for k in range(16))
            assert Y[i, j] == float(want), (i, j)
    # and every single pair: A row = code a at k=0 only, W row = code b at k=0
    for a in range(16):
        A = np.zeros((1, 16), np.uint8)
        A[0, 0] = a
        W = np.zeros((16, 16), np.uint8)
        W[:, 0] = np.arange(16)
        Y = orc.gemm_w4a4((pack(A), np.full((1, 1), ONE, np.uint8), 1.0),
                          (pack(W), np.full((16, 1), ONE, np.uint8), 1.0))
        for b in range(16):
            assert Y[0, b] == float(g[a] * g[b])


def test_every_e4m3_scale(orc):
    ev = e4m3_values()
    rng = np.random.default_rng(11)
    K = 32
    ca = rng.integers(0, 16, size=(1, K)).astype(np.uint8)
    cw = rng.integers(0, 16, size=(127, K)).astype(np.uint8)
    g = _golden_e2m1()
    sw = np.zeros((127, 2), np.uint8)
    sw[:, 0] = np.arange(127)  # block 0 of weight row n has scale code n
    sw[:, 1] = ONE
    Y = orc.gemm_w4a4((pack(ca), np.full((1, 2), ONE, np.uint8), 1.0), (pack(cw), sw, 1.0))
    for n in range(127):
        b0 = sum(g[int(ca[0, k])] * g[int(cw[n, k])] for k in range(16))
        b1 = sum(g[int(ca[0, k])] * g[int(cw[n, k])] for k in range(16, 32))
        assert Y[0, n] == float(b0) * ev[n] + float(b1)


def test_one_hot_rows_read_out_weights(orc):
    rng = np.random.default_rng(12)
    N, K = 24, 64
    cw = rng.integers(0, 16, size=(N, K)).astype(np.uint8)
    sw = rng.integers(0, 0x7F, size=(N, K // 16)).astype(np.uint8)
    sgw = np.float32(0.37)
    ev = e4m3_values()
    g = _golden_e2m1()
    A = np.zeros((K, K), np.uint8)
    A[np.arange(K), np.arange(K)] = 2  # code of 1.0 at position k
    sa = np.full((K, K // 16), ONE, np.uint8)
    sga = np.float32(2.0 ** -3)
    Y = orc.gemm_w4a4((pack(A), sa, sga), (pack(cw), sw, sgw))
    for k in range(K):
        for n in range(N):
            want = float(g[int(cw[n, k])]) * ev[sw[n, k // 16]] * float(sgw) * float(sga)
            assert Y[k, n] == want


def _random_nvfp4(rng, R, K, sg):
    c = rng.integers(0, 16, size=(R, K)).astype(np.uint8)
    s = rng.integers(0, 0x7F, size=(R, K // 16)).astype(np.uint8)
    return pack(c), s, np.float32(sg)


def test_matches_numpy_matmul_of_dequantised(orc):
    rng = np.random.default_rng(13)
    a = _random_nvfp4(rng, 40, 256, 0.013)
    w = _random_nvfp4(rng, 56, 256, 2.7)
    Y = orc.gemm_w4a4(a, w)
    ref = orc.nvfp4_dequant(*a) @ orc.nvfp4_dequant(*w).T
    np.testing.assert_allclose(Y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    rows = np.array([39, 0, 17])
    np.testing.assert_array_equal(orc.gemm_w4a4(a, w, rows=rows), Y[rows])


def test_block_permutation_invariance(orc):
    rng = np.random.default_rng(14)
    K = 256
    ac, as_, ag = _random_nvfp4(rng, 8, K, 1.0)
    wc, ws, wg = _random_nvfp4(rng, 8, K, 1.0)
    perm = rng.permutation(K // 16)
    def permute(c, s):
        cb = c.reshape(c.shape[0], K // 16, 8)[:, perm].reshape(c.shape)
        return np.ascontiguousarray(cb), np.ascontiguousarray(s[:, perm])
    Y0 = orc.gemm_w4a4((ac, as_, ag), (wc, ws, wg))
    pa, psa = permute(ac, as_)
    pw, psw = permute(wc, ws)
    Y1 = orc.gemm_w4a4((pa, psa, ag), (pw, psw, wg))
    np.testing.assert_allclose(Y0, Y1, rtol=1e-12, atol=1e-12 * np.abs(Y0).max())


def test_macro_gemm(orc):
    rng = np.random.default_rng(15)
    K = 512
    ac, as_, _ = _random_nvfp4(rng, 12, K, 1.0)
    wc, ws, _ = _random_nvfp4(rng, 20, K, 1.0)
    am = np.float16(rng.uniform(0.01, 3, size=(12, 2))).view(np.uint16)
    wm = np.float16(rng.uniform(0.01, 3, size=(20, 2))).view(np.uint16)
    Y = orc.gemm_w4a4_macro((ac, as_, am), (wc, ws, wm))
    ref = orc.nvfp4_dequant_macro(ac, as_, am) @ orc.nvfp4_dequant_macro(wc, ws, wm).T
    np.testing.assert_allclose(Y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    # equal macro scales S reduce to the tensor-scale product with s_g = S
    S = np.float16(0.75)
    Ym = orc.gemm_w4a4_macro((ac, as_, np.full_like(am, S.view(np.uint16))),
                             (wc, ws, np.full_like(wm, S.view(np.uint16))))
    Yt = orc.gemm_w4a4((ac, as_, np.float32(S)), (wc, ws, np.float32(S)))
    np.testing.assert_allclose(Ym, Yt, rtol=1e-12, atol=1e-12 * np.abs(Yt).max())


def test_w4a8(orc):
    rng = np.random.default_rng(16)
    M, N, K = 9, 33, 128
    a = rng.integers(0, 256, size=(M, K)).astype(np.uint8)
    a[(a & 0x7F) == 0x7F] = 0  # no NaN codes
    st = rng.uniform(0.01, 2, size=M).astype(np.float32)
    w = _random_nvfp4(rng, N, K, 0.21)
    Y = orc.gemm_w4a8(a, st, w)
    ev = e4m3_values()
    ref = (ev[a] * st[:, None].astype(np.float64)) @ orc.nvfp4_dequant(*w).T
    np.testing.assert_allclose(Y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    # one-hot FP8 rows (value 1.0, s_t = 1) read out weights
    A = np.zeros((K, K), np.uint8)
    A[np.arange(K), np.arange(K)] = ONE
    Y1 = orc.gemm_w4a8(A, np.ones(K, np.float32), w)
    np.testing.assert_array_equal(Y1, orc.nvfp4_dequant(*w).T)


def test_grouped_equals_per_expert_dense(orc):
    rng = np.random.default_rng(17)
    T, K, N, E = 40, 128, 24, 5
    a = _random_nvfp4(rng, T, K, 0.5)
    counts = np.array([7, 0, 19, 1, 13])
    row_idx, offsets = synth.moe_routing_from_counts(counts, T)
    wc = rng.integers(0, 256, size=(E, N, K // 2)).astype(np.uint8)
    ws = rng.integers(0, 0x7F, size=(E, N, K // 16)).astype(np.uint8)
    wsg = rng.uniform(0.1, 2, size=E).astype(np.float32)
    Y = orc.gemm_grouped_w4a4(a, row_idx, offsets, wc, ws, wsg)
    assert Y.shape == (counts.sum(), N)
    for e in range(E):
        lo, hi = offsets[e], offsets[e + 1]
        if hi == lo:
            continue
        rows = row_idx[lo:hi].astype(np.int64)
        ref = orc.gemm_w4a4(a, (wc[e], ws[e], wsg[e]), rows=rows)
        np.testing.assert_array_equal(Y[lo:hi], ref)
    # contiguous rows (no index list)
    Yc = orc.gemm_grouped_w4a4(a, None, np.array([0, 10, 10, 30, 31, 40]), wc, ws, wsg)
    np.testing.assert_array_equal(Yc[10:30], orc.gemm_w4a4(a, (wc[2], ws[2], wsg[2]), rows=np.arange(10, 30)))


def test_grouped_w4a8_by_dequantised_matmul(orc):
    # each expert's rows against numpy's float64 product of the decoded FP8
    # rows (times their token scales) and the expert's dequantised weights
    rng = np.random.default_rng(23)
    T, K, N, E = 20, 64, 16, 4
    a = rng.integers(0, 256, size=(T, K)).astype(np.uint8)
    a[(a & 0x7F) == 0x7F] = 0  # no NaN codes
    st = rng.uniform(0.01, 2, size=T).astype(np.float32)
    counts = np.array([5, 0, 12, 3])
    row_idx, offsets = synth.moe_routing_from_counts(counts, T)
    wc = rng.integers(0, 256, size=(E, N, K // 2)).astype(np.uint8)
    ws = rng.integers(0x20, 0x48, size=(E, N, K // 16)).astype(np.uint8)
    wsg = np.array([0.5, 1.0, 0.25, 2.0], np.float32)
    Y = orc.gemm_grouped_w4a8(a, st, row_idx, offsets, wc, ws, wsg)
    ev = e4m3_values()
    for e in range(E):
        lo, hi = offsets[e], offsets[e + 1]
        rows = row_idx[lo:hi]
        ref = (ev[a[rows]] * st[rows, None].astype(np.float64)) @ orc.nvfp4_dequant(wc[e], ws[e], wsg[e]).T
        np.testing.assert_allclose(Y[lo:hi], ref, rtol=1e-12, atol=1e-12 * max(np.abs(ref).max(initial=0), 1))
    # contiguous rows: output row j reads activation row j
    Yc = orc.gemm_grouped_w4a8(a, st, None, np.array([0, 4, 4, 19, 20]), wc, ws, wsg)
    ref = (ev[a[4:19]] * st[4:19, None].astype(np.float64)) @ orc.nvfp4_dequant(wc[2], ws[2], wsg[2]).T
    np.testing.assert_allclose(Yc[4:19], ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
