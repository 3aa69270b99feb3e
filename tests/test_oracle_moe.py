"""Pins for the oracle's mixture-of-experts feed-forward pieces: SiLU, the
SwiGLU up projection and the gate-weighted down-projection combine.

SiLU: closed forms (SiLU(0) = 0, SiLU(ln 3) = 0.75 ln 3, the odd-part
identity SiLU(x) - SiLU(-x) = x) and scipy's logistic function.
SwiGLU: a hand-evaluated one-element case, and per-expert dense products
through the plain W4A4 contraction.  Combine: a hand-evaluated two-route
case, single routes with unit weight reading out the product rows,
linearity in the routing weights, column sums over tokens, and the
residual input."""
import math

import numpy as np
import pytest
import scipy.special

import synth

ONE = 0x38                  # E4M3 code of 1.0
C_1, C_2, C_N1 = 2, 4, 10   # E2M1 codes of 1.0, 2.0, -1.0


def _random_nvfp4(rng, rows, K, sg):
    codes = rng.integers(0, 256, size=(rows, K // 2)).astype(np.uint8)
    scales = rng.integers(0x20, 0x48, size=(rows, K // 16)).astype(np.uint8)
    return codes, scales, np.float32(sg)


def test_silu_closed_forms(orc):
    assert orc.silu(0.0) == 0.0
    assert orc.silu(math.log(3.0)) == pytest.approx(0.75 * math.log(3.0), rel=1e-15)
    x = np.linspace(-30, 30, 1201)
    np.testing.assert_allclose(orc.silu(x) - orc.silu(-x), x, rtol=0, atol=1e-13)
    np.testing.assert_allclose(orc.silu(x), x * scipy.special.expit(x), rtol=1e-14, atol=1e-300)
    assert orc.silu(-1000.0) == 0.0 and orc.silu(1000.0) == 1000.0


def test_swiglu_one_element(orc):
    # K = 16, one expert, one routed row: a = 1.0 at k = 0; gate row 1.0 at
    # k = 0 and up row 2.0 at k = 0, tensor scales 0.5 (alpha = 0.25):
    # G = 0.25, U = 0.5, h = SiLU(0.25) * 0.5
    K = 16
    a_c = np.zeros((1, K), np.uint8)
    a_c[0, 0] = C_1
    g_c = np.zeros((1, 1, K), np.uint8)
    g_c[0, 0, 0] = C_1
    u_c = np.zeros((1, 1, K), np.uint8)
    u_c[0, 0, 0] = C_2
    pk = lambda c: (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)
    sc = np.full((1, 1, 1), ONE, np.uint8)
    h = orc.moe_up_swiglu((pk(a_c), sc[0], 0.5), None, np.array([0, 1]), (pk(g_c), sc), (pk(u_c), sc),
                          np.array([0.5], np.float32))
    assert h.shape == (1, 1)
    assert h[0, 0] == pytest.approx(0.25 / (1 + math.exp(-0.25)) * 0.5, rel=1e-15)


def test_swiglu_equals_dense_per_expert(orc):
    rng = np.random.default_rng(3)
    T, K, I, E = 30, 64, 16, 3
    a = _random_nvfp4(rng, T, K, 0.3)
    counts = np.array([11, 0, 25])
    row_idx, offsets = synth.moe_routing_from_counts(counts, T)
    gate = (rng.integers(0, 256, size=(E, I, K // 2)).astype(np.uint8),
            rng.integers(0x20, 0x48, size=(E, I, K // 16)).astype(np.uint8))
    up = (rng.integers(0, 256, size=(E, I, K // 2)).astype(np.uint8),
          rng.integers(0x20, 0x48, size=(E, I, K // 16)).astype(np.uint8))
    sg = np.array([0.5, 1.0, 0.25], np.float32)
    h = orc.moe_up_swiglu(a, row_idx, offsets, gate, up, sg)
    for e in (0, 2):
        rows = row_idx[offsets[e]:offsets[e + 1]].astype(np.int64)
        G = orc.gemm_w4a4(a, (gate[0][e], gate[1][e], sg[e]), rows=rows)
        U = orc.gemm_w4a4(a, (up[0][e], up[1][e], sg[e]), rows=rows)
        ref = G / (1.0 + np.exp(-G)) * U
        np.testing.assert_allclose(h[offsets[e]:offsets[e + 1]], ref, rtol=1e-15, atol=0)
    # gate and up swapped is a different function (the roles are not symmetric)
    h_sw = orc.moe_up_swiglu(a, row_idx, offsets, up, gate, sg)
    assert not np.allclose(h, h_sw)


def test_combine_two_routes_by_hand(orc):
    # two routed rows (experts 0 and 1) of token 1 out of 3; h rows are 1.0
    # and -1.0 at k = 0, both experts' single weight row is 2.0 at k = 0,
    # weights 0.25 and 0.75: y[1] = 0.25 * 2 + 0.75 * (-2) = -1, others 0
    K = 16
    hc = np.zeros((2, K), np.uint8)
    hc[0, 0], hc[1, 0] = C_1, C_N1
    wc = np.zeros((2, 1, K), np.uint8)
    wc[:, 0, 0] = C_2
    pk = lambda c: (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)
    y = orc.moe_down_combine((pk(hc), np.full((2, 1), ONE, np.uint8), 1.0), np.array([0, 1, 2]), pk(wc),
                             np.full((2, 1, 1), ONE, np.uint8), np.ones(2, np.float32),
                             np.array([1, 1], np.int32), np.array([0.25, 0.75], np.float32), 3)
    np.testing.assert_array_equal(y, [[0.0], [-1.0], [0.0]])


def test_combine_properties(orc):
    rng = np.random.default_rng(9)
    T, K, N, E, R = 12, 64, 24, 4, 30
    h = _random_nvfp4(rng, R, K, 0.7)
    offsets = np.array([0, 8, 8, 21, 30])
    wc = rng.integers(0, 256, size=(E, N, K // 2)).astype(np.uint8)
    ws = rng.integers(0x20, 0x48, size=(E, N, K // 16)).astype(np.uint8)
    wsg = np.array([0.5, 1.0, 2.0, 0.125], np.float32)
    tok = rng.integers(0, T, size=R).astype(np.int32)
    gw = rng.uniform(0.05, 1.0, size=R).astype(np.float32)
    D = orc.gemm_grouped_w4a4(h, None, offsets, wc, ws, wsg)
    y = orc.moe_down_combine(h, offsets, wc, ws, wsg, tok, gw, T)
    # column sums over tokens = weighted column sums over routed rows
    np.testing.assert_allclose(y.sum(axis=0), (gw[:, None].astype(np.float64) * D).sum(axis=0), rtol=1e-12)
    # linear in the weights
    np.testing.assert_allclose(orc.moe_down_combine(h, offsets, wc, ws, wsg, tok, 2 * gw, T), 2 * y, rtol=1e-15)
    # one route per token with unit weight reads out the product rows
    tok1 = np.arange(R, dtype=np.int32)
    y1 = orc.moe_down_combine(h, offsets, wc, ws, wsg, tok1, np.ones(R, np.float32), R)
    np.testing.assert_array_equal(y1, D)
    # a token nobody routes to stays at its residual value
    y0 = rng.standard_normal((T + 1, N))
    yr = orc.moe_down_combine(h, offsets, wc, ws, wsg, tok, gw, T + 1, y0=y0)
    np.testing.assert_array_equal(yr[T], y0[T])
    np.testing.assert_allclose(yr[:T], y0[:T] + y, rtol=1e-12, atol=1e-12)
