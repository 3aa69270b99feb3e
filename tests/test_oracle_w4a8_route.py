"""Why the W4A8 route upconverts to FP16 instead of running the FP8 MMA kind.

The sensitive layers of "llama.cpp Put Precision Policy Inside the Model.
That Matters More Than W4A4" ("One model can need more than one precision")
take FP8 activations against the NVFP4 weights.  The tensor cores' FP8 kind
with block scales (kind::mxf8f6f4) runs at twice the FP16 rate, but it takes
E4M3 elements with one power-of-two (UE8M0) scale per 32 elements, so the
NVFP4 weights (E2M1 code x E4M3 scale per 16) would have to be requantised.
This test measures that requantisation against the GEMM tolerance on a
configuration-4 layer: with the FP32 tensor scale left to the epilogue (the
most favourable case), the requantised product still misses
max_n |err| <= 1e-3 * ||row||_2, while the FP16 upconversion the library uses
is exact.  Oracle and numpy only; no GPU."""
import numpy as np

import oracle
import synth
from helpers import row_tolerance_ok

C4 = synth.CONFIGS[4]


def mx_fp8_requantise(v):
    """OCP-MX FP8 (E4M3 elements) of a [R, K] float64 matrix: per 32 elements
    along K a shared power-of-two scale 2^(floor(log2 amax) - 8) (8 is the
    E4M3 maximum exponent) and each element rounded to E4M3 by the oracle's
    encoder; returns the dequantised values."""
    blk = v.reshape(v.shape[0], -1, 32)
    amax = np.abs(blk).max(axis=2, keepdims=True)
    e = np.where(amax > 0, np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - 8, 0.0)
    scaled = (blk / np.exp2(e)).astype(np.float32)
    assert np.array_equal(scaled.astype(np.float64) * np.exp2(e), blk)  # power-of-two scaling is exact
    codes = oracle.e4m3_encode_array(scaled.ravel())
    table = np.array([oracle.e4m3_value(c) for c in range(256)])
    return (table[codes].reshape(blk.shape) * np.exp2(e)).reshape(v.shape)


def test_mx_fp8_weight_route_misses_the_gemm_tolerance():
    rows = 32
    x = synth.activations(4, 200, rows, C4["K"], C4["outlier_frac"], C4["outlier_factor"])
    a8, st = oracle.fp8_token_encode(x)
    wc, ws, sg = oracle.nvfp4_encode(synth.weights(4, 100, C4["N"], C4["K"]))
    exact = oracle.gemm_w4a8(a8, st, (wc, ws, sg))
    # code x block scale, the tensor scale applied after the contraction
    w_cs = oracle.nvfp4_dequant(wc, ws, 1.0)
    w_mx = mx_fp8_requantise(w_cs)
    changed = np.mean(w_mx != w_cs)
    table = np.array([oracle.e4m3_value(c) for c in range(256)])
    a = table[a8] * st[:, None].astype(np.float64)
    lossy = (a @ w_mx.T) * float(sg)
    ok, worst = row_tolerance_ok(lossy, exact)
    assert changed > 0.1, "E4M3 elements cannot hold a large share of the NVFP4 weight values"
    assert not ok and worst > 2e-3, f"the requantised route would pass (worst {worst:.3e})"
    # the exact route: FP16 holds every E2M1 x E4M3 weight value and every E4M3 activation
    assert np.array_equal(w_cs.astype(np.float16).astype(np.float64), w_cs)
    assert np.array_equal(table[:127].astype(np.float16).astype(np.float64), table[:127])
