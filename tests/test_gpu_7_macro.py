"""FP16 macro-scale W4A4 GEMM (one FP16 scale per 256 elements of a row,
"Two-Level Block Scaling") against the oracle: configuration 1 in full,
ragged shapes, sampled prefill rows, and the reduction to the tensor-scale
path when every macro-scale is the same value."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_common import dev_bf16, host, nv, quantize_pinned, y_np
from helpers import row_tolerance_ok

pytestmark = pytest.mark.gpu


def _macro_case(M, N, K, xcfg=1, seed=60):
    xb = synth.activations(9, seed, M, K, 0.01, 50.0)
    wb = synth.weights(9, seed + 1, N, K)
    w, wc, ws, wm = quantize_pinned(wb, mode=nv.SCALE_MACRO_FP16)
    ow = oracle.nvfp4_encode_macro(wb)
    np.testing.assert_array_equal(wc, ow[0])
    np.testing.assert_array_equal(ws, ow[1])
    np.testing.assert_array_equal(wm, ow[2])
    return xb, w, (wc, ws, wm)


@pytest.mark.parametrize("M,N,K", [(128, 256, 512), (200, 384, 768), (8, 1024, 2048), (130, 130, 256)])
@pytest.mark.parametrize("out_dtype", [nv.OUT_BF16, nv.OUT_FP32])
def test_macro_gemm_against_oracle(M, N, K, out_dtype):
    xb, w, wq = _macro_case(M, N, K)
    y = nv.gemm(w, x=dev_bf16(xb), out_dtype=out_dtype)   # quantises X in macro mode on the fly
    ref = oracle.gemm_w4a4_macro(oracle.nvfp4_encode_macro(xb), wq)
    ok, worst = row_tolerance_ok(y_np(y), ref, out_bf16=out_dtype == nv.OUT_BF16)
    assert ok, f"{M}x{N}x{K}: {worst}"
    # pre-quantised activations give the same result
    a, *_ = quantize_pinned(xb, mode=nv.SCALE_MACRO_FP16)
    y2 = nv.gemm(w, a_q=a, out_dtype=out_dtype)
    np.testing.assert_array_equal(y_np(y2), y_np(y))


def test_macro_prefill_sampled_rows():
    xb, w, wq = _macro_case(4096, 8192, 8192, seed=62)
    y = y_np(nv.gemm(w, x=dev_bf16(xb)))
    # the first and last rows plus 256 seeded ones, as for the tensor-scale
    # prefill
    rows = np.concatenate([[0, 4095], np.random.default_rng(62).choice(np.arange(1, 4095), 256, replace=False)])
    ref = oracle.gemm_w4a4_macro(oracle.nvfp4_encode_macro(xb), wq, rows=rows)
    ok, worst = row_tolerance_ok(y[rows], ref, out_bf16=True)
    assert ok, worst


def test_equal_macro_scales_reduce_to_tensor_scale_path():
    # codes and scales from a tensor-mode encode; every macro-scale set to the
    # tensor scale (an FP16-exact power of two): both GEMM paths agree
    M, N, K = 128, 256, 512
    xb = synth.activations(9, 64, M, K, 0.01, 50.0)
    wb = synth.weights(9, 65, N, K)
    a, *_ = quantize_pinned(xb)
    w, *_ = quantize_pinned(wb)
    y_t = y_np(nv.gemm(w, a_q=a, out_dtype=nv.OUT_FP32))
    a_s, w_s = float(host(a.second)[0]), float(host(w.second)[0])
    # force exact power-of-two tensor scales so FP16 holds them exactly
    pa, pw = 2.0 ** np.round(np.log2(a_s)), 2.0 ** np.round(np.log2(w_s))
    a.second.fill_(pa)
    w.second.fill_(pw)
    y_t = y_np(nv.gemm(w, a_q=a, out_dtype=nv.OUT_FP32))
    am = torch.full((M, K // 256), 0, dtype=torch.int16, device="cuda")
    wm = torch.full((N, K // 256), 0, dtype=torch.int16, device="cuda")
    am.fill_(int(np.float16(pa).view(np.int16)))
    wm.fill_(int(np.float16(pw).view(np.int16)))
    am_t = nv.NVFP4Tensor(a.codes, a.scales, am, M, K, nv.SCALE_MACRO_FP16)
    wm_t = nv.NVFP4Tensor(w.codes, w.scales, wm, N, K, nv.SCALE_MACRO_FP16)
    y_m = y_np(nv.gemm(wm_t, a_q=am_t, out_dtype=nv.OUT_FP32))
    ok, worst = row_tolerance_ok(y_m, y_t, rel=1e-5)
    assert ok, worst
