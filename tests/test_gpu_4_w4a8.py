"""W4A8 route (FP8 activations x NVFP4 weights) against the oracle: exact
single-term cases, the per-layer shape of the policy stack on sampled rows,
and ragged shapes."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_common import dev_bf16, host, nv, nvfp4_device, quantize_pinned, y_np
from helpers import row_tolerance_ok

pytestmark = pytest.mark.gpu

ONE = 0x38


def pack(codes):
    codes = np.asarray(codes, np.uint8)
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)


def test_one_hot_fp8_rows_exact():
    # FP8 row k holds 1.0 at column k (s_t = 1): Y reads out dequantised weights
    rng = np.random.default_rng(31)
    N, K = 128, 128
    cw = rng.integers(0, 16, size=(N, K)).astype(np.uint8)
    sw = rng.integers(0x20, 0x50, size=(N, K // 16)).astype(np.uint8)
    w = nvfp4_device(pack(cw), sw, 0.5, N, K)
    a = np.zeros((K, K), np.uint8)
    a[np.arange(K), np.arange(K)] = ONE
    st = np.ones(K, np.float32)
    y = nv.w4a8_gemm(torch.from_numpy(a).cuda(), torch.from_numpy(st).cuda(), w, out_dtype=nv.OUT_FP32)
    ref = oracle.gemm_w4a8(a, st, (pack(cw), sw, 0.5))
    np.testing.assert_array_equal(y_np(y), ref)


def test_all_fp8_codes_times_all_weight_codes_exact():
    # a[m, k] runs over every finite E4M3 code (k < 16 nonzero per row), weights
    # over every E2M1 code with unit scale: exact 16-term sums
    K = 64
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    M = 128
    a = np.zeros((M, K), np.uint8)
    for m in range(M):
        a[m, :16] = codes[(np.arange(16) + 16 * m) % codes.size]
    cw = np.zeros((16, K), np.uint8)
    for j in range(16):
        cw[j, :16] = (np.arange(16) + j) % 16
    sw = np.full((16, K // 16), ONE, np.uint8)
    w = nvfp4_device(pack(cw), sw, 1.0, 16, K)
    st = np.ones(M, np.float32)
    y = nv.w4a8_gemm(torch.from_numpy(a).cuda(), torch.from_numpy(st).cuda(), w, out_dtype=nv.OUT_FP32)
    ref = oracle.gemm_w4a8(a, st, (pack(cw), sw, 1.0))
    np.testing.assert_array_equal(y_np(y), ref)


@pytest.mark.parametrize("M,N,K", [(2048, 4096, 4096), (130, 384, 320), (1, 256, 64), (300, 1000, 1024)])
def test_w4a8_route_against_oracle(M, N, K):
    xb = synth.activations(4, 20, M, K, 0.01, 50.0)
    wb = synth.weights(4, 21, N, K)
    w, wc, ws, wg = quantize_pinned(wb)
    y = nv.gemm(w, x=dev_bf16(xb), policy=nv.POLICY_Q8)   # per-token FP8 quantiser + W4A8 GEMM
    a8, st = oracle.fp8_token_encode(xb)
    rows = np.arange(M) if M <= 300 else np.concatenate([[0, M - 1], np.random.default_rng(M).choice(M, 30, replace=False)])
    ref = oracle.gemm_w4a8(a8, st, (wc, ws, wg[0]), rows=rows)
    ok, worst = row_tolerance_ok(y_np(y)[rows], ref, out_bf16=True)
    assert ok, worst
    # the separately exposed pieces give the same result
    a_dev, st_dev = nv.quantize_fp8(dev_bf16(xb))
    y2 = nv.w4a8_gemm(a_dev, st_dev, w)
    np.testing.assert_array_equal(y_np(y2), y_np(y))
