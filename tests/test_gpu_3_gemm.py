"""W4A4 block-scaled GEMM on the tensor cores against the oracle.

Exact cases (FP32 output; every partial sum is exactly representable):
all 16x16 E2M1 code pairs, every non-negative E4M3 scale, one-hot rows, on
one 128-row tile and across several M tiles, partial tiles and K stages.
Tolerance cases: max_n |Y - Y_ref| <= 1e-3 * ||Y_ref[m, :]||_2 per row
against the FP64 oracle, on configuration 1 in full, the decode shapes
(M = 1, 8, 16 against the 28672 x 8192 weights) in full, the prefill shapes
on 256 seeded rows plus the first and last, and ragged shapes that exercise
M/N/K tails, stream-K and many-tile shapes."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_common import dev_bf16, host, nv, nvfp4_device, quantize_pinned, y_np
from helpers import row_tolerance_ok

pytestmark = pytest.mark.gpu

ONE = 0x38
C = synth.CONFIGS


def pack(codes):
    codes = np.asarray(codes, np.uint8)
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)


def gemm_q(a, w, out_dtype=nv.OUT_FP32):
    y = nv.gemm(w, a_q=a, out_dtype=out_dtype)
    return y_np(y)


@pytest.mark.parametrize("M", [16, 128])
def test_all_code_pairs_exact(M):
    # A row i: code (i + k) % 16 for k < 16, W row j: (j + 3k) % 16; K = 64 with
    # zeros past k = 16; unit scales and tensor scales.  M = 16 runs the
    # swapped (decode) orientation, M = 128 the direct one.
    K = 64
    ca = np.zeros((M, K), np.uint8)
    cw = np.zeros((16, K), np.uint8)
    for i in range(M):
        ca[i, :16] = [(i + k) % 16 for k in range(16)]
    for j in range(16):
        cw[j, :16] = [(j + 3 * k) % 16 for k in range(16)]
    sa = np.full((M, K // 16), ONE, np.uint8)
    sw = np.full((16, K // 16), ONE, np.uint8)
    a = nvfp4_device(pack(ca), sa, 1.0, M, K)
    w = nvfp4_device(pack(cw), sw, 1.0, 16, K)
    Y = gemm_q(a, w)
    ref = oracle.gemm_w4a4((pack(ca), sa, 1.0), (pack(cw), sw, 1.0))
    np.testing.assert_array_equal(Y, ref)


@pytest.mark.parametrize("M,N", [(384, 16), (256, 300), (513, 272)])
def test_all_code_pairs_exact_many_tiles(M, N):
    # several 128-row tiles, K = 256 (one stage): A row i has code (i + k) % 16
    # at every k, W row j code (j + 3k) % 16, unit scales; each output is a
    # sum of 256 products of E2M1 values, exact in FP32.  The shapes leave
    # partial tiles in M and N.
    K = 256
    assert nv.gemm_kernel_path(M, N, K) == nv.PATH_WHOLE_TILES
    k = np.arange(K)
    ca = ((np.arange(M)[:, None] + k[None, :]) % 16).astype(np.uint8)
    cw = ((np.arange(N)[:, None] + 3 * k[None, :]) % 16).astype(np.uint8)
    sa = np.full((M, K // 16), ONE, np.uint8)
    sw = np.full((N, K // 16), ONE, np.uint8)
    a = nvfp4_device(pack(ca), sa, 1.0, M, K)
    w = nvfp4_device(pack(cw), sw, 1.0, N, K)
    Y = gemm_q(a, w)
    ref = oracle.gemm_w4a4((pack(ca), sa, 1.0), (pack(cw), sw, 1.0))
    np.testing.assert_array_equal(Y, ref)


@pytest.mark.parametrize("M,K", [(128, 64), (256, 256), (300, 1024)])
def test_every_e4m3_scale_exact(M, K):
    # only block 1 (k = 16..31) of the weights is non-zero, so every output is
    # one scaled block sum: E4M3(m % 127) * E4M3(n) * sum_k a*w, exact in FP32.
    # M = 128 is one tile, the others several (the block sits in the first
    # stage; K = 1024 adds stages of zeros).
    rng = np.random.default_rng(21)
    ca = rng.integers(0, 16, size=(M, K)).astype(np.uint8)
    cw = np.zeros((127, K), np.uint8)
    cw[:, 16:32] = rng.integers(0, 16, size=(127, 16))
    sa = np.full((M, K // 16), ONE, np.uint8)
    sw = np.full((127, K // 16), ONE, np.uint8)
    sw[:, 1] = np.arange(127)
    sa[:, 1] = (np.arange(M) % 127).astype(np.uint8)
    a = nvfp4_device(pack(ca), sa, 1.0, M, K)
    w = nvfp4_device(pack(cw), sw, 1.0, 127, K)
    Y = gemm_q(a, w)
    ref = oracle.gemm_w4a4((pack(ca), sa, 1.0), (pack(cw), sw, 1.0))
    np.testing.assert_array_equal(Y, ref)


def test_every_e4m3_scale_exact_b_groups():
    # B scales across tiles: 512 weight rows (two 256-row tiles, four 128-row
    # scale groups) each carrying a different E4M3 scale in block 5 of the
    # second stage (k = 336..351), and every activation scale there
    rng = np.random.default_rng(23)
    M, N, K = 256, 512, 512
    ca = rng.integers(0, 16, size=(M, K)).astype(np.uint8)
    cw = np.zeros((N, K), np.uint8)
    cw[:, 336:352] = rng.integers(0, 16, size=(N, 16))
    sa = np.full((M, K // 16), ONE, np.uint8)
    sw = np.full((N, K // 16), ONE, np.uint8)
    sw[:, 21] = (np.arange(N) % 127).astype(np.uint8)
    sa[:, 21] = ((np.arange(M) * 7) % 127).astype(np.uint8)
    a = nvfp4_device(pack(ca), sa, 1.0, M, K)
    w = nvfp4_device(pack(cw), sw, 1.0, N, K)
    Y = gemm_q(a, w)
    ref = oracle.gemm_w4a4((pack(ca), sa, 1.0), (pack(cw), sw, 1.0))
    np.testing.assert_array_equal(Y, ref)


def test_one_hot_rows_read_out_weights():
    rng = np.random.default_rng(22)
    N, K = 256, 256
    cw = rng.integers(0, 16, size=(N, K)).astype(np.uint8)
    sw = rng.integers(0x20, 0x50, size=(N, K // 16)).astype(np.uint8)
    A = np.zeros((K, K), np.uint8)
    A[np.arange(K), np.arange(K)] = 2
    sa = np.full((K, K // 16), ONE, np.uint8)
    a = nvfp4_device(pack(A), sa, 0.125, K, K)
    w = nvfp4_device(pack(cw), sw, 0.75, N, K)
    Y = gemm_q(a, w)
    ref = oracle.gemm_w4a4((pack(A), sa, 0.125), (pack(cw), sw, 0.75))
    np.testing.assert_array_equal(Y, ref)


def _layer(cfg, M, N, K, xtid=0, wtid=1):
    c = C[cfg]
    xb = synth.activations(cfg, xtid, M, K, c["outlier_frac"], c["outlier_factor"])
    wb = synth.weights(cfg, wtid, N, K)
    return xb, wb


def _check(y, ref, what, bf16=True):
    ok, worst = row_tolerance_ok(y, ref, out_bf16=bf16)
    assert ok, f"{what}: worst row error ratio {worst:.3e} > 1e-3"


@pytest.mark.parametrize("out_dtype", [nv.OUT_BF16, nv.OUT_FP32])
def test_config1_full(out_dtype):
    xb, wb = _layer(1, 128, 256, 512)
    w, wc, ws, wg = quantize_pinned(wb)
    oc, os_, og = oracle.nvfp4_encode(wb)
    np.testing.assert_array_equal(wc, oc)
    np.testing.assert_array_equal(ws, os_)
    y = nv.gemm(w, x=dev_bf16(xb), out_dtype=out_dtype)  # quantises X on the fly
    ref = oracle.gemm_w4a4(oracle.nvfp4_encode(xb), (oc, os_, og))
    _check(y_np(y), ref, "config 1", out_dtype == nv.OUT_BF16)
    # the pre-quantised activation path gives the same numbers
    a, *_ = quantize_pinned(xb)
    y2 = nv.gemm(w, a_q=a, out_dtype=out_dtype)
    np.testing.assert_array_equal(y_np(y2), y_np(y))


@pytest.fixture(scope="module")
def w_28672():
    wb = synth.weights(2, 1, 28672, 8192)
    w, wc, ws, wg = quantize_pinned(wb)
    return w, (wc, ws, wg[0])


@pytest.mark.parametrize("M", [1, 8, 16])
def test_decode_full(w_28672, M):
    w, wq = w_28672
    xb = synth.activations(2, 0, M, 8192, 0.005, 100.0)
    y = nv.gemm(w, x=dev_bf16(xb))
    ref = oracle.gemm_w4a4(oracle.nvfp4_encode(xb), wq)
    _check(y_np(y), ref, f"decode M={M}")


@pytest.mark.parametrize("N", [8192, 28672])
def test_prefill_sampled_rows(w_28672, N):
    # configuration 3 in the launch configuration the bench times (whole
    # tiles, BF16 output); 256 seeded rows plus the first and last
    if N == 28672:
        w, wq = w_28672
    else:
        wb = synth.weights(3, 1, 8192, 8192)
        w, wc, ws, wg = quantize_pinned(wb)
        wq = (wc, ws, wg[0])
    assert nv.gemm_kernel_path(4096, N, 8192) == nv.PATH_WHOLE_TILES
    xb = synth.activations(3, 0, 4096, 8192, 0.005, 100.0)
    y = y_np(nv.gemm(w, x=dev_bf16(xb)))
    rows = np.concatenate([[0, 4095], np.random.default_rng(N).choice(np.arange(1, 4095), 256, replace=False)])
    ref = oracle.gemm_w4a4(oracle.nvfp4_encode(xb), wq, rows=rows)
    _check(y[rows], ref, f"prefill N={N}")


@pytest.mark.parametrize("M,N,K", [(200, 384, 320), (129, 136, 64), (1, 130, 128), (64, 4096, 1024),
                                   (300, 1000, 256), (8, 1024, 8192), (33, 512, 2048), (2048, 256, 576)])
@pytest.mark.parametrize("out_dtype", [nv.OUT_BF16, nv.OUT_FP32])
def test_ragged_shapes(M, N, K, out_dtype):
    xb = synth.activations(9, 10, M, K, 0.01, 50.0)
    wb = synth.weights(9, 11, N, K)
    w, wc, ws, wg = quantize_pinned(wb)
    y = nv.gemm(w, x=dev_bf16(xb), out_dtype=out_dtype)
    ref = oracle.gemm_w4a4(oracle.nvfp4_encode(xb), (wc, ws, wg[0]))
    _check(y_np(y), ref, f"{M}x{N}x{K}", out_dtype == nv.OUT_BF16)


# Many-tile shapes: a last M tile of 1 or 44 rows (257, 300), partial N tiles
# and scale groups (N = 130, 384, 1000), one and many stages, more tiles
# than SMs (1024 x 4864: 8 x 19 tiles)
@pytest.mark.parametrize("M,N,K", [(257, 256, 256), (300, 130, 512), (384, 384, 768), (1000, 1000, 1024),
                                   (640, 2560, 2304), (1024, 4864, 1024)])
@pytest.mark.parametrize("out_dtype", [nv.OUT_BF16, nv.OUT_FP32])
def test_many_tile_shapes(M, N, K, out_dtype):
    assert nv.gemm_kernel_path(M, N, K) == nv.PATH_WHOLE_TILES
    xb = synth.activations(9, 12, M, K, 0.01, 50.0)
    wb = synth.weights(9, 13, N, K)
    w, wc, ws, wg = quantize_pinned(wb)
    work = nv.Workspace(nv.workspace_size(nv.OP_GEMM, M, N, K))
    y = nv.gemm(w, x=dev_bf16(xb), out_dtype=out_dtype, ws=work)
    assert work.status() == nv.OK
    ref = oracle.gemm_w4a4(oracle.nvfp4_encode(xb), (wc, ws, wg[0]))
    _check(y_np(y), ref, f"{M}x{N}x{K}", out_dtype == nv.OUT_BF16)


# The epilogue stores whole 32-byte row runs when every row of the output
# starts 32-byte aligned, 16-byte vectors when only 16-byte alignment holds
# and single elements otherwise: row strides and column offsets that give
# each level, for both output types, with the bytes around y untouched.
@pytest.mark.parametrize("out_dtype", [nv.OUT_BF16, nv.OUT_FP32])
# (row length N + extra elements, first column col0)
@pytest.mark.parametrize("extra,col0", [(0, 0), (8, 0), (16, 8), (32, 16), (3, 0)])
def test_output_alignment_levels(out_dtype, extra, col0):
    M, N, K = 300, 512, 512
    xb = synth.activations(9, 46, M, K, 0.01, 50.0)
    wb = synth.weights(9, 47, N, K)
    w, wc, ws, wg = quantize_pinned(wb)
    tdt = torch.bfloat16 if out_dtype == nv.OUT_BF16 else torch.float32
    big = torch.full((M, N + extra), 7.0, dtype=tdt, device="cuda")
    nv.gemm(w, x=dev_bf16(xb), y=big[:, col0:col0 + N], out_dtype=out_dtype)
    full = y_np(big)
    ref = oracle.gemm_w4a4(oracle.nvfp4_encode(xb), (wc, ws, wg[0]))
    _check(full[:, col0:col0 + N], ref, f"ld +{extra}, col {col0}", out_dtype == nv.OUT_BF16)
    assert (full[:, :col0] == 7.0).all() and (full[:, col0 + N:] == 7.0).all()
    if out_dtype == nv.OUT_BF16 and extra >= 4:
        # an output that does not start 16-byte aligned is refused
        with pytest.raises(nv.NVFP4Error) as e:
            nv.gemm(w, x=dev_bf16(xb), y=big[:, 4:4 + N], out_dtype=out_dtype)
        assert e.value.status == nv.ERR_INVALID_ARG


def test_output_row_stride_and_empty():
    xb, wb = _layer(1, 40, 256, 512)
    w, wc, ws, wg = quantize_pinned(wb)
    big = torch.full((40, 300), 7.0, dtype=torch.bfloat16, device="cuda")
    nv.gemm(w, x=dev_bf16(xb), y=big[:, :256])
    ref = oracle.gemm_w4a4(oracle.nvfp4_encode(xb), (wc, ws, wg[0]))
    full = y_np(big)
    _check(full[:, :256], ref, "strided output")
    assert (full[:, 256:] == 7.0).all()
    y = nv.gemm(w, x=torch.zeros((0, 512), dtype=torch.bfloat16, device="cuda"))
    assert y.shape == (0, 256)


# Shapes that run stream-K (M <= 128 and whole N tiles fill the SMs poorly):
# about 10 CTAs per tile (8, 4096, 8192), a ragged last N tile
# (16, 2944, 8192), the 128-wide N tile (8, 896, 16384) and M = 33.  The
# same call twice must give identical bits (flags cleared, slots reused).
@pytest.mark.parametrize("M,N,K", [(8, 4096, 8192), (16, 2944, 8192), (8, 896, 16384), (33, 4096, 8192)])
def test_streamk_shapes(M, N, K):
    xb = synth.activations(9, 40, M, K, 0.01, 50.0)
    wb = synth.weights(9, 41, N, K)
    w, wc, ws, wg = quantize_pinned(wb)
    work = nv.Workspace(nv.workspace_size(nv.OP_GEMM, M, N, K))
    x = dev_bf16(xb)
    y1 = y_np(nv.gemm(w, x=x, ws=work, out_dtype=nv.OUT_FP32))
    y2 = y_np(nv.gemm(w, x=x, ws=work, out_dtype=nv.OUT_FP32))
    assert work.status() == nv.OK
    np.testing.assert_array_equal(y1, y2)
    ref = oracle.gemm_w4a4(oracle.nvfp4_encode(xb), (wc, ws, wg[0]))
    _check(y1, ref, f"stream-K {M}x{N}x{K}", False)


def test_streamk_m128_sampled_rows():
    wb = synth.weights(9, 43, 4096, 8192)
    w, wc, ws, wg = quantize_pinned(wb)
    xb = synth.activations(2, 5, 128, 8192, 0.005, 100.0)
    y = y_np(nv.gemm(w, x=dev_bf16(xb)))
    rows = np.array([0, 1, 31, 32, 63, 64, 100, 127])
    ref = oracle.gemm_w4a4(oracle.nvfp4_encode(xb), (wc, ws, wg[0]), rows=rows)
    _check(y[rows], ref, "stream-K M=128")
