"""W4A4 GEMM with the next layer's NVFP4 quantiser fused into its epilogue
(nvfp4_gemm_nvfp4_out) against the oracle's encode of the oracle's product
under the same given tensor scale.

Exact cases: operands built from E2M1 codes with power-of-two block and
tensor scales, so every partial sum and alpha * acc are exact in binary32
and the product the kernel encodes is the oracle's product exactly; codes,
tiled scales (padding rows included) and the reported amax must then match
bit for bit.  The only freedom left is the sign of an exactly zero output,
which the accumulation order decides; codes of zero outputs are compared
without their sign bit.

Realistic cases (the pages' activation/weight statistics at decode and
prefill sizes): the kernel's binary32 product differs from the FP64 product
by rounding, so an encode decision may flip where a value sits on a rounding
boundary.  Checked: at least 99.9 % of scale bytes and codes equal the
oracle's, every dequantised output lies within one block step (plus the
GEMM tolerance) of the FP64 product, and the amax is within the GEMM
tolerance."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_common import dev_bf16, host, nv, nvfp4_device
from helpers import row_tolerance_ok, tile_scales, untile_scales

pytestmark = pytest.mark.gpu

C = synth.CONFIGS
E4M3_HALF, E4M3_ONE, E4M3_TWO = 0x30, 0x38, 0x40


def exact_operand(rng, rows, K, scale_codes):
    codes = rng.integers(0, 256, size=(rows, K // 2)).astype(np.uint8)
    scales = rng.choice(np.array(scale_codes, np.uint8), size=(rows, K // 16))
    return codes, scales


def nibbles(packed):
    packed = np.asarray(packed, np.uint8)
    out = np.empty((packed.shape[0], packed.shape[1] * 2), np.uint8)
    out[:, 0::2] = packed & 0xF
    out[:, 1::2] = packed >> 4
    return out


def fused(w, s_y, a_q=None, x=None, amax=True):
    dev = w.codes.device
    s = torch.tensor([s_y], dtype=torch.float32, device=dev)
    y_amax = torch.zeros(1, dtype=torch.float32, device=dev) if amax else None
    out = nv.gemm_nvfp4_out(w, s, x=x, a_q=a_q, y_amax=y_amax)
    codes = host(out.codes)
    tiled = host(out.scales)
    am = float(host(y_amax)[0]) if amax else None
    return out, codes, tiled, am


def check_exact(y_ref, s_y, codes, tiled):
    M, N = y_ref.shape
    y32 = y_ref.astype(np.float32)
    assert np.array_equal(y32.astype(np.float64), y_ref), "test operands must give an exact product"
    rc, rs = oracle.nvfp4_encode_f32_scaled(y32, s_y)
    np.testing.assert_array_equal(tiled, tile_scales(rs, M, N))
    gn, rn = nibbles(codes), nibbles(rc)
    zero = y_ref == 0
    gn[zero] &= 7
    rn[zero] &= 7
    np.testing.assert_array_equal(gn, rn)
    return rc, rs


@pytest.mark.parametrize("M,N,K,scale_codes", [
    (200, 384, 512, (E4M3_HALF, E4M3_ONE, E4M3_TWO)),   # two M tiles, ragged; BN 128 tiles
    (8, 1024, 512, (E4M3_HALF, E4M3_ONE, E4M3_TWO)),    # decode-sized M
    (1, 512, 256, (E4M3_ONE,)),                          # single row, single K stage
    (8, 4096, 8192, (E4M3_ONE,)),                        # a shape the FP32 path runs stream-K
    (384, 768, 1024, (E4M3_HALF, E4M3_ONE)),             # three full M tiles, BN 256 tiles
])
def test_exact_operands_bit_exact(M, N, K, scale_codes):
    rng = np.random.default_rng(M * 7919 + N * 31 + K)
    ac, as_ = exact_operand(rng, M, K, scale_codes)
    wc, ws = exact_operand(rng, N, K, scale_codes)
    ac[M // 2] = 0                                        # one all-zero output row
    sa, sw = 0.125, 4.0                                   # alpha = 0.5 exactly
    y_ref = oracle.gemm_w4a4((ac, as_, sa), (wc, ws, sw))
    amax = float(np.abs(y_ref).max())
    a = nvfp4_device(ac, as_, sa, M, K)
    w = nvfp4_device(wc, ws, sw, N, K)
    for s_y in (np.float32(amax / 2688.0), np.float32(amax / 2688.0 / 64.0)):   # in range; saturating
        _, codes, tiled, am = fused(w, float(s_y), a_q=a)
        check_exact(y_ref, s_y, codes, tiled)
        assert am == np.float32(amax)


def test_zero_tensor_scale():
    # s_y = 0: every block scale is 0, so every code is a signed zero
    rng = np.random.default_rng(5)
    M, N, K = 40, 256, 256
    ac, as_ = exact_operand(rng, M, K, (E4M3_ONE,))
    wc, ws = exact_operand(rng, N, K, (E4M3_ONE,))
    y_ref = oracle.gemm_w4a4((ac, as_, 1.0), (wc, ws, 1.0))
    _, codes, tiled, _ = fused(nvfp4_device(wc, ws, 1.0, N, K), 0.0, a_q=nvfp4_device(ac, as_, 1.0, M, K),
                               amax=False)
    check_exact(y_ref, np.float32(0.0), codes, tiled)
    assert not tiled.any()


def test_chained_layers_exact():
    # layer 1 writes NVFP4 straight into layer 2's activation operand; the
    # oracle runs both layers from the oracle's own encodes (equal to the
    # kernel's, asserted first)
    rng = np.random.default_rng(11)
    M, K1, N1, N2 = 136, 512, 768, 512
    ac, as_ = exact_operand(rng, M, K1, (E4M3_HALF, E4M3_ONE, E4M3_TWO))
    w1c, w1s = exact_operand(rng, N1, K1, (E4M3_HALF, E4M3_ONE, E4M3_TWO))
    w2 = synth.weights(1, 77, N2, N1)
    w2c, w2s, w2g = oracle.nvfp4_encode(w2)
    y1 = oracle.gemm_w4a4((ac, as_, 0.25), (w1c, w1s, 2.0))
    s_y = np.float32(np.abs(y1).max() / 2688.0)
    out, codes, tiled, _ = fused(nvfp4_device(w1c, w1s, 2.0, N1, K1), float(s_y),
                                 a_q=nvfp4_device(ac, as_, 0.25, M, K1))
    rc, rs = check_exact(y1, s_y, codes, tiled)
    w2d = nvfp4_device(w2c, w2s, w2g, N2, N1)
    y2 = host(nv.gemm(w2d, a_q=out, out_dtype=nv.OUT_FP32)).astype(np.float64)
    ref = oracle.gemm_w4a4((rc, rs, s_y), (w2c, w2s, w2g))
    ok, worst = row_tolerance_ok(y2, ref)
    assert ok, worst


def check_realistic(y_ref, s_y, codes, tiled, am):
    M, N = y_ref.shape
    rc, rs = oracle.nvfp4_encode_f32_scaled(y_ref.astype(np.float32), s_y)
    gs = untile_scales(tiled, M, N)
    assert (gs == rs).mean() >= 0.999
    gn, rn = nibbles(codes), nibbles(rc)
    zero = y_ref == 0
    gn[zero] &= 7
    rn[zero] &= 7
    assert (gn == rn).mean() >= 0.999
    deq = oracle.nvfp4_dequant(codes, gs, s_y)
    # one block step: E2M1 spacing is at most 2 (between 4 and 6), so a
    # correctly rounded code is within the block scale d of y
    e4m3 = np.array([oracle.e4m3_value(c) for c in range(256)], np.float64)
    d_blk = np.repeat(e4m3[gs] * np.float64(s_y), 16, axis=1)
    row_norm = np.sqrt((y_ref ** 2).sum(axis=1, keepdims=True))
    assert (np.abs(deq - y_ref) <= d_blk * (1 + 1e-6) + 1e-3 * row_norm).all()
    assert abs(am - np.abs(y_ref).max()) <= 1e-3 * row_norm.max()


@pytest.mark.parametrize("M", [1, 8, 16])
def test_decode_shapes_realistic(M):
    N, K = 4096, C[2]["K"]
    xb = synth.activations(2, 40 + M, M, K, C[2]["outlier_frac"], C[2]["outlier_factor"])
    wb = synth.weights(2, 41, N, K)
    ac, as_, ag = oracle.nvfp4_encode(xb)
    wc, ws, wg = oracle.nvfp4_encode(wb)
    y_ref = oracle.gemm_w4a4((ac, as_, ag), (wc, ws, wg))
    s_y = np.float32(np.abs(y_ref).max() / 2688.0)
    w = nvfp4_device(wc, ws, wg, N, K)
    # from pre-quantised activations and from BF16 through the on-the-fly quantiser
    for kw in (dict(a_q=nvfp4_device(ac, as_, ag, M, K)), dict(x=dev_bf16(xb))):
        _, codes, tiled, am = fused(w, float(s_y), **kw)
        check_realistic(y_ref, s_y, codes, tiled, am)


def test_prefill_tile_realistic():
    M, N, K = 320, 2048, 4096
    xb = synth.activations(3, 50, M, K, C[3]["outlier_frac"], C[3]["outlier_factor"])
    wb = synth.weights(3, 51, N, K)
    ac, as_, ag = oracle.nvfp4_encode(xb)
    wc, ws, wg = oracle.nvfp4_encode(wb)
    y_ref = oracle.gemm_w4a4((ac, as_, ag), (wc, ws, wg))
    s_y = np.float32(np.abs(y_ref).max() / 2688.0)
    _, codes, tiled, am = fused(nvfp4_device(wc, ws, wg, N, K), float(s_y), x=dev_bf16(xb))
    check_realistic(y_ref, s_y, codes, tiled, am)


def test_argument_errors():
    rng = np.random.default_rng(3)
    ac, as_ = exact_operand(rng, 8, 256, (E4M3_ONE,))
    wc, ws = exact_operand(rng, 96, 256, (E4M3_ONE,))
    a = nvfp4_device(ac, as_, 1.0, 8, 256)
    w = nvfp4_device(wc, ws, 1.0, 96, 256)          # N = 96: the output's K is not a multiple of 64
    s = torch.ones(1, dtype=torch.float32, device="cuda")
    with pytest.raises(nv.NVFP4Error) as e:
        nv.gemm_nvfp4_out(w, s, a_q=a, out=nv.NVFP4Tensor(torch.empty((8, 48), dtype=torch.uint8, device="cuda"),
                                                          torch.empty(2048, dtype=torch.uint8, device="cuda"), s,
                                                          8, 96))
    assert e.value.status == nv.ERR_UNSUPPORTED_SHAPE
