"""Pins for the oracle's NVFP4 / macro / per-token FP8 encoders.

Pins: the hand-derived row of tests/golden/nvfp4_row_example.txt, closed
forms (power-of-two tensor scales), exact round trips of representable
tensors, scaling and sign invariants, the zero and non-finite cases, the
reduction of macro mode to tensor mode, and torch's float8_e4m3fn cast for
the per-token FP8 route.
"""
import os

import numpy as np
import pytest
import torch

import synth
from conftest import GOLDEN


def bf16(vals):
    return synth.bf16_bits(np.asarray(vals, np.float32))


def _load_row_example():
    d = {}
    with open(os.path.join(GOLDEN, "nvfp4_row_example.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, rest = line.split(" ", 1)
            d[key] = rest.split()
    x = []
    for b in range(8):
        for tok in d[f"block{b}"]:
            v, p = tok.split(",")
            x.append(np.float32(float(v) * 2.0 ** int(p)))
    sg = np.uint32(int(d["s_g"][0], 16)).view(np.float32)
    scales = np.array([int(t, 16) for t in d["scales"]], np.uint8)
    codes = np.array([int(t, 16) for t in d["codes"]], np.uint8)
    return np.array(x, np.float32), sg, scales, codes


def test_golden_row_example(orc):
    x, sg, scales, codes = _load_row_example()
    assert x.size == 128 and codes.size == 64 and scales.size == 8
    xb = synth.bf16_bits(x)
    assert np.array_equal(synth.bf16_to_f32(xb), x)  # every input is exact in BF16
    c, s, g = orc.nvfp4_encode(xb[None, :])
    assert g == sg
    assert np.array_equal(s[0], scales)
    assert np.array_equal(c[0], codes), [hex(v) for v in c[0]]


@pytest.mark.parametrize("p", [-20, -8, 0, 5])
@pytest.mark.parametrize("j", [-9, -6, -3, 0, 2, 6])
def test_power_of_two_scale_closed_form(orc, p, j):
    # tensor amax 2688 * 2^p gives s_g = 2^p exactly; a block whose amax is
    # 6 * 2^j * 2^p then has u = 2^j exactly and scale E4M3(2^j).
    x = np.zeros((1, 32), np.float32)
    x[0, 0] = 2688.0 * 2.0 ** p
    x[0, 16] = 6.0 * 2.0 ** (j + p)
    c, s, g = orc.nvfp4_encode(bf16(x))
    assert g == np.float32(2.0 ** p)
    assert orc.e4m3_value(int(s[0, 1])) == 2.0 ** j
    assert orc.e4m3_value(int(s[0, 0])) == 448.0
    assert c[0, 8] & 0xF == 7  # the block maximum encodes as 6


def _representable(rng, R, K, p):
    """Codes, scale bytes and s_g = 2^p such that every block holds a +-6 code
    and one block has scale 448; the BF16 tensor v(c)*v(e)*2^p is exact."""
    E2M1 = [0, .5, 1, 1.5, 2, 3, 4, 6]
    nb = K // 16
    sc = rng.integers(0x08, 0x7F, size=(R, nb)).astype(np.uint8)  # normal scales
    sc[0, 0] = 0x7E
    mag = rng.integers(0, 8, size=(R, K))
    mag.reshape(R, nb, 16)[:, :, 0] = 7
    sign = rng.integers(0, 2, size=(R, K))
    vals = np.array(E2M1)[mag] * np.where(sign, -1.0, 1.0)
    scale_vals = np.array([float(torch.tensor([int(b)], dtype=torch.uint8).view(torch.float8_e4m3fn).float())
                           for b in range(256)])
    x = vals * np.repeat(scale_vals[sc], 16, axis=1) * 2.0 ** p
    codes = (mag | (sign << 3)).astype(np.uint8)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return x.astype(np.float32), packed, sc


@pytest.mark.parametrize("p", [-12, -3, 4])
def test_representable_tensor_round_trips(orc, p):
    rng = np.random.default_rng(100 + p)
    x, packed, sc = _representable(rng, 6, 256, p)
    xb = bf16(x)
    assert np.array_equal(synth.bf16_to_f32(xb), x)
    c, s, g = orc.nvfp4_encode(xb)
    assert g == np.float32(2.0 ** p)
    assert np.array_equal(s, sc)
    # a zero with a negative sign keeps its sign bit; compare values and signs
    assert np.array_equal(c, packed)
    deq = orc.nvfp4_dequant(c, s, g)
    assert np.array_equal(deq, x.astype(np.float64))


def test_power_of_two_invariance_and_negation(orc):
    x = synth.activations(1, 0, 16, 512, 0.01, 50.0)
    c0, s0, g0 = orc.nvfp4_encode(x)
    for k in (-7, 3, 11):
        xk = bf16(synth.bf16_to_f32(x) * np.float32(2.0 ** k))
        ck, sk, gk = orc.nvfp4_encode(xk)
        assert np.array_equal(ck, c0) and np.array_equal(sk, s0)
        assert gk == np.float32(g0 * np.float32(2.0 ** k))
    cn, sn, gn = orc.nvfp4_encode(x ^ np.uint16(0x8000))
    assert np.array_equal(sn, s0) and gn == g0
    assert np.array_equal(cn, c0 ^ np.uint8(0x88))


def test_zero_tensor(orc):
    x = np.zeros((3, 64), np.uint16)
    c, s, g = orc.nvfp4_encode(x)
    assert g == 0 and not s.any() and not c.any()
    c, s, g = orc.nvfp4_encode(x | np.uint16(0x8000))  # -0.0 everywhere
    assert g == 0 and not s.any() and np.all(c == 0x88)


def test_nonfinite_rejected(orc):
    x = np.zeros((2, 32), np.uint16)
    for bad in (0x7F80, 0xFF80, 0x7FC0):
        y = x.copy()
        y[1, 5] = bad
        with pytest.raises(orc.OracleError):
            orc.nvfp4_encode(y)
        with pytest.raises(orc.OracleError):
            orc.fp8_token_encode(y)


def test_block_error_bound(orc):
    # every element's dequantised value is the E2M1 grid point nearest to
    # x / d, so |x - x_hat| <= d * (half the local grid spacing) (+ rounding)
    x = synth.activations(1, 1, 32, 512, 0.01, 50.0)
    c, s, g = orc.nvfp4_encode(x)
    xf = synth.bf16_to_f32(x).astype(np.float64)
    deq = orc.nvfp4_dequant(c, s, g)
    d = np.repeat(np.array([[orc.e4m3_value(int(b)) for b in row] for row in s]), 16, axis=1) * float(g)
    q = np.abs(xf) / np.where(d > 0, d, 1)
    half = np.where(q < 2, 0.25, np.where(q < 4, 0.5, 1.0))
    ok = (np.abs(xf - deq) <= d * half * (1 + 1e-6)) | ((q >= 6) & (np.abs(deq) == 6 * d))
    assert ok.all()


def test_macro_reduces_to_tensor_mode(orc):
    # every 256-group has amax A with A / 2688 exactly representable in FP16,
    # so S = s_g and both modes produce identical codes and scales
    rng = np.random.default_rng(7)
    x = rng.standard_normal((5, 768)).astype(np.float32)
    x = np.clip(x, -2.5, 2.5)  # below A = 2.625
    A = np.float32(2688.0 * 2 ** -10)
    x[:, ::256] = A
    xb = bf16(x)
    c1, s1, g1 = orc.nvfp4_encode(xb)
    c2, s2, m2 = orc.nvfp4_encode_macro(xb)
    assert g1 == np.float32(2 ** -10)
    assert np.all(m2 == np.float16(2 ** -10).view(np.uint16))
    assert np.array_equal(c1, c2) and np.array_equal(s1, s2)


def test_macro_scale_values_and_saturation(orc):
    rng = np.random.default_rng(8)
    x = synth.bf16_to_f32(synth.activations(1, 2, 4, 512, 0.01, 50.0)).copy()
    x[1, 300] = 3.0e8  # amax/2688 above the FP16 range -> S saturates at 65504
    xb = bf16(x)
    c, s, m = orc.nvfp4_encode_macro(xb)
    xf = synth.bf16_to_f32(xb)
    for r in range(4):
        for grp in range(2):
            amax = np.float32(np.abs(xf[r, grp * 256:(grp + 1) * 256]).max())
            want = np.float16(min(float(amax / np.float32(2688.0)), 65504.0)).view(np.uint16)
            assert m[r, grp] == want
    assert m[1, 1] == 0x7BFF


def test_fp8_token_closed_form_and_torch(orc):
    x = synth.activations(4, 0, 8, 256, 0.01, 50.0)
    a, st = orc.fp8_token_encode(x)
    xf = synth.bf16_to_f32(x)
    amax = np.abs(xf).max(axis=1)
    assert np.array_equal(st, (amax / np.float32(448.0)).astype(np.float32))
    r = (np.float32(1.0) / st).astype(np.float32)
    q = (xf * r[:, None]).astype(np.float32)
    assert np.abs(q).max() <= 448.0 * (1 + 1e-6)
    q = np.clip(q, -448.0, 448.0)  # torch's cast does not saturate
    ref = torch.from_numpy(q).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(a, ref)


def test_fp8_token_power_of_two_rows_round_trip(orc):
    rng = np.random.default_rng(9)
    codes = rng.integers(0, 0x7F, size=(4, 64)).astype(np.uint8)
    codes[:, 0] = 0x7E  # each row's maximum is 448
    sign = rng.integers(0, 2, size=codes.shape).astype(np.uint8) << 7
    vals = torch.from_numpy(codes | sign).view(torch.float8_e4m3fn).float().numpy()
    p = np.array([-9, -2, 0, 5])
    x = vals * np.exp2(p)[:, None].astype(np.float32)
    a, st = orc.fp8_token_encode(bf16(x))
    assert np.array_equal(st, np.exp2(p).astype(np.float32))
    assert np.array_equal(a, codes | sign)


# ---- encode of binary32 values under a given tensor scale -------------------
# (the fused next-layer quantiser: the scale comes from calibration or a
# previous step instead of this tensor's amax)

def test_f32_scaled_equals_tensor_mode_when_scale_is_amax_over_2688(orc):
    for cfg, tid in [(1, 0), (2, 0), (9, 5)]:
        bits = synth.activations(cfg, tid, 24, 512, 0.01, 50.0)
        c, s, sg = orc.nvfp4_encode(bits)
        x = synth.bf16_to_f32(bits)
        c2, s2 = orc.nvfp4_encode_f32_scaled(x, sg)
        np.testing.assert_array_equal(c2, c)
        np.testing.assert_array_equal(s2, s)


def test_f32_scaled_saturates_when_the_scale_is_too_small(orc):
    # a constant block v with v / (6 s) = 1000 > 448: scale code 448 (0x7E)
    # and codes E2M1(v / (448 s)) = E2M1(13.4) -> 6 (0x7, sign kept)
    s = 1.0 / 2688.0
    v = 1000.0 * 6.0 * s
    x = np.full((2, 32), v, np.float32)
    x[1] = -v
    c, sc = orc.nvfp4_encode_f32_scaled(x, s)
    assert (sc == 0x7E).all()
    assert (c[0] == 0x77).all() and (c[1] == 0xFF).all()


def test_f32_scaled_zero_scale_gives_zero_codes_with_sign(orc):
    x = np.array([[0.5, -0.5] * 8], np.float32)
    c, sc = orc.nvfp4_encode_f32_scaled(x, 0.0)
    assert (sc == 0).all()
    assert (c == 0x80).all()            # even elements +0, odd elements -0


def test_f32_scaled_rejects_nonfinite_and_bad_scales(orc):
    x = np.zeros((1, 16), np.float32)
    x[0, 3] = np.inf
    with pytest.raises(orc.OracleError):
        orc.nvfp4_encode_f32_scaled(x, 1.0)
    with pytest.raises(orc.OracleError):
        orc.nvfp4_encode_f32_scaled(np.zeros((1, 16), np.float32), -1.0)
