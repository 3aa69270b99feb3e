"""Pins for the oracle's element formats (E2M1, E4M3, FP16, BF16).

Each pin comes from outside the oracle: the hand-derived E2M1 table of
tests/golden/e2m1_codes.txt, torch's float8_e4m3fn cast, numpy's float16
cast, and round-half-to-even at a fixed binary precision (Python's round()).
"""
import math
import os
import struct

import numpy as np
import pytest
import torch

from conftest import GOLDEN


def _golden_e2m1():
    rows = []
    with open(os.path.join(GOLDEN, "e2m1_codes.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                c, v = line.split()
                rows.append((int(c), float(v)))
    return rows


def _f32(x):
    return struct.unpack("<f", struct.pack("<f", x))[0]


def rne_to_precision(x, mant_bits, min_exp, max_val):
    """Textbook round-to-nearest-even of |x| onto a binary grid with
    `mant_bits` fraction bits, smallest normal exponent `min_exp` (subnormals
    spaced 2^(min_exp - mant_bits)), saturated at max_val.  Uses Python's
    round(), which breaks ties to the even integer."""
    a = abs(x)
    e = max(math.frexp(a)[1] - 1, min_exp) if a > 0 else min_exp
    ulp = 2.0 ** (e - mant_bits)
    q = round(a / ulp) * ulp
    q = min(q, max_val)
    return -q if math.copysign(1.0, x) < 0 else q


def test_e2m1_table_matches_golden(orc):
    rows = _golden_e2m1()
    assert len(rows) == 16
    for c, v in rows:
        got = orc.e2m1_value(c)
        assert got == v and math.copysign(1, got) == math.copysign(1, v), (c, got, v)


def test_e2m1_encode_against_round_half_even(orc):
    rng = np.random.default_rng(1)
    xs = list(rng.uniform(-8, 8, 20000)) + list(rng.uniform(-0.8, 0.8, 5000))
    # every midpoint and every grid point, and their float neighbours
    grid = [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    mids = [(a + b) / 2 for a, b in zip(grid, grid[1:])]
    for p in grid + mids + [6.5, 7, 100, 1e30]:
        for s in (1, -1):
            v = s * p
            xs += [v, float(np.nextafter(np.float32(v), np.float32(np.inf))),
                   float(np.nextafter(np.float32(v), np.float32(-np.inf)))]
    for x in xs:
        x = _f32(x)
        want = rne_to_precision(x, 1, 0, 6.0)
        got = orc.e2m1_value(orc.e2m1_encode(x))
        assert got == want and math.copysign(1, got) == math.copysign(1, want), (x, got, want)


def test_e2m1_round_trip_all_codes(orc):
    for c in range(16):
        assert orc.e2m1_encode(orc.e2m1_value(c)) == c


def test_e4m3_decode_all_codes_match_torch(orc):
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        got = orc.e4m3_value(c)
        if math.isnan(ref[c]):
            assert math.isnan(got), c
        else:
            assert got == ref[c] and math.copysign(1, got) == math.copysign(1, ref[c]), c
    assert orc.e4m3_value(0x7E) == 448.0 and orc.e4m3_value(0x01) == 2.0 ** -9


def test_e4m3_encode_in_range_matches_torch(orc):
    rng = np.random.default_rng(2)
    xs = np.concatenate([
        rng.uniform(-448, 448, 20000), rng.uniform(-1, 1, 20000),
        rng.uniform(-2 ** -6, 2 ** -6, 20000),
        np.exp2(rng.uniform(-12, 8.8, 20000)),
    ]).astype(np.float32)
    # torch's cast is round-to-nearest-even inside the finite range
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for x, r in zip(xs.tolist(), ref.tolist()):
        assert orc.e4m3_encode(x) == r, (x, orc.e4m3_encode(x), r)


def test_e4m3_encode_ties_and_saturation(orc):
    # every midpoint between neighbouring positive codes goes to the even code
    for c in range(0, 0x7E):
        lo, hi = orc.e4m3_value(c), orc.e4m3_value(c + 1)
        mid = (lo + hi) / 2
        assert _f32(mid) == mid
        want = c if c % 2 == 0 else c + 1
        assert orc.e4m3_encode(mid) == want, (c, mid)
        assert orc.e4m3_encode(-mid) == 0x80 | want
    for x in (448.0, 449.0, 464.0, 465.0, 1e6, 3e38, float("inf")):
        assert orc.e4m3_encode(x) == 0x7E
        assert orc.e4m3_encode(-x) == 0xFE
    for x in (1e-4, 2 ** -10, -2 ** -10):  # below half the smallest subnormal
        assert orc.e4m3_encode(x) & 0x7F == 0
    assert orc.e4m3_encode(-0.0) == 0x80


def test_e4m3_against_round_half_even(orc):
    rng = np.random.default_rng(3)
    for x in np.concatenate([rng.uniform(-500, 500, 5000),
                             np.exp2(rng.uniform(-14, 9, 5000))]).astype(np.float32).tolist():
        want = rne_to_precision(x, 3, -6, 448.0)
        assert orc.e4m3_value(orc.e4m3_encode(x)) == want, x


def test_e4m3_round_trip_all_finite_codes(orc):
    for c in list(range(0, 0x7F)) + list(range(0x80, 0xFF)):
        assert orc.e4m3_encode(orc.e4m3_value(c)) == c, c


def test_fp16_matches_numpy(orc):
    rng = np.random.default_rng(4)
    xs = np.concatenate([rng.uniform(-65000, 65000, 5000),
                         np.exp2(rng.uniform(-26, 15.9, 20000)),
                         -np.exp2(rng.uniform(-26, 15.9, 5000))]).astype(np.float32)
    ref = xs.astype(np.float16).view(np.uint16)
    for x, r in zip(xs.tolist(), ref.tolist()):
        assert orc.fp16_encode(x) == r, (x, hex(orc.fp16_encode(x)), hex(r))
    for h in (0x0000, 0x0001, 0x03FF, 0x0400, 0x3C00, 0x7BFF, 0x8001, 0xFBFF):
        assert orc.fp16_value(h) == float(np.uint16(h).view(np.float16))
    # saturation instead of infinity
    assert orc.fp16_encode(65520.0) == 0x7BFF and orc.fp16_encode(1e30) == 0x7BFF
    assert orc.fp16_encode(-1e30) == 0xFBFF


def test_bf16_value(orc):
    for b in (0x0000, 0x3F80, 0xBF80, 0x7F7F, 0x0001, 0x4228):
        want = struct.unpack("<f", struct.pack("<I", b << 16))[0]
        assert orc.bf16_value(b) == want


@pytest.mark.parametrize("fmt", ["e2m1", "e4m3"])
def test_encode_preserves_sign_of_zero_results(orc, fmt):
    enc = orc.e2m1_encode if fmt == "e2m1" else orc.e4m3_encode
    neg = 0x8 if fmt == "e2m1" else 0x80
    tiny = 0.2 if fmt == "e2m1" else 1e-4
    assert enc(-tiny) == neg and enc(tiny) == 0 and enc(-0.0) == neg and enc(0.0) == 0


def test_bf16_round_matches_torch_cast(orc):
    # the oracle's bf16_round against torch's float32 -> bfloat16 cast (round to
    # nearest even): random values across many binades, exact ties (the
    # dropped half exactly 0x8000 with even and odd kept bits) and signed zero
    rng = np.random.default_rng(7)
    v = (rng.standard_normal(20000) * np.exp2(rng.integers(-60, 60, 20000))).astype(np.float32)
    ties = (np.arange(512, dtype=np.uint32) << 16 | 0x8000).view(np.float32)
    v = np.concatenate([v, ties, -ties, np.array([0.0, -0.0], np.float32)])
    got = orc.bf16_round(v.astype(np.float64))
    want = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(got, want)
