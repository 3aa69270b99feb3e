"""GPU quantisers against the oracle, bit for bit: packed E2M1 codes, E4M3
scale bytes and the second-level scale, on every configuration's tensors
(full size) and on edge cases; the per-token FP8 route likewise."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_common import dev_bf16, host, nv, quantize_gpu

pytestmark = pytest.mark.gpu

C = synth.CONFIGS


def _x(cfg, tid, M, K):
    c = C[cfg]
    return synth.activations(cfg, tid, M, K, c["outlier_frac"], c["outlier_factor"])


CASES = {
    "c1_x": lambda: _x(1, 0, 128, 512),
    "c1_w": lambda: synth.weights(1, 1, 256, 512),
    "c2_x_m1": lambda: _x(2, 0, 1, 8192),
    "c2_x_m8": lambda: _x(2, 0, 8, 8192),
    "c2_x_m16": lambda: _x(2, 0, 16, 8192),
    "c3_x": lambda: _x(3, 0, 4096, 8192),
    "c4_x": lambda: _x(4, 0, 2048, 4096),
    "c4_w": lambda: synth.weights(4, 1, 4096, 4096),
    "c5_x": lambda: _x(5, 0, 2048, 2048),
    "c5_down_in": lambda: _x(5, 2, 16384, 768),
}


def assert_same(bits, mode=nv.SCALE_TENSOR_FP32, layout=nv.LAYOUT_MMA_TILED):
    _, codes, scales, second = quantize_gpu(bits, mode, layout)
    if mode == nv.SCALE_TENSOR_FP32:
        oc, os_, og = oracle.nvfp4_encode(bits)
        assert second[0].view(np.uint32) == np.float32(og).view(np.uint32)
    else:
        oc, os_, om = oracle.nvfp4_encode_macro(bits)
        np.testing.assert_array_equal(second, om)
    bad_s = np.argwhere(scales != os_)
    assert bad_s.size == 0, f"{len(bad_s)} scale mismatches, first {bad_s[:3]}"
    bad_c = np.argwhere(codes != oc)
    assert bad_c.size == 0, f"{len(bad_c)} code mismatches, first {bad_c[:3]}"


@pytest.mark.parametrize("name", list(CASES))
def test_config_tensors_bit_exact(name):
    assert_same(CASES[name]())


@pytest.mark.parametrize("name", ["c1_x", "c2_x_m8", "c4_w"])
def test_row_major_layout_bit_exact(name):
    assert_same(CASES[name](), layout=nv.LAYOUT_ROW_MAJOR)


def test_largest_weight_tensor_bit_exact():
    # the 28672 x 8192 projection weights of the decode and prefill shapes
    assert_same(synth.weights(2, 1, 28672, 8192))


@pytest.mark.parametrize("name", ["c1_x", "c3_x", "c4_w"])
def test_macro_mode_bit_exact(name):
    assert_same(CASES[name](), mode=nv.SCALE_MACRO_FP16)


def _edge_cases():
    rng = np.random.default_rng(5)
    out = {}
    out["zeros"] = np.zeros((3, 128), np.uint16)
    out["neg_zeros"] = np.full((2, 64), 0x8000, np.uint16)
    x = np.zeros((5, 256), np.float32)
    x[2, 77] = -3.0e4
    out["single_outlier"] = synth.bf16_bits(x)
    out["bf16_subnormals"] = (rng.integers(0, 0x80, size=(4, 128)) | (rng.integers(0, 2, size=(4, 128)) << 15)).astype(np.uint16)
    out["huge"] = synth.bf16_bits(rng.uniform(-3e38, 3e38, size=(3, 64)).astype(np.float32))
    out["tiny_and_big"] = synth.bf16_bits(np.concatenate([rng.uniform(-1e-30, 1e-30, (2, 64)),
                                                          rng.uniform(-1e30, 1e30, (2, 64))]).astype(np.float32))
    out["ragged_rows_130"] = synth.activations(9, 1, 130, 320, 0.01, 50.0)
    out["one_row_k64"] = synth.activations(9, 2, 1, 64, 0.0, 1.0)
    out["all_grid_values"] = synth.bf16_bits(
        np.tile(np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6], np.float32), (4, 16)))
    out["midpoints"] = synth.bf16_bits(
        np.tile(np.array([6, .25, .75, 1.25, 1.75, 2.5, 3.5, 5, -6, -.25, -.75, -1.25, -1.75, -2.5, -3.5, -5],
                         np.float32), (3, 8)))
    return out


EDGE = _edge_cases()


@pytest.mark.parametrize("name", list(EDGE))
@pytest.mark.parametrize("layout", [nv.LAYOUT_MMA_TILED, nv.LAYOUT_ROW_MAJOR])
def test_edge_cases_bit_exact(name, layout):
    assert_same(EDGE[name], layout=layout)


def test_padded_scale_rows_are_zero():
    bits = synth.activations(9, 3, 130, 256, 0.01, 50.0)
    t = nv.quantize(dev_bf16(bits))
    from helpers import untile_scales
    full = untile_scales(host(t.scales), 256, 256)
    assert not full[130:].any()


def test_strided_input():
    bits = synth.activations(9, 4, 24, 512, 0.01, 50.0)
    wide = np.zeros((24, 640), np.uint16)
    wide[:, :512] = bits
    x = dev_bf16(wide)[:, :512]
    t = nv.quantize(x)
    oc, os_, og = oracle.nvfp4_encode(bits)
    np.testing.assert_array_equal(host(t.codes), oc)
    assert host(t.second)[0] == og


def test_nonfinite_input_sets_device_status():
    bits = synth.activations(9, 5, 8, 256, 0.0, 1.0)
    bits[3, 17] = 0x7FC0  # NaN
    ws = nv.Workspace(nv.workspace_size(nv.OP_QUANTIZE, 8, 0, 256))
    nv.quantize(dev_bf16(bits), ws=ws)
    assert ws.status() == nv.ERR_NONFINITE_INPUT
    assert ws.status() == nv.OK  # reading clears it
    bits[3, 17] = 0xFF80  # -inf, macro mode and the FP8 route too
    nv.quantize(dev_bf16(bits), mode=nv.SCALE_MACRO_FP16, ws=ws)
    assert ws.status() == nv.ERR_NONFINITE_INPUT
    nv.quantize_fp8(dev_bf16(bits), ws=ws)
    assert ws.status() == nv.ERR_NONFINITE_INPUT


def test_empty_input():
    x = torch.zeros((0, 256), dtype=torch.bfloat16, device="cuda")
    t = nv.quantize(x)
    assert host(t.second)[0] == 0


@pytest.mark.parametrize("shape", [(2048, 4096), (8, 8192), (1, 64), (130, 320)])
def test_fp8_per_token_bit_exact(shape):
    bits = synth.activations(4, 7, shape[0], shape[1], 0.01, 50.0)
    a, st = nv.quantize_fp8(dev_bf16(bits))
    oa, ost = oracle.fp8_token_encode(bits)
    np.testing.assert_array_equal(host(st).view(np.uint32), ost.view(np.uint32))
    ga = host(a)
    bad = np.argwhere(ga != oa)
    assert bad.size == 0, f"{len(bad)} FP8 mismatches, first {bad[:3]}"


def test_fp8_edge_cases():
    for name in ("zeros", "neg_zeros", "bf16_subnormals", "huge", "tiny_and_big", "single_outlier"):
        bits = EDGE[name]
        a, st = nv.quantize_fp8(dev_bf16(bits))
        oa, ost = oracle.fp8_token_encode(bits)
        np.testing.assert_array_equal(host(st).view(np.uint32), ost.view(np.uint32), err_msg=name)
        np.testing.assert_array_equal(host(a), oa, err_msg=name)


# Around the single-launch (one cluster, at most 32768 chunks of 8 values)
# and two-pass paths, and two-pass shapes whose rows are shorter than a
# CTA's stride (the index cursor wraps rows) or not a divisor of it.
@pytest.mark.parametrize("shape", [(32, 8192), (33, 8192), (4, 16384), (5000, 64), (300, 1088), (7, 4160),
                                   (4097, 128)])
def test_path_boundaries_bit_exact(shape):
    M, K = shape
    assert_same(synth.activations(9, 70 + M, M, K, 0.01, 50.0))


def test_nonfinite_input_two_pass_path():
    bits = synth.activations(9, 6, 64, 8192, 0.0, 1.0)   # 65536 chunks: two passes
    bits[63, 8191] = 0x7F80  # +inf in the very last element
    ws = nv.Workspace(nv.workspace_size(nv.OP_QUANTIZE, 64, 0, 8192))
    nv.quantize(dev_bf16(bits), ws=ws)
    assert ws.status() == nv.ERR_NONFINITE_INPUT


# The two-pass path loads 32-byte blocks when x and its row stride are 32-byte
# aligned and falls back to 16-byte loads otherwise: a 16-byte start offset
# and a row stride of 520 elements take the fallback.
@pytest.mark.parametrize("offset,pitch", [(8, 8200), (0, 8200), (8, 8192 + 16)])
def test_two_pass_alignment_fallback_bit_exact(offset, pitch):
    M, K = 64, 8192                      # 65536 chunks: two passes
    bits = synth.activations(9, 80 + offset, M, K, 0.01, 50.0)
    wide = np.zeros((M, pitch), np.uint16)
    wide[:, offset:offset + K] = bits
    x = dev_bf16(wide)[:, offset:offset + K]
    t = nv.quantize(x)
    oc, os_, og = oracle.nvfp4_encode(bits)
    np.testing.assert_array_equal(host(t.codes), oc)
    from helpers import untile_scales
    np.testing.assert_array_equal(untile_scales(host(t.scales), 128, K)[:M], os_)
    assert host(t.second)[0] == og


def _every_magnitude_tensor(top_bits, seed):
    """[64, 8192] BF16 (two-pass, contiguous: the staged path) whose 32768
    16-element blocks take every positive BF16 magnitude pattern 0x0001 ..
    top_bits as their maximum in turn (random sign and position), the other
    15 elements random magnitudes not above it; the tensor maximum is
    top_bits, which fixes the tensor scale."""
    rng = np.random.default_rng(seed)
    nb = 64 * 8192 // 16
    pats = (np.arange(nb) % top_bits + 1).astype(np.uint32)
    other = (rng.random((nb, 16)) * (pats[:, None] + 1)).astype(np.uint32)
    other = np.minimum(other, pats[:, None])
    other[np.arange(nb), rng.integers(0, 16, nb)] = pats
    sign = rng.integers(0, 2, (nb, 16)).astype(np.uint32) << 15
    return (other | sign).astype(np.uint16).reshape(64, 8192)


# The staged encode pass takes block scales from a per-CTA table when the
# tensor scale lies in [2^-100, 2^100] and the block maximum is at least
# 2^-123, and the direct division otherwise: every block magnitude up to
# the tensor maximum, with tensor maxima whose scale is inside the range
# (1.0: s = 2^-11.4), just inside and just outside either end
# (s = 2^-99.93, 2^-100.07, 2^99.95, 2^100.07) and far above it (2^116.6).
@pytest.mark.parametrize("top", [0x3F80, 0x1330, 0x1320, 0x7720, 0x7730, 0x7F7F])
def test_staged_path_every_block_magnitude(top):
    assert_same(_every_magnitude_tensor(top, top))
    assert_same(_every_magnitude_tensor(top, top + 1), layout=nv.LAYOUT_ROW_MAJOR)
