"""Grouped (mixture-of-experts) W4A4 GEMM against the oracle: the
configuration-5 up projection (gathered token rows, 128 experts, top-8) and
down projection (contiguous rows), checked expert by expert on a sample of
experts that includes the largest and smallest, plus a small full case with
forced-empty experts and a heavy (Plackett-Luce Zipf) routing."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_common import dev_bf16, host, nv, quantize_pinned, y_np
from helpers import row_tolerance_ok

pytestmark = pytest.mark.gpu

C5 = synth.CONFIGS[5]


def stacked_weights(E, N, K, tid):
    """E experts' BF16 weights quantised one expert at a time (one tensor scale
    each) and stacked; returns the device tensor and the host codes/scales."""
    codes, scales, sgs = [], [], []
    dev_codes, dev_scales = [], []
    for e in range(E):
        wb = synth.weights(5, tid * 1000 + e, N, K)
        t, c, s, g = quantize_pinned(wb)
        codes.append(c)
        scales.append(s)
        sgs.append(g[0])
        dev_codes.append(t.codes)
        dev_scales.append(t.scales)
    w = nv.NVFP4Tensor(torch.cat(dev_codes), torch.cat(dev_scales),
                       torch.tensor(np.array(sgs, np.float32)).cuda(), E * N, K)
    return w, np.stack(codes), np.stack(scales), np.array(sgs, np.float32)


def check_experts(y, a_q, row_idx, offsets, wc, ws, wg, experts):
    for e in experts:
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        rows = row_idx[lo:hi].astype(np.int64) if row_idx is not None else np.arange(lo, hi)
        ref = oracle.gemm_w4a4(a_q, (wc[e], ws[e], wg[e]), rows=rows)
        ok, worst = row_tolerance_ok(y[lo:hi], ref, out_bf16=True)
        assert ok, f"expert {e}: {worst}"


@pytest.fixture(scope="module")
def up_weights():
    return stacked_weights(C5["E"], C5["inter"], C5["H"], 1)


def test_moe_up_projection(up_weights):
    w, wc, ws, wg = up_weights
    row_idx, offsets, counts, _ = synth.moe_routing()
    xb = synth.activations(5, 0, C5["T"], C5["H"], C5["outlier_frac"], C5["outlier_factor"])
    a, ac, as_, ag = quantize_pinned(xb)
    T = int(offsets[-1])
    y = nv.grouped_gemm(a, torch.from_numpy(offsets).cuda(), w, C5["inter"], T,
                        row_idx=torch.from_numpy(row_idx).cuda())
    yn = y_np(y)
    order = np.argsort(counts)
    experts = sorted(set(order[:3].tolist() + order[-3:].tolist() + [0, 1, 64, 127]))
    check_experts(yn, (ac, as_, ag[0]), row_idx, offsets, wc, ws, wg, experts)


def test_moe_down_projection():
    E, N, K = C5["E"], C5["H"], C5["inter"]
    w, wc, ws, wg = stacked_weights(E, N, K, 2)
    row_idx, offsets, counts, _ = synth.moe_routing()
    T = int(offsets[-1])
    xb = synth.activations(5, 2, T, K, C5["outlier_frac"], C5["outlier_factor"])
    a, ac, as_, ag = quantize_pinned(xb)
    y = nv.grouped_gemm(a, torch.from_numpy(offsets).cuda(), w, N, T)
    yn = y_np(y)
    order = np.argsort(counts)
    experts = sorted(set(order[:2].tolist() + order[-2:].tolist() + [5, 77]))
    check_experts(yn, (ac, as_, ag[0]), None, offsets, wc, ws, wg, experts)


@pytest.mark.parametrize("indexed", [True, False])
def test_small_full_with_empty_experts(indexed):
    E, N, K, T = 6, 256, 320, 90
    counts = np.array([0, 37, 0, 1, 130, 0])
    w, wc, ws, wg = stacked_weights(E, N, K, 3)
    xb = synth.activations(9, 30, T if indexed else int(counts.sum()), K, 0.01, 50.0)
    a, ac, as_, ag = quantize_pinned(xb)
    if indexed:
        row_idx, offsets = synth.moe_routing_from_counts(np.minimum(counts, T), T)
    else:
        row_idx, offsets = None, np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    total = int(offsets[-1])
    y = nv.grouped_gemm(a, torch.from_numpy(offsets).cuda(), w, N, total,
                        row_idx=None if row_idx is None else torch.from_numpy(row_idx).cuda(),
                        out_dtype=nv.OUT_FP32)
    ref = oracle.gemm_grouped_w4a4((ac, as_, ag[0]), row_idx, offsets, wc, ws, wg)
    ok, worst = row_tolerance_ok(y_np(y), ref)
    assert ok, worst


@pytest.mark.parametrize("out_dtype", [nv.OUT_BF16, nv.OUT_FP32])
def test_contiguous_expert_boundaries_every_row(out_dtype):
    # contiguous rows tile from the 128-row boundary at or below each
    # expert's first row; these boundaries fall at every kind of offset
    # (inside a block, on a block edge, a 1-row expert, an empty one, an
    # expert spanning three blocks), and every row is checked against its
    # own expert's product, so a tile that stored the previous expert's
    # leading rows would fail
    E, N, K = 7, 256, 512
    counts = np.array([1, 127, 129, 0, 255, 70, 128])
    w, wc, ws, wg = stacked_weights(E, N, K, 4)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    total = int(offsets[-1])
    xb = synth.activations(9, 31, total, K, 0.01, 50.0)
    a, ac, as_, ag = quantize_pinned(xb)
    y = nv.grouped_gemm(a, torch.from_numpy(offsets).cuda(), w, N, total, out_dtype=out_dtype)
    ref = oracle.gemm_grouped_w4a4((ac, as_, ag[0]), None, offsets, wc, ws, wg)
    ok, worst = row_tolerance_ok(y_np(y), ref, out_bf16=out_dtype == nv.OUT_BF16)
    assert ok, worst


def test_heavy_zipf_routing(up_weights):
    w, wc, ws, wg = up_weights
    row_idx, offsets, counts, _ = synth.moe_routing(literal=True)
    assert counts.max() > 1000
    xb = synth.activations(5, 0, C5["T"], C5["H"], C5["outlier_frac"], C5["outlier_factor"])
    a, ac, as_, ag = quantize_pinned(xb)
    y = nv.grouped_gemm(a, torch.from_numpy(offsets).cuda(), w, C5["inter"], int(offsets[-1]),
                        row_idx=torch.from_numpy(row_idx).cuda())
    e_big = int(np.argmax(counts))
    check_experts(y_np(y), (ac, as_, ag[0]), row_idx, offsets, wc, ws, wg, [e_big, int(np.argmin(counts))])
