"""Grouped W4A8 (FP8 per-token activations x NVFP4 expert weights) and the
policy-routed grouped GEMM of BF16 activations against the oracle: the
128-expert top-8 up projection (gathered rows) and down projection
(contiguous rows) on sampled experts, small full cases with empty experts,
and the route each policy selects.  Operands are the oracle's encodes."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_common import dev_bf16, nv, nvfp4_device, y_np
from helpers import row_tolerance_ok

pytestmark = pytest.mark.gpu

C5 = synth.CONFIGS[5]


def expert_weights(E, N, K, tid):
    cs, ss, gs = [], [], []
    for e in range(E):
        c, s, g = oracle.nvfp4_encode(synth.weights(5, tid * 1000 + e, N, K))
        cs.append(c)
        ss.append(s)
        gs.append(g)
    wc, ws, wg = np.stack(cs), np.stack(ss), np.array(gs, np.float32)
    dev = nvfp4_device(wc.reshape(E * N, K // 2), ws.reshape(E * N, K // 16), wg, E * N, K)
    return dev, wc, ws, wg


def fp8_device(xb):
    a8, st = oracle.fp8_token_encode(xb)
    return a8, st, torch.from_numpy(a8).cuda(), torch.from_numpy(st).cuda()


def check_sampled(y, a8, st, row_idx, offsets, wc, ws, wg, experts, out_bf16=True):
    for e in experts:
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        ridx = None if row_idx is None else row_idx[lo:hi]
        off = np.array([0, hi - lo], np.int64)
        if ridx is None:   # contiguous rows: the expert's activation rows are lo..hi-1
            ref = oracle.gemm_grouped_w4a8(a8[lo:hi], st[lo:hi], None, off, wc[e:e + 1], ws[e:e + 1], wg[e:e + 1])
        else:
            ref = oracle.gemm_grouped_w4a8(a8, st, ridx, off, wc[e:e + 1], ws[e:e + 1], wg[e:e + 1])
        ok, worst = row_tolerance_ok(y[lo:hi], ref, out_bf16=out_bf16)
        assert ok, f"expert {e}: {worst}"


def test_up_projection_c5():
    E, H, I = C5["E"], C5["H"], C5["inter"]
    w, wc, ws, wg = expert_weights(E, I, H, 1)
    row_idx, offsets, counts, _ = synth.moe_routing()
    xb = synth.activations(5, 0, C5["T"], H, C5["outlier_frac"], C5["outlier_factor"])
    a8, st, a8_d, st_d = fp8_device(xb)
    R = int(offsets[-1])
    y = nv.grouped_w4a8_gemm(a8_d, st_d, torch.from_numpy(offsets).cuda(), w, I, R,
                             row_idx=torch.from_numpy(row_idx).cuda())
    order = np.argsort(counts)
    experts = sorted(set(order[:2].tolist() + order[-2:].tolist() + [0, 64, 127]))
    check_sampled(y_np(y), a8, st, row_idx, offsets, wc, ws, wg, experts)


def test_down_projection_c5_contiguous():
    E, H, I = C5["E"], C5["H"], C5["inter"]
    w, wc, ws, wg = expert_weights(E, H, I, 2)
    row_idx, offsets, counts, _ = synth.moe_routing()
    R = int(offsets[-1])
    xb = synth.activations(5, 2, R, I, C5["outlier_frac"], C5["outlier_factor"])
    a8, st, a8_d, st_d = fp8_device(xb)
    y = nv.grouped_w4a8_gemm(a8_d, st_d, torch.from_numpy(offsets).cuda(), w, H, R)
    order = np.argsort(counts)
    check_sampled(y_np(y), a8, st, None, offsets, wc, ws, wg, sorted(set(order[:2].tolist() + order[-2:].tolist())))


@pytest.mark.parametrize("indexed", [True, False])
def test_small_full_with_empty_experts(indexed):
    E, N, K, T = 6, 256, 320, 90
    counts = np.array([0, 37, 0, 1, 130, 0]) if not indexed else np.array([0, 37, 0, 1, 90, 0])
    w, wc, ws, wg = expert_weights(E, N, K, 3)
    rows_a = T if indexed else int(counts.sum())
    xb = synth.activations(9, 31, rows_a, K, 0.01, 50.0)
    a8, st, a8_d, st_d = fp8_device(xb)
    if indexed:
        row_idx, offsets = synth.moe_routing_from_counts(counts, T)
    else:
        row_idx, offsets = None, np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    R = int(offsets[-1])
    y = nv.grouped_w4a8_gemm(a8_d, st_d, torch.from_numpy(offsets).cuda(), w, N, R,
                             row_idx=None if row_idx is None else torch.from_numpy(row_idx).cuda(),
                             out_dtype=nv.OUT_FP32)
    ref = oracle.gemm_grouped_w4a8(a8, st, row_idx, offsets, wc, ws, wg)
    ok, worst = row_tolerance_ok(y_np(y), ref)
    assert ok, worst


@pytest.mark.parametrize("policy,sensitive,route", [(nv.POLICY_Q4, 0, 4), (nv.POLICY_Q8, 0, 8),
                                                     (nv.POLICY_AUTO, 1, 8), (nv.POLICY_AUTO, 0, 4)])
def test_policy_routed_grouped(policy, sensitive, route):
    E, N, K, T = 5, 384, 512, 200
    counts = np.array([60, 0, 143, 7, 90])
    w, wc, ws, wg = expert_weights(E, N, K, 4)
    xb = synth.activations(9, 32, T, K, 0.01, 50.0)
    row_idx, offsets = synth.moe_routing_from_counts(counts, T)
    R = int(offsets[-1])
    assert nv.policy_route(policy, sensitive) == route
    y = y_np(nv.grouped_gemm_x(dev_bf16(xb), torch.from_numpy(offsets).cuda(), w, N, R,
                               row_idx=torch.from_numpy(row_idx).cuda(), out_dtype=nv.OUT_FP32, policy=policy,
                               sensitive=sensitive))
    if route == 8:
        a8, st = oracle.fp8_token_encode(xb)
        ref = oracle.gemm_grouped_w4a8(a8, st, row_idx, offsets, wc, ws, wg)
    else:
        ref = oracle.gemm_grouped_w4a4(oracle.nvfp4_encode(xb), row_idx, offsets, wc, ws, wg)
    ok, worst = row_tolerance_ok(y, ref)
    assert ok, worst


def test_out_of_range_index_gives_zero_row():
    E, N, K, T = 2, 128, 128, 16
    w, wc, ws, wg = expert_weights(E, N, K, 5)
    xb = synth.activations(9, 33, T, K, 0.01, 50.0)
    a8, st, a8_d, st_d = fp8_device(xb)
    row_idx = np.array([0, 3, 5, 99, 2, 7], np.int32)   # routed row 3 points past the activations
    offsets = np.array([0, 4, 6], np.int64)
    y = y_np(nv.grouped_w4a8_gemm(a8_d, st_d, torch.from_numpy(offsets).cuda(), w, N, 6,
                                  row_idx=torch.from_numpy(row_idx).cuda(), out_dtype=nv.OUT_FP32))
    assert (y[3] == 0).all()
    good = np.array([0, 1, 2, 4, 5])
    ridx = row_idx.copy()
    ridx[3] = 0
    ref = oracle.gemm_grouped_w4a8(a8, st, ridx, offsets, wc, ws, wg)
    ok, worst = row_tolerance_ok(y[good], ref[good])
    assert ok, worst
