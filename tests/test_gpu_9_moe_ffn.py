"""Mixture-of-experts feed-forward epilogues of the grouped W4A4 GEMM
against the oracle: the SwiGLU up projection (BF16/FP32 and NVFP4 outputs)
and the gate-weighted down-projection combine, on the 128-expert top-8
routing workload (checked on sampled experts / sampled tokens) and on small
full cases with empty experts, a residual and out-of-range token indices.
All operands are the oracle's encodes of the synthetic BF16 tensors."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_common import host, nv, nvfp4_device, y_np
from helpers import interleave_gate_up, row_tolerance_ok, tile_scales, untile_scales

pytestmark = pytest.mark.gpu

C5 = synth.CONFIGS[5]


def expert_weights(E, n_rows, K, tid):
    """Oracle encodes of E experts' BF16 weights [n_rows, K] (one tensor
    scale each): codes [E, n_rows, K/2], scales [E, n_rows, K/16], sg [E]."""
    cs, ss, gs = [], [], []
    for e in range(E):
        c, s, g = oracle.nvfp4_encode(synth.weights(5, tid * 1000 + e, n_rows, K))
        cs.append(c)
        ss.append(s)
        gs.append(g)
    return np.stack(cs), np.stack(ss), np.array(gs, np.float32)


def stacked_device(codes, scales, sg):
    E, n, half = codes.shape
    K = half * 2
    return nvfp4_device(codes.reshape(E * n, half), scales.reshape(E * n, K // 16), sg, E * n, K)


def gate_up_weights(E, I, K, tid):
    c, s, g = expert_weights(E, 2 * I, K, tid)       # rows [gate; up] per expert
    gate, up = (c[:, :I], s[:, :I]), (c[:, I:], s[:, I:])
    dev = stacked_device(interleave_gate_up(gate[0], up[0]), interleave_gate_up(gate[1], up[1]), g)
    return dev, gate, up, g


def sub_experts(offsets, row_idx, experts, *per_expert):
    """The routed rows of the listed experts as a smaller grouped problem."""
    rows, counts = [], []
    for e in experts:
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        rows.append(np.arange(lo, hi))
        counts.append(hi - lo)
    rows = np.concatenate(rows)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    sel = [tuple(x[list(experts)] for x in arr) if isinstance(arr, tuple) else arr[list(experts)]
           for arr in per_expert]
    return rows, off, (None if row_idx is None else row_idx[rows]), sel


@pytest.fixture(scope="module")
def c5_up():
    E, H, I = C5["E"], C5["H"], C5["inter"]
    row_idx, offsets, counts, logits = synth.moe_routing()
    xb = synth.activations(5, 0, C5["T"], H, C5["outlier_frac"], C5["outlier_factor"])
    a = oracle.nvfp4_encode(xb)
    w, gate, up, g = gate_up_weights(E, I, H, 3)
    return dict(row_idx=row_idx, offsets=offsets, counts=counts, logits=logits, a=a,
                a_dev=nvfp4_device(a[0], a[1], a[2], C5["T"], H), w=w, gate=gate, up=up, g=g)


def up_reference(d, experts):
    rows, off, ridx, (gate, up, g) = sub_experts(d["offsets"], d["row_idx"], experts, d["gate"], d["up"], d["g"])
    return rows, oracle.moe_up_swiglu(d["a"], ridx, off, gate, up, g)


def sample_experts(counts):
    order = np.argsort(counts)
    return sorted(set(order[:2].tolist() + order[-2:].tolist() + [0, 64, 127]))


@pytest.mark.parametrize("out_dtype", [nv.OUT_BF16, nv.OUT_FP32])
def test_up_swiglu_c5(c5_up, out_dtype):
    d = c5_up
    R = int(d["offsets"][-1])
    h = nv.moe_up_swiglu(d["a_dev"], torch.from_numpy(d["offsets"]).cuda(), d["w"], C5["inter"], R,
                         row_idx=torch.from_numpy(d["row_idx"]).cuda(), out_dtype=out_dtype)
    hn = y_np(h)
    rows, ref = up_reference(d, sample_experts(d["counts"]))
    ok, worst = row_tolerance_ok(hn[rows], ref, out_bf16=out_dtype == nv.OUT_BF16)
    assert ok, worst


def nibbles(packed):
    out = np.empty((packed.shape[0], packed.shape[1] * 2), np.uint8)
    out[:, 0::2] = packed & 0xF
    out[:, 1::2] = packed >> 4
    return out


def test_up_swiglu_c5_nvfp4_out(c5_up):
    d = c5_up
    R, I = int(d["offsets"][-1]), C5["inter"]
    rows, ref = up_reference(d, sample_experts(d["counts"]))
    s_h = np.float32(np.abs(ref).max() / 2688.0)
    amax = torch.zeros(1, dtype=torch.float32, device="cuda")
    hq = nv.moe_up_swiglu(d["a_dev"], torch.from_numpy(d["offsets"]).cuda(), d["w"], I, R,
                          row_idx=torch.from_numpy(d["row_idx"]).cuda(),
                          s_h=torch.tensor([s_h], device="cuda"), h_amax=amax)
    codes = host(hq.codes)[rows]
    gs = untile_scales(host(hq.scales), R, I)[rows]
    rc, rs = oracle.nvfp4_encode_f32_scaled(ref.astype(np.float32), s_h)
    assert (gs == rs).mean() >= 0.999
    gn, rn = nibbles(codes), nibbles(rc)
    gn[ref == 0] &= 7
    rn[ref == 0] &= 7
    assert (gn == rn).mean() >= 0.999
    e4m3 = np.array([oracle.e4m3_value(c) for c in range(256)], np.float64)
    d_blk = np.repeat(e4m3[gs] * np.float64(s_h), 16, axis=1)
    row_norm = np.sqrt((ref ** 2).sum(axis=1, keepdims=True))
    deq = oracle.nvfp4_dequant(codes, gs, s_h)
    assert (np.abs(deq - ref) <= d_blk * (1 + 1e-6) + 1e-3 * row_norm).all()
    # the reported amax covers every routed row, so it bounds the sample's
    assert float(host(amax)[0]) >= np.abs(ref).max() * (1 - 1e-3)


@pytest.fixture(scope="module")
def c5_down(c5_up):
    E, H, I = C5["E"], C5["H"], C5["inter"]
    d = c5_up
    R = int(d["offsets"][-1])
    hb = synth.activations(5, 4, R, I, C5["outlier_frac"], C5["outlier_factor"])
    h = oracle.nvfp4_encode(hb)
    wc, ws, wg = expert_weights(E, H, I, 4)
    gate_w = synth.moe_gate_weights(d["logits"], d["row_idx"], d["offsets"], C5["topk"])
    return dict(h=h, h_dev=nvfp4_device(h[0], h[1], h[2], R, I), wc=wc, ws=ws, wg=wg,
                w_dev=stacked_device(wc, ws, wg), gate_w=gate_w)


def test_down_combine_c5_sampled_tokens(c5_up, c5_down):
    d, q = c5_up, c5_down
    T, H = C5["T"], C5["H"]
    tok = d["row_idx"]
    y = torch.zeros((T, H), dtype=torch.float32, device="cuda")
    nv.moe_down_combine(q["h_dev"], torch.from_numpy(d["offsets"]).cuda(), q["w_dev"], H,
                        torch.from_numpy(tok).cuda(), torch.from_numpy(q["gate_w"]).cuda(), y)
    yn = y_np(y)
    # the oracle over every routed row of a token sample (its rows stay in
    # expert order, so they form a grouped problem of their own)
    sample = np.concatenate([[0, T - 1], np.random.default_rng(1).choice(np.arange(1, T - 1), 30, replace=False)])
    keep = np.isin(tok, sample)
    rows = np.nonzero(keep)[0]
    expert_of_row = np.repeat(np.arange(C5["E"]), np.diff(d["offsets"]))
    counts = np.bincount(expert_of_row[rows], minlength=C5["E"])
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    h = q["h"]
    ref = oracle.moe_down_combine((h[0][rows], h[1][rows], h[2]), off, q["wc"], q["ws"], q["wg"], tok[rows],
                                  q["gate_w"][rows], T)
    ok, worst = row_tolerance_ok(yn[sample], ref[sample])
    assert ok, worst
    untouched = np.setdiff1d(np.arange(T), tok)
    assert (yn[untouched] == 0).all()


def small_problem(seed, T=64, H=256, I=256, counts=(0, 37, 0, 1, 64, 0, 24)):
    rng = np.random.default_rng(seed)
    E = len(counts)
    row_idx, offsets = synth.moe_routing_from_counts(np.array(counts), T)
    xb = synth.activations(9, 60 + seed, T, H, 0.01, 50.0)
    return rng, E, row_idx, offsets, xb


def test_small_full_chain_with_residual():
    # x -> up + SwiGLU (NVFP4 out) -> down + combine into a residual, whole
    # problem; empty experts, one row with an out-of-range token index
    rng, E, row_idx, offsets, xb = small_problem(2)
    T, H, I = 64, 256, 256
    R = int(offsets[-1])
    a = oracle.nvfp4_encode(xb)
    w, gate, up, g = gate_up_weights(E, I, H, 7)
    h_ref = oracle.moe_up_swiglu(a, row_idx, offsets, gate, up, g)
    s_h = np.float32(np.abs(h_ref).max() / 2688.0)
    off_d = torch.from_numpy(offsets).cuda()
    hq = nv.moe_up_swiglu(nvfp4_device(a[0], a[1], a[2], T, H), off_d, w, I, R,
                          row_idx=torch.from_numpy(row_idx).cuda(), s_h=torch.tensor([s_h], device="cuda"))
    # padding rows of the last 128-row scale tile are zero
    tiled = host(hq.scales)
    full = untile_scales(tiled, -(-R // 128) * 128, I)
    assert not full[R:].any()
    hc, hs = oracle.nvfp4_encode_f32_scaled(h_ref.astype(np.float32), s_h)
    wc, ws, wg = expert_weights(E, H, I, 8)
    tok = row_idx.copy()
    gate_w = rng.uniform(0.05, 1.0, size=R).astype(np.float32)
    tok_dev = tok.copy()
    tok_dev[5] = T + 3                                   # adds nothing
    y0 = rng.standard_normal((T, H)).astype(np.float32)
    y = torch.from_numpy(y0.copy()).cuda()
    nv.moe_down_combine(hq, off_d, stacked_device(wc, ws, wg), H, torch.from_numpy(tok_dev).cuda(),
                        torch.from_numpy(gate_w).cuda(), y)
    gw_ref = gate_w.copy()
    gw_ref[5] = 0.0
    contrib = oracle.moe_down_combine((hc, hs, s_h), offsets, wc, ws, wg, tok, gw_ref, T)
    got = y_np(y) - y0.astype(np.float64)
    ok, worst = row_tolerance_ok(got, contrib, rel=2e-3)
    assert ok, worst


@pytest.mark.parametrize("out_dtype", [nv.OUT_BF16, nv.OUT_FP32])
def test_small_up_swiglu_full(out_dtype):
    rng, E, row_idx, offsets, xb = small_problem(3)
    T, H, I = 64, 256, 256
    R = int(offsets[-1])
    a = oracle.nvfp4_encode(xb)
    w, gate, up, g = gate_up_weights(E, I, H, 9)
    ref = oracle.moe_up_swiglu(a, row_idx, offsets, gate, up, g)
    big = torch.full((R + 3, I + 64), 5.0, dtype=torch.bfloat16 if out_dtype == nv.OUT_BF16 else torch.float32,
                     device="cuda")
    nv.moe_up_swiglu(nvfp4_device(a[0], a[1], a[2], T, H), torch.from_numpy(offsets).cuda(), w, I, R,
                     row_idx=torch.from_numpy(row_idx).cuda(), out_dtype=out_dtype, h=big[:R, :I])
    full = y_np(big)
    ok, worst = row_tolerance_ok(full[:R, :I], ref, out_bf16=out_dtype == nv.OUT_BF16)
    assert ok, worst
    assert (full[R:] == 5.0).all() and (full[:, I:] == 5.0).all()


def test_argument_errors():
    rng, E, row_idx, offsets, xb = small_problem(4)
    a = oracle.nvfp4_encode(xb)
    w, *_ = gate_up_weights(E, 128, 256, 11)
    ad = nvfp4_device(a[0], a[1], a[2], 64, 256)
    off = torch.from_numpy(offsets).cuda()
    with pytest.raises(nv.NVFP4Error) as e:      # I not a multiple of 128
        nv.moe_up_swiglu(ad, off, w, 192, int(offsets[-1]), row_idx=torch.from_numpy(row_idx).cuda())
    assert e.value.status == nv.ERR_UNSUPPORTED_SHAPE
