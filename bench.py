#!/usr/bin/env python
"""Benchmark of the NVFP4 W4A4 inference-GEMM hot path on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload decode|prefill|policy|moe] [--no-extras]

Prints ONE JSON line.  The headline workload is the decode-shape MLP up
projection (X [8, 8192] BF16 against NVFP4 weights [28672, 8192]); a step
quantises the BF16 activations (global amax + block encode) and runs the
block-scaled FP4 GEMM, i.e. one pass of the whole W4A4 path.  The metric is
the memory-bound one, GB/s of algorithmic bytes, with the GEMM kernel's
roofline fraction against the measured HBM bandwidth.  The prefill shape
(TFLOP/s against the FP4 tensor peak), the per-layer-policy stack and the
MoE grouped GEMM are measured in the same run under "workloads".

Inputs are seeded synthetic data (synth/); weights rotate over 4 copies
(528 MB > the 126 MB L2) so every step streams them from HBM.  Device-side
numbers (value, roofline) time a CUDA-graph replay of the K steps with CUDA
events on the launching stream; e2e times plain API calls with host copies.  Multi-GPU
runs (torchrun) are independent replicas: each rank runs the same workload
on its own GPU and `value` sums them (weak scaling).

--impl reference times the CPU oracle (oracle/, test infrastructure) on a
bounded sample of the same workload on this machine's host cores.
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

NOMINAL_FP4_OVER_BF16 = 13.5 / 2.25     # dense tensor-core ratio of B300
FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS = 6400.0, 1800.0

# DRAM bytes (read + write) per launch of the roofline kernel, from one ncu
# capture of the current kernel (profiles/ holds the capture and command);
# None until a capture of the current kernel exists.
TRAFFIC = {"decode": 135.40e6,    # w4a4_kernel<256,false,16>, 8x28672x8192: 132.32 MB read + 3.08 MB written
           "prefill": None}       # w4a4_kernel<256,false>: counters not yet retaken since the one-copy scale fetch


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1400.0, "fallback"


# ---------------------------------------------------------------- clocks sampler
class ClockSampler:
    FIELDS = ["clocks.sm", "clocks.max.sm", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap"]
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={','.join(self.FIELDS)}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        sm, mx, reasons = [], [], set()
        for t, line in self.lines:
            if not (t0 - 0.15 <= t <= t1 + 0.15):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, v in zip(self.NAMES, parts[2:]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- multi-rank (replicas)
def max_over_ranks(ms, dist, device):
    """The slowest rank's time: every rank contributes its own ms (MAX
    all-reduce); a single process returns its own."""
    if dist is None:
        return ms
    import torch
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(value_rank, ms_rank, ms_max, world):
    """Whole-job throughput of `world` replicas doing the same work: the
    units all ranks processed over the slowest rank's time."""
    return value_rank * ms_rank / ms_max * world


# ---------------------------------------------------------------- GPU workloads
class Ctx:
    def __init__(self, torch, nv, dev):
        self.torch, self.nv, self.dev = torch, nv, dev

    def bf16(self, bits):
        t = self.torch
        return t.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(self.dev).view(t.bfloat16)

    def quantized_weights(self, bits, copies=1):
        t, nv = self.torch, self.nv
        w = nv.quantize(self.bf16(bits))
        out = [w]
        for _ in range(copies - 1):
            out.append(nv.NVFP4Tensor(w.codes.clone(), w.scales.clone(), w.second.clone(), w.rows, w.K))
        t.cuda.synchronize()
        return out

    def time(self, fn, steps, warmup, graph=True):
        """Mean ms per call of fn(i) over `steps` calls after `warmup` calls,
        CUDA events on the stream the calls are launched on.  With graph=True
        the `steps` calls are captured once into a CUDA graph and one replay
        is timed (the launch path a serving loop uses: no host gaps between
        kernels); graph=False times the calls as issued from Python."""
        t = self.torch
        for i in range(warmup):
            fn(i)
        t.cuda.synchronize()
        s, e = t.cuda.Event(enable_timing=True), t.cuda.Event(enable_timing=True)
        if graph:
            g = t.cuda.CUDAGraph()
            with t.cuda.graph(g, capture_error_mode="relaxed"):
                for i in range(steps):
                    fn(warmup + i)
            g.replay()  # one untimed replay
            t.cuda.synchronize()
            s.record()
            g.replay()
            e.record()
            t.cuda.synchronize()
            return s.elapsed_time(e) / steps
        s.record()
        for i in range(steps):
            fn(warmup + i)
        e.record()
        t.cuda.synchronize()
        return s.elapsed_time(e) / steps


def nvfp4_bytes(rows, K):
    return rows * K // 2 + rows * K // 16


def _e4m3_table():
    """Value of every E4M3 byte (sign bit 7, exponent bits 6-3 with bias 7,
    mantissa bits 2-0; exponent 0 is subnormal m * 2^-9; S.1111.111 is NaN)."""
    v = np.empty(256)
    for b in range(256):
        e, m = (b >> 3) & 15, b & 7
        mag = m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
        v[b] = np.nan if (b & 0x7F) == 0x7F else (-mag if b & 0x80 else mag)
    return v


E4M3_VALUES = _e4m3_table()


def scale_stats(q):
    """Scale statistics of an NVFP4 tensor (tensor-scale mode) for the bench
    log: its FP32 tensor scale and the smallest and largest non-zero E4M3
    block scale (zero bytes, including the tiled layout's padding rows, are
    left out), plus the share of zero blocks among the tensor's real blocks."""
    sb = q.scales.cpu().numpy().ravel()
    nz = sb[sb != 0]
    vals = E4M3_VALUES[nz]
    blocks = q.rows * (q.K // 16)
    return {"tensor_scale": float(q.second.cpu().reshape(-1)[0]),
            "block_scale_min": float(vals.min()) if nz.size else 0.0,
            "block_scale_max": float(vals.max()) if nz.size else 0.0,
            "zero_block_frac": float(1.0 - nz.size / max(blocks, 1))}


def workload_decode(c, M, steps, warmup, rot=4, with_e2e=False, peaks_=None):
    t, nv = c.torch, c.nv
    N, K = 28672, 8192
    ws = synth.weights(2, 1, N, K)
    W = c.quantized_weights(ws, copies=rot)
    del ws
    xb = synth.activations(2, 0, M, K, 0.005, 100.0)
    x = c.bf16(xb)
    y = t.empty((M, N), dtype=t.bfloat16, device=c.dev)
    work = nv.Workspace(nv.workspace_size(nv.OP_GEMM, M, N, K))
    a_q = nv.quantize(x, ws=work)

    # algorithmic bytes: W (codes + scales), X read, quantised X write + read, Y write
    w_bytes = nvfp4_bytes(N, K)
    step_bytes = w_bytes + M * K * 2 + 2 * nvfp4_bytes(M, K) + M * N * 2
    gemm_bytes = w_bytes + nvfp4_bytes(M, K) + M * N * 2

    def step(i):
        nv.gemm(W[i % rot], x=x, y=y, ws=work)

    def gemm_only(i):
        nv.gemm(W[i % rot], a_q=a_q, y=y, ws=work)

    ms = c.time(step, steps, warmup)
    gms = c.time(gemm_only, steps, warmup)
    st = work.status()
    stream = None
    if with_e2e:
        # the copy engine's streaming rate on the same rotating weight codes,
        # with the GEMM's boxes and nothing else (nvfp4_diag_tma_stream): at
        # the decode kernel's grid (one CTA per 256-row tile) and at one CTA
        # per SM; the ceiling the decode GEMM's HBM fraction meets in practice
        status = t.zeros(1, dtype=t.int32, device=c.dev)
        codes = [w.codes.view(t.uint8).reshape(N, K // 2) for w in W]
        stream = {}
        for grid in (N // 256, nv.sm_count()):
            sms = c.time(lambda i, g=grid: nv.tma_stream(codes[i % rot], g, status), steps, warmup)
            stream[f"gbs_grid{grid}"] = codes[0].numel() / (sms * 1e-3) / 1e9
        stream["status"] = int(status.item())
        stream["bytes"] = codes[0].numel()
    stats = {"x": scale_stats(a_q), "w": scale_stats(W[0])}   # after the timed loops
    # the quantiser is one launch (one thread-block cluster) up to 32768
    # chunks of 8 values, two staged passes above that; then the GEMM
    launches = (1 if M * K // 8 <= 32768 else 2) + 1
    res = {"ms": ms, "gemm_ms": gms, "step_bytes": step_bytes, "gemm_bytes": gemm_bytes,
           "value": step_bytes / (ms * 1e-3) / 1e9, "launches_per_step": launches, "device_status": st,
           "scale_stats": stats}
    if stream is not None:
        res["stream"] = stream
    if with_e2e:
        hx = t.from_numpy(xb.view(np.int16)).pin_memory()
        hy = t.empty((M, N), dtype=t.int16).pin_memory()
        xd = t.empty((M, K), dtype=t.int16, device=c.dev)

        def e2e(i):
            xd.copy_(hx, non_blocking=True)
            nv.gemm(W[i % rot], x=xd.view(t.bfloat16), y=y, ws=work)
            hy.copy_(y.view(t.int16), non_blocking=True)

        # issued from Python call by call (best of 3 timed loops: host launch
        # jitter dominates single loops), and the same calls captured into a
        # CUDA graph, copies included, as a serving loop would replay them
        ems = min(c.time(e2e, steps, warmup, graph=False) for _ in range(3))
        gms_e2e = c.time(e2e, steps, warmup, graph=True)
        pms = e2e_pipelined(c, W, rot, hx, M, N, K, work, steps, warmup)
        res["e2e"] = {"value": step_bytes / (pms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": pms,
                      "how": "pipelined: step i's input copy, step i-1's GEMM and step i-2's result copy "
                             "in flight together (copy-in, compute and copy-out streams, double-buffered "
                             "device X and Y, ordered by events), captured into one CUDA graph",
                      "value_serial_python": step_bytes / (ems * 1e-3) / 1e9, "ms_per_step_serial_python": ems,
                      "value_serial_graph": step_bytes / (gms_e2e * 1e-3) / 1e9,
                      "ms_per_step_serial_graph": gms_e2e,
                      "h2d_bytes_per_step": M * K * 2, "d2h_bytes_per_step": M * N * 2}
    del W
    return res


def e2e_pipelined(c, W, rot, hx, M, N, K, work, steps, warmup):
    """End to end with the copies overlapped across steps, as a serving loop
    runs them: every step still copies its input from pinned host memory and
    its result back, but step i's input copy, the GEMM of step i - 1 and the
    result copy of step i - 2 run together on three streams.  Device X and Y
    are double-buffered; events order each buffer's reuse (the copy into
    X[b] waits for the GEMM that read it two steps before, the GEMM into
    Y[b] for the copy-out that read it).  The whole loop is captured into
    one CUDA graph; ms per step of one timed replay."""
    t, nv = c.torch, c.nv
    xd = [t.empty((M, K), dtype=t.int16, device=c.dev) for _ in range(2)]
    yd = [t.empty((M, N), dtype=t.bfloat16, device=c.dev) for _ in range(2)]
    hy = [t.empty((M, N), dtype=t.int16).pin_memory() for _ in range(2)]
    s_in, s_out = t.cuda.Stream(), t.cuda.Stream()

    def body(n, base):
        main = t.cuda.current_stream()
        fork = t.cuda.Event()
        fork.record(main)
        s_in.wait_event(fork)
        s_out.wait_event(fork)
        done_cmp, done_out = [None, None], [None, None]
        last_in = last_out = None
        for i in range(n):
            b = i % 2
            with t.cuda.stream(s_in):
                if done_cmp[b] is not None:
                    s_in.wait_event(done_cmp[b])
                xd[b].copy_(hx, non_blocking=True)
                last_in = t.cuda.Event()
                last_in.record(s_in)
            main.wait_event(last_in)
            if done_out[b] is not None:
                main.wait_event(done_out[b])
            nv.gemm(W[(base + i) % rot], x=xd[b].view(t.bfloat16), y=yd[b], ws=work)
            done_cmp[b] = t.cuda.Event()
            done_cmp[b].record(main)
            with t.cuda.stream(s_out):
                s_out.wait_event(done_cmp[b])
                hy[b].copy_(yd[b].view(t.int16), non_blocking=True)
                done_out[b] = t.cuda.Event()
                done_out[b].record(s_out)
                last_out = done_out[b]
        main.wait_event(last_in)   # join both side streams
        main.wait_event(last_out)

    body(warmup, 0)
    t.cuda.synchronize()
    g = t.cuda.CUDAGraph()
    with t.cuda.graph(g, capture_error_mode="relaxed"):
        body(steps, warmup)
    g.replay()  # one untimed replay
    t.cuda.synchronize()
    s, e = t.cuda.Event(enable_timing=True), t.cuda.Event(enable_timing=True)
    s.record()
    g.replay()
    e.record()
    t.cuda.synchronize()
    return s.elapsed_time(e) / steps


def workload_prefill(c, N, steps, warmup, rot=2, x_rot=3):
    """Prefill GEMM (X [4096, 8192] x W [N, 8192]^T) with its activation
    quantiser.  Weights rotate over `rot` copies and activations over
    `x_rot` copies (3 x 67 MB), so no step finds its inputs in the 126 MB L2
    from an earlier step."""
    t, nv = c.torch, c.nv
    M, K = 4096, 8192
    W = c.quantized_weights(synth.weights(3, 1, N, K), copies=rot)
    x0 = synth.activations(3, 0, M, K, 0.005, 100.0)
    xs = [c.bf16(x0) for _ in range(x_rot)]
    y = t.empty((M, N), dtype=t.bfloat16, device=c.dev)
    work = nv.Workspace(nv.workspace_size(nv.OP_GEMM, M, N, K))
    a_q = nv.quantize(xs[0], ws=work)
    flops = 2.0 * M * N * K

    def step(i):
        nv.gemm(W[i % rot], x=xs[i % x_rot], y=y, ws=work)

    def gemm_only(i):
        nv.gemm(W[i % rot], a_q=a_q, y=y, ws=work)

    ms = c.time(step, steps, warmup)
    gms = c.time(gemm_only, steps, warmup)
    qbytes = M * K * 2 + nvfp4_bytes(M, K)

    def quant_only(i):
        nv.quantize(xs[i % x_rot], out=a_q, ws=work)

    qms = c.time(quant_only, steps, warmup)
    st = work.status()
    del W, xs
    return {"ms": ms, "gemm_ms": gms, "flops": flops, "value": flops / (ms * 1e-3) / 1e12, "launches_per_step": 3,
            "gemm_tflops": flops / (gms * 1e-3) / 1e12, "quant_ms": qms, "quant_bytes": qbytes,
            "quant_gbs": qbytes / (qms * 1e-3) / 1e9, "device_status": st}


def workload_prefill_macro(c, N, steps, warmup, rot=2):
    """The FP16 macro-scale GEMM (one FP16 scale per 256 elements of each row
    replacing the tensor scale) at the prefill shape X [4096, 8192] x W
    [N, 8192]^T on pre-quantised macro-mode activations; weights rotate over
    `rot` copies."""
    t, nv = c.torch, c.nv
    M, K = 4096, 8192
    wb = synth.weights(3, 1, N, K)
    W = []
    for _ in range(rot):
        W.append(nv.quantize(c.bf16(wb), mode=nv.SCALE_MACRO_FP16))
    del wb
    a_q = nv.quantize(c.bf16(synth.activations(3, 0, M, K, 0.005, 100.0)), mode=nv.SCALE_MACRO_FP16)
    y = t.empty((M, N), dtype=t.bfloat16, device=c.dev)
    work = nv.Workspace(nv.workspace_size(nv.OP_GEMM, M, N, K))

    def gemm_only(i):
        nv.gemm(W[i % rot], a_q=a_q, y=y, ws=work)

    gms = c.time(gemm_only, steps, warmup)
    st = work.status()
    del W
    flops = 2.0 * M * N * K
    return {"gemm_ms": gms, "gemm_tflops": flops / (gms * 1e-3) / 1e12, "device_status": st}


def workload_policy(c, steps, warmup, policy):
    t, nv = c.torch, c.nv
    cfg = synth.CONFIGS[4]
    M, N, K, L = cfg["M"], cfg["N"], cfg["K"], cfg["layers"]
    Ws = [c.quantized_weights(synth.weights(4, 100 + i, N, K))[0] for i in range(L)]
    flags = synth.sensitive_flags(L, cfg["n_sensitive"])
    x = c.bf16(synth.activations(4, 0, M, K, cfg["outlier_frac"], cfg["outlier_factor"]))
    ys = [t.empty((M, N), dtype=t.bfloat16, device=c.dev) for _ in range(2)]
    work = nv.Workspace(nv.workspace_size(nv.OP_GEMM, M, N, K))

    def step(i):
        cur = x
        for li in range(L):
            out = ys[li % 2]
            nv.gemm(Ws[li], x=cur, y=out, policy=policy, sensitive=int(flags[li]), ws=work)
            cur = out

    ms = c.time(step, steps, warmup)
    flops = 2.0 * M * N * K * L
    routes = [nv.policy_route(policy, int(f)) for f in flags]
    layer_stats = [scale_stats(w) for w in Ws]   # after the timed loop
    return {"ms": ms, "flops": flops, "value": flops / (ms * 1e-3) / 1e12, "routes": routes,
            "w_scale_stats": layer_stats,
            "launches_per_step": sum(3 if r == 4 else 2 for r in routes), "device_status": work.status()}


def workload_fused_stack(c, steps, warmup):
    """The all-W4A4 policy stack with every layer but the last writing the
    next layer's NVFP4 activations from its epilogue (nvfp4_gemm_nvfp4_out):
    layer 0 quantises the BF16 input on the fly, the last layer writes BF16.
    Static per-layer output scales s_l = amax_l / 2688, calibrated once
    before timing, layer by layer, from the amax the fused epilogue reports."""
    t, nv = c.torch, c.nv
    cfg = synth.CONFIGS[4]
    M, N, K, L = cfg["M"], cfg["N"], cfg["K"], cfg["layers"]
    Ws = [c.quantized_weights(synth.weights(4, 100 + i, N, K))[0] for i in range(L)]
    x = c.bf16(synth.activations(4, 0, M, K, cfg["outlier_frac"], cfg["outlier_factor"]))
    work = nv.Workspace(nv.workspace_size(nv.OP_GEMM, M, N, K))
    scales = [t.ones(1, dtype=t.float32, device=c.dev) for _ in range(L - 1)]
    acts = [nv.empty_nvfp4(M, N, device=c.dev) for _ in range(2)]
    y = t.empty((M, N), dtype=t.bfloat16, device=c.dev)
    amax = t.zeros(1, dtype=t.float32, device=c.dev)

    def layer(li, y_amax=None):
        a_in = None if li == 0 else acts[(li - 1) % 2]
        if li == L - 1:
            nv.gemm(Ws[li], a_q=a_in, y=y, policy=nv.POLICY_Q4, ws=work)
        else:
            nv.gemm_nvfp4_out(Ws[li], scales[li], x=x if li == 0 else None, a_q=a_in, y_amax=y_amax,
                              out=acts[li % 2], ws=work)

    for li in range(L - 1):             # calibration
        amax.zero_()
        layer(li, amax)
        scales[li].copy_(amax / 2688.0)
        layer(li)
    t.cuda.synchronize()

    def step(i):
        for li in range(L):
            layer(li)

    ms = c.time(step, steps, warmup)
    flops = 2.0 * M * N * K * L
    return {"ms": ms, "flops": flops, "value": flops / (ms * 1e-3) / 1e12, "launches_per_step": L + 2,
            "device_status": work.status()}


def workload_moe(c, steps, warmup):
    t, nv = c.torch, c.nv
    cfg = synth.CONFIGS[5]
    T, H, E, I = cfg["T"], cfg["H"], cfg["E"], cfg["inter"]
    row_idx, offsets, counts, _ = synth.moe_routing()
    R = int(offsets[-1])

    def stacked(N, K, tid):
        parts = [c.quantized_weights(synth.weights(5, tid * 1000 + e, N, K))[0] for e in range(E)]
        return nv.NVFP4Tensor(t.cat([p.codes for p in parts]), t.cat([p.scales for p in parts]),
                              t.cat([p.second for p in parts]), E * N, K)

    w_up, w_dn = stacked(I, H, 1), stacked(H, I, 2)
    x = c.bf16(synth.activations(5, 0, T, H, cfg["outlier_frac"], cfg["outlier_factor"]))
    xd = c.bf16(synth.activations(5, 2, R, I, cfg["outlier_frac"], cfg["outlier_factor"]))
    off = t.from_numpy(offsets).to(c.dev)
    ridx = t.from_numpy(row_idx).to(c.dev)
    y_up = t.empty((R, I), dtype=t.bfloat16, device=c.dev)
    y_dn = t.empty((R, H), dtype=t.bfloat16, device=c.dev)
    work = nv.Workspace(nv.workspace_size(nv.OP_QUANTIZE, R, 0, max(H, I)))
    a_up = nv.quantize(x, ws=work)
    a_dn = nv.quantize(xd, ws=work)

    def step(i):
        nv.quantize(x, out=a_up, ws=work)
        nv.grouped_gemm(a_up, off, w_up, I, R, row_idx=ridx, y=y_up, ws=work)
        nv.quantize(xd, out=a_dn, ws=work)
        nv.grouped_gemm(a_dn, off, w_dn, H, R, y=y_dn, ws=work)

    ms = c.time(step, steps, warmup)
    wbytes = 2 * E * nvfp4_bytes(I, H)
    step_bytes = (wbytes + T * H * 2 + 2 * nvfp4_bytes(T, H) + R * I * 2          # up
                  + R * I * 2 + 2 * nvfp4_bytes(R, I) + R * H * 2)                 # down
    flops = 2.0 * R * I * H * 2
    return {"ms": ms, "bytes": step_bytes, "value": step_bytes / (ms * 1e-3) / 1e9, "launches_per_step": 6,
            "tflops": flops / (ms * 1e-3) / 1e12, "counts_min": int(counts.min()),
            "counts_max": int(counts.max()), "device_status": work.status()}


def workload_moe_ffn(c, steps, warmup):
    """The mixture-of-experts feed-forward block with every fusion: the BF16
    tokens quantised once, the grouped up projection gathering token rows and
    applying SwiGLU in its epilogue, written as NVFP4 under a calibrated
    static scale, then the grouped down projection adding each routed row,
    times its routing weight, into its token's FP32 output row."""
    t, nv = c.torch, c.nv
    cfg = synth.CONFIGS[5]
    T, H, E, I = cfg["T"], cfg["H"], cfg["E"], cfg["inter"]
    row_idx, offsets, counts, logits = synth.moe_routing()
    R = int(offsets[-1])
    gate_w = synth.moe_gate_weights(logits, row_idx, offsets, cfg["topk"])

    def stacked(N, K, tid):
        parts = [c.quantized_weights(synth.weights(5, tid * 1000 + e, N, K))[0] for e in range(E)]
        return nv.NVFP4Tensor(t.cat([p.codes for p in parts]), t.cat([p.scales for p in parts]),
                              t.cat([p.second for p in parts]), E * N, K)

    # random-init weights: the gate/up interleave is a row permutation of
    # i.i.d. rows, so drawing the stacked [2I, H] block directly is the same
    w_gu, w_dn = stacked(2 * I, H, 6), stacked(H, I, 7)
    x = c.bf16(synth.activations(5, 0, T, H, cfg["outlier_frac"], cfg["outlier_factor"]))
    off = t.from_numpy(offsets).to(c.dev)
    ridx = t.from_numpy(row_idx).to(c.dev)
    gw = t.from_numpy(gate_w).to(c.dev)
    y = t.zeros((T, H), dtype=t.float32, device=c.dev)
    work = nv.Workspace(max(nv.workspace_size(nv.OP_QUANTIZE, T, 0, H),
                            nv.workspace_size(nv.OP_GROUPED_GEMM, R, 2 * I, H, E)))
    a = nv.quantize(x, ws=work)
    s_h = t.ones(1, dtype=t.float32, device=c.dev)
    amax = t.zeros(1, dtype=t.float32, device=c.dev)
    h_q = nv.empty_nvfp4(R, I, device=c.dev)
    nv.moe_up_swiglu(a, off, w_gu, I, R, row_idx=ridx, s_h=s_h, h_amax=amax, h_q=h_q, ws=work)
    s_h.copy_(amax / 2688.0)                 # calibration
    t.cuda.synchronize()

    def step(i):
        nv.quantize(x, out=a, ws=work)
        nv.moe_up_swiglu(a, off, w_gu, I, R, row_idx=ridx, s_h=s_h, h_q=h_q, ws=work)
        y.zero_()
        nv.moe_down_combine(h_q, off, w_dn, H, ridx, gw, y, ws=work)

    ms = c.time(step, steps, warmup)
    wbytes = E * (nvfp4_bytes(2 * I, H) + nvfp4_bytes(H, I))
    step_bytes = (wbytes + T * H * 2 + 2 * nvfp4_bytes(T, H) + 2 * nvfp4_bytes(R, I)  # x, a, h
                  + 2 * T * H * 4)                                                    # y zero + combine
    flops = 6.0 * R * H * I
    return {"ms": ms, "bytes": step_bytes, "value": step_bytes / (ms * 1e-3) / 1e9, "launches_per_step": 4,
            "tflops": flops / (ms * 1e-3) / 1e12, "device_status": work.status()}


def workload_kv_decode(c, steps, warmup, B=16, H=64, H_kv=8, ctx=4096, fmt=0, copies=3):
    """Decode attention over an NVFP4 paged KV cache (Llama-3-70B-class
    grouping: 64 query heads over 8 KV heads, head_dim 128), 16 sequences of
    4096 cached tokens each, plus the append of each sequence's new token:
    the step reads the whole cache once.  Cache bytes are synthetic (random
    codes, scale bytes in a normal range); pages shuffled across the pool.
    Steps rotate over `copies` caches (3 x 75 MB NVFP4, 3 x 134 MB FP8), so
    no step finds its cache in the 126 MB L2 from an earlier step."""
    t, nv = c.torch, c.nv
    P, D = nv.KV_PAGE, nv.KV_HEAD_DIM
    pages_per = ctx // P + 1
    n_pages = B * pages_per
    g = t.Generator(device=c.dev)
    g.manual_seed(0)
    ks = t.tensor([8.0 / 2688], device=c.dev)
    vs = t.tensor([4.0 / 2688], device=c.dev)
    cache = nv.KvCache.empty(n_pages, H_kv, ks, vs, device=c.dev, fmt=fmt)
    pg = cache.pages
    if fmt == nv.KV_FP8:   # finite E4M3 codes with random signs
        pg.copy_(t.randint(0, 0x70, pg.shape, dtype=t.uint8, device=c.dev, generator=g)
                 | (t.randint(0, 2, pg.shape, dtype=t.uint8, device=c.dev, generator=g) << 7))
    else:                  # random codes, scale bytes in a normal range
        pg.copy_(t.randint(0, 256, pg.shape, dtype=t.uint8, device=c.dev, generator=g))
        for lo, hi in ((2048, 2304), (4352, 4608), (6656, 6912), (8960, 9216)):
            pg[..., lo:hi] = t.randint(0x28, 0x48, pg[..., lo:hi].shape, dtype=t.uint8, device=c.dev, generator=g)
    caches = [cache] + [nv.KvCache(pg.clone(), ks, vs, fmt) for _ in range(copies - 1)]
    perm = t.randperm(n_pages, device=c.dev, generator=g).to(t.int32)
    table = perm.view(B, pages_per).contiguous()
    ctx_lens = t.full((B,), ctx, dtype=t.int32, device=c.dev)
    pos = t.full((B,), ctx, dtype=t.int32, device=c.dev)
    q = t.randn((B, H, D), device=c.dev, generator=g).to(t.bfloat16)
    k_new = t.randn((B, H_kv, D), device=c.dev, generator=g).to(t.bfloat16)
    v_new = t.randn((B, H_kv, D), device=c.dev, generator=g).to(t.bfloat16)
    out = t.empty((B, H, D), dtype=t.bfloat16, device=c.dev)
    work = nv.Workspace(nv.workspace_size(nv.OP_KV_DECODE, B, H, ctx + 1, H_kv))
    sm = 1.0 / math.sqrt(D)
    ctx1 = t.full((B,), ctx + 1, dtype=t.int32, device=c.dev)

    def step(i):
        kv = caches[i % copies]
        nv.kv_append(kv, k_new, v_new, pos, table)
        nv.kv_decode_attention(kv, q, ctx1, table, ctx + 1, sm, out=out, ws=work)

    def attn_only(i):
        nv.kv_decode_attention(caches[i % copies], q, ctx_lens, table, ctx, sm, out=out, ws=work)

    ms = c.time(step, steps, warmup)
    ams = c.time(attn_only, steps, warmup)
    cache_bytes = B * H_kv * ctx * 2 * (D if fmt == nv.KV_FP8 else D // 2 + D // 16)
    return {"ms": ms, "attn_ms": ams, "bytes": cache_bytes, "value": cache_bytes / (ms * 1e-3) / 1e9,
            "attn_gbs": cache_bytes / (ams * 1e-3) / 1e9, "device_status": work.status()}


# ---------------------------------------------------------------- CPU oracle (baseline / reference arm)
def oracle_decode_setup(M=8, n_rows=2048):
    """Inputs of the oracle's decode sample, made once (untimed): the first
    n_rows of the 28672 weight rows, encoded by the oracle itself (offline
    weights), and the step's activations X [M, 8192]."""
    import oracle
    K = 8192
    wq = oracle.nvfp4_encode(synth.weights(2, 1, 28672, K)[:n_rows])
    xb = synth.activations(2, 0, M, K, 0.005, 100.0)
    nbytes = nvfp4_bytes(n_rows, K) + M * K * 2 + 2 * nvfp4_bytes(M, K) + M * n_rows * 2
    return oracle, wq, xb, nbytes


def oracle_decode_step(setup, reps=1):
    """The oracle's decode step (encode X, dequantise-and-contract in FP64)
    on the sample.  Returns (GB/s, seconds per step, bytes per step)."""
    oracle, wq, xb, nbytes = setup
    t0 = time.perf_counter()
    for _ in range(reps):
        aq = oracle.nvfp4_encode(xb)
        oracle.gemm_w4a4(aq, wq)
    dt = (time.perf_counter() - t0) / reps
    return nbytes / dt / 1e9, dt, nbytes


def _median_time(fn, reps):
    ts = []
    for _ in range(reps):
        t0 = time.perf_counter()
        fn()
        ts.append(time.perf_counter() - t0)
    return float(np.median(ts))


def cpu_baseline_plan():
    """The oracle timed on this host, per configuration: the encoder on each
    configuration's full tensors (all cores, and one thread on the
    activations), and the FP64 dequantise-and-contract step in full for
    configurations 1 and 2 (M = 1, 8, 16), on 256 seeded rows plus the first
    and last for configuration 3 (N = 8192), on 256 seeded rows of one layer
    for configuration 4 and on the first 16 experts of configuration 5's up
    projection (the last two labelled as samples, with the full-problem time
    extrapolated).  Medians of repeats; about 20-30 s in all.  Returns
    (headline dict: the configuration-2 M = 8 decode step, per-config dict)."""
    import oracle
    cores = os.cpu_count() or 1
    oracle.set_threads(cores)
    out = {}

    def enc_entry(bits, reps=3, single=False):
        n = bits.size
        nbytes = n * 2 + n // 2 + n // 16
        t = _median_time(lambda: oracle.nvfp4_encode(bits), reps)
        e = {"elements": int(n), "s": t, "melem_per_s": n / t / 1e6, "gbs": nbytes / t / 1e9, "threads": cores}
        if single:
            oracle.set_threads(1)
            t1 = _median_time(lambda: oracle.nvfp4_encode(bits), 1)
            oracle.set_threads(cores)
            e.update({"s_1thread": t1, "melem_per_s_1thread": n / t1 / 1e6})
        return e

    def gemm_entry(aq, wq, M, N, K, rows=None, reps=1, scale_to=None):
        nr = M if rows is None else len(rows)
        t = _median_time(lambda: oracle.gemm_w4a4(aq, wq, rows=rows), reps)
        flop = 2.0 * nr * N * K
        e = {"rows": int(nr), "s": t, "gflops_f64": flop / t / 1e9}
        if scale_to is not None:
            e["full_problem_s_extrapolated"] = t * scale_to
        return e

    # configuration 1
    x1, w1 = synth.activations(1, 0, 128, 512, 0.01, 50.0), synth.weights(1, 1, 256, 512)
    a1, q1 = oracle.nvfp4_encode(x1), oracle.nvfp4_encode(w1)
    out["c1"] = {"encode_x": enc_entry(x1, single=True), "encode_w": enc_entry(w1),
                 "gemm": gemm_entry(a1, q1, 128, 256, 512, reps=3)}
    # configuration 2 (decode): full W, M = 1, 8, 16
    K = 8192
    w2 = synth.weights(2, 1, 28672, K)
    c2 = {"encode_w": enc_entry(w2, reps=1)}
    q2 = oracle.nvfp4_encode(w2)
    del w2
    head = None
    for M in (1, 8, 16):
        xb = synth.activations(2, 0, M, K, 0.005, 100.0)
        c2[f"encode_x_m{M}"] = enc_entry(xb, single=True)
        aq = oracle.nvfp4_encode(xb)
        g = gemm_entry(aq, q2, M, 28672, K, reps=3 if M == 8 else 1)
        nbytes = nvfp4_bytes(28672, K) + M * K * 2 + 2 * nvfp4_bytes(M, K) + M * 28672 * 2
        g["step_gbs"] = nbytes / (g["s"] + c2[f"encode_x_m{M}"]["s"]) / 1e9
        c2[f"gemm_m{M}"] = g
        if M == 8:
            head = {"value": g["step_gbs"], "unit": "GB/s", "cores": cores, "kind": "oracle",
                    "sample": "configuration 2 decode step in full (encode X [8,8192], FP64 contraction with "
                              "all 28672 weight rows), median of 3"}
    out["c2"] = c2
    del q2
    # configuration 3 (prefill): encoder on X, contraction on 258 rows against N = 8192
    x3 = synth.activations(3, 0, 4096, K, 0.005, 100.0)
    w3 = synth.weights(3, 1, 8192, K)
    rows = np.concatenate([[0, 4095], np.random.default_rng(8192).choice(np.arange(1, 4095), 256, replace=False)])
    a3, q3 = oracle.nvfp4_encode(x3), oracle.nvfp4_encode(w3)
    out["c3"] = {"encode_x": enc_entry(x3, reps=1, single=True), "encode_w": enc_entry(w3, reps=1),
                 "gemm_n8192_sampled": gemm_entry(a3, q3, 4096, 8192, K, rows=rows, scale_to=4096 / len(rows))}
    del x3, w3, a3, q3
    # configuration 4: one layer, 256 seeded rows
    x4, w4 = synth.activations(4, 0, 2048, 4096, 0.01, 50.0), synth.weights(4, 1, 4096, 4096)
    a4, q4 = oracle.nvfp4_encode(x4), oracle.nvfp4_encode(w4)
    r4 = np.random.default_rng(4).choice(2048, 256, replace=False)
    out["c4"] = {"encode_x": enc_entry(x4, single=True), "encode_w": enc_entry(w4),
                 "gemm_layer_sampled": gemm_entry(a4, q4, 2048, 4096, 4096, rows=r4, scale_to=2048 / 256)}
    del x4, w4, a4, q4
    # configuration 5: up projection, experts 0..15 of the default routing
    idx, offs, _, _ = synth.moe_routing()
    c5 = synth.CONFIGS[5]
    xm = synth.activations(5, 0, 2048, 2048, c5["outlier_frac"], c5["outlier_factor"])
    wup = synth.weights(5, 1, 16 * 768, 2048)
    out["c5_encode_w_up_16_experts"] = enc_entry(wup, reps=1)
    am = oracle.nvfp4_encode(xm)
    qc, qs, qg = oracle.nvfp4_encode(wup)
    E16 = 16
    sub_off = offs[:E16 + 1] - offs[0]
    sub_idx = idx[offs[0]:offs[E16]]
    t = _median_time(lambda: oracle.gemm_grouped_w4a4(am, sub_idx, sub_off, qc.reshape(E16, 768, 1024),
                                                      qs.reshape(E16, 768, 128), np.full(E16, qg, np.float32)), 1)
    routed = int(sub_off[-1])
    out["c5_up_16_experts"] = {"routed_rows": routed, "s": t, "gflops_f64": 2.0 * routed * 768 * 2048 / t / 1e9,
                               "full_problem_s_extrapolated": t * float(offs[-1] - offs[0]) / max(routed, 1)}
    return head, out


def cpu_cores():
    try:
        import oracle
        return oracle.threads()
    except Exception:
        return os.cpu_count() or 1


# ---------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["decode", "prefill", "policy", "moe", "macro"], default="decode")
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the CPU oracle leg (profiling runs)")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    hbm, bf16, bf16_sus, peak_src = peaks()
    fp4_nominal = bf16 * NOMINAL_FP4_OVER_BF16
    metric = "NVFP4 W4A4 GEMM TFLOPS & % dense FP4 peak (prefill); GB/s & % HBM (decode)"

    if args.impl == "reference":
        if rank != 0:
            return 0
        n_rows = 2048
        setup = oracle_decode_setup(n_rows=n_rows)   # once, untimed
        for _ in range(args.warmup):
            oracle_decode_step(setup)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            oracle_decode_step(setup)
        total = time.perf_counter() - t0
        v = setup[3] * max(args.steps, 1) / max(total, 1e-9) / 1e9
        cores = cpu_cores()
        line = {"impl": "reference", "metric": metric, "value": v, "unit": "GB/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / max(args.steps, 1),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic",
                "config": {"workload": "decode_mlp_up M=8 N=28672 K=8192 (sample: first 2048 weight rows)"},
                "cpu_baseline": {"value": v, "unit": "GB/s", "cores": cores, "kind": "oracle",
                                 "sample": f"decode step on {n_rows} of 28672 weight rows per step"},
                "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return 0

    # the oracle's baseline runs first, before any GPU work, on rank 0 alone
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu, per_config = cpu_baseline_plan()
        cpu["per_config"] = per_config

    import torch
    import nvfp4_block_scaled_30_b300 as nv
    nv.lib()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (there is no CPU fallback)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    c = Ctx(torch, nv, dev)
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.4)
    # dense FP4 tensor-core rate of this GPU (the prefill roofline's peak):
    # the MMA issue-rate kernel, one CTA per SM, operands resident on chip
    fp4_iters = 400000      # ~0.1 s per launch, long enough for the clock samples
    nv.fp4_mma_rate(200)
    t_fp4 = time.time()
    runs = [nv.fp4_mma_rate(fp4_iters) for _ in range(3)]
    fp4_clocks = sampler.summary(t_fp4, time.time())
    fp4_flop_clk_sm, fp4_ms, n_sm = max(runs, key=lambda r: r[0] / r[1] if r[1] > 0 else 0)
    fp4_ms = min(r[1] for r in runs)
    fp4_peak = fp4_iters * 4 * nv.FP4_MMA_FLOP * n_sm / (fp4_ms * 1e-3) / 1e12
    fp4_info = {"tflops_measured": fp4_peak, "flop_per_clock_per_sm": fp4_flop_clk_sm, "sms": n_sm,
                "sm_mhz_median": fp4_clocks.get("sm_mhz"),
                "tflops_at_max_clock": fp4_flop_clk_sm * n_sm * 2032e6 / 1e12,
                "tflops_nominal_ratio_of_bf16": fp4_nominal,
                "how": f"{fp4_iters} x 4 tcgen05.mma kind::mxf4nvf4 M=128 N=256 K=64 per SM, CUDA events"}

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    barrier()
    t_start = time.time()
    if args.workload == "decode":
        r = workload_decode(c, 8, args.steps, args.warmup, with_e2e=True)
        unit, value_rank = "GB/s", r["value"]
    elif args.workload == "prefill":
        r = workload_prefill(c, 28672, args.steps, args.warmup)
        unit, value_rank = "TFLOP/s", r["value"]
    elif args.workload == "policy":
        r = workload_policy(c, args.steps, args.warmup, nv.POLICY_AUTO)
        unit, value_rank = "TFLOP/s", r["value"]
    elif args.workload == "macro":
        r = workload_prefill_macro(c, 8192, args.steps, args.warmup)
        r.update({"ms": r["gemm_ms"], "value": r["gemm_tflops"], "launches_per_step": 1})
        unit, value_rank = "TFLOP/s", r["value"]
    else:
        r = workload_moe(c, args.steps, args.warmup)
        unit, value_rank = "GB/s", r["value"]
    barrier()
    t_end = time.time()
    ms = max_over_ranks(r["ms"], dist, dev)
    value = job_value(value_rank, r["ms"], ms, world)

    clocks = sampler.summary(t_start, t_end)

    extras = {}
    if not args.no_extras and rank == 0:
        es = max(20, min(args.steps, 200))
        for M in (1, 16):
            d = workload_decode(c, M, es, args.warmup)
            extras[f"decode_m{M}"] = {"value": d["value"], "unit": "GB/s", "ms": d["ms"],
                                      "gemm_gbs": d["gemm_bytes"] / (d["gemm_ms"] * 1e-3) / 1e9,
                                      "gemm_frac_hbm": d["gemm_bytes"] / (d["gemm_ms"] * 1e-3) / 1e9 / hbm}
        if args.workload != "prefill":
            for N in (8192, 28672):
                p = workload_prefill(c, N, min(es, 50), args.warmup)
                extras[f"prefill_n{N}"] = {"value": p["value"], "unit": "TFLOP/s", "ms": p["ms"],
                                           "gemm_tflops": p["gemm_tflops"],
                                           "gemm_frac_fp4": p["gemm_tflops"] / fp4_peak,
                                           "gemm_frac_fp4_nominal": p["gemm_tflops"] / fp4_nominal,
                                           "quant_gbs": p["quant_gbs"], "quant_frac_hbm": p["quant_gbs"] / hbm}
        pm = workload_prefill_macro(c, 8192, min(es, 50), args.warmup)
        extras["prefill_macro_n8192"] = {"gemm_tflops": pm["gemm_tflops"], "gemm_ms": pm["gemm_ms"],
                                         "gemm_frac_fp4": pm["gemm_tflops"] / fp4_peak,
                                         "device_status": pm["device_status"],
                                         "config": "FP16 macro-scale GEMM X[4096,8192] x W[8192,8192]^T"}
        for pol, name in ((nv.POLICY_AUTO, "auto"), (nv.POLICY_Q4, "q4"), (nv.POLICY_Q8, "q8")):
            q = workload_policy(c, min(es, 20), 2, pol)
            extras[f"policy_stack_{name}"] = {"value": q["value"], "unit": "TFLOP/s", "ms": q["ms"],
                                              "routes": q["routes"]}
            if name == "auto":   # the stack's weights are the same for every policy
                extras["policy_stack_auto"]["layer_w_scale_stats"] = q["w_scale_stats"]
        fq = workload_fused_stack(c, min(es, 20), 2)
        extras["policy_stack_q4_fused"] = {"value": fq["value"], "unit": "TFLOP/s", "ms": fq["ms"]}
        kd = workload_kv_decode(c, min(es, 50), 3)
        extras["kv_decode_attention"] = {"value": kd["value"], "unit": "GB/s", "ms": kd["ms"],
                                         "frac_hbm": kd["value"] / hbm, "attn_gbs": kd["attn_gbs"],
                                         "attn_frac_hbm": kd["attn_gbs"] / hbm,
                                         "config": "16 seqs x 4096 tokens, 64 q heads / 8 kv heads, d 128"}
        kd8 = workload_kv_decode(c, min(es, 50), 3, fmt=nv.KV_FP8)
        extras["kv_decode_attention_fp8"] = {"value": kd8["value"], "unit": "GB/s", "ms": kd8["ms"],
                                             "frac_hbm": kd8["value"] / hbm, "attn_gbs": kd8["attn_gbs"],
                                             "attn_frac_hbm": kd8["attn_gbs"] / hbm,
                                             "config": "FP8 cache, 16 seqs x 4096 tokens, 64/8 heads, d 128"}
        mf = workload_moe_ffn(c, min(es, 50), 2)
        extras["moe_ffn_fused"] = {"value": mf["value"], "unit": "GB/s", "ms": mf["ms"], "tflops": mf["tflops"],
                                   "frac_hbm": mf["value"] / hbm}
        mo = workload_moe(c, min(es, 50), 2)
        extras["moe_grouped"] = {"value": mo["value"], "unit": "GB/s", "ms": mo["ms"], "tflops": mo["tflops"],
                                 "frac_hbm": mo["value"] / hbm, "counts": [mo["counts_min"], mo["counts_max"]]}

    if args.workload == "decode":
        ach = r["gemm_bytes"] / (r["gemm_ms"] * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
                "traffic": TRAFFIC.get("decode"), "kernel": "w4a4_kernel<256,false> (112 CTAs, one 256-row weight tile each)",
                "peak_source": f"{peak_src} hbm_gbs"}
        if r.get("stream"):
            best = max(v for k, v in r["stream"].items() if k.startswith("gbs_"))
            roof["stream_ceiling"] = dict(r["stream"], frac_of_hbm=best / hbm, gemm_frac_of_stream=ach / best,
                                          how="nvfp4_diag_tma_stream: the weight codes by the GEMM's TMA boxes, "
                                              "6-stage ring, no compute")
        cfg = {"workload": "decode_mlp_up: X[8,8192] bf16 -> NVFP4, W NVFP4[28672,8192], Y bf16",
               "global_batch": 8, "l2": "4 rotating weight copies (528 MB > 126 MB L2)"}
    elif args.workload == "prefill":
        ach = r["gemm_tflops"]
        roof = {"bound": "tensor", "achieved": ach, "peak": fp4_peak, "unit": "TFLOP/s", "frac": ach / fp4_peak,
                "traffic": TRAFFIC.get("prefill"), "kernel": "w4a4_kernel<256,false>",
                "peak_source": "measured in this run: tcgen05 mxf4nvf4 issue-rate kernel (fp4_peak)",
                "frac_of_nominal": ach / fp4_nominal}
        cfg = {"workload": "prefill_proj: X[4096,8192], W NVFP4[28672,8192]", "global_batch": 4096,
               "l2": "inputs larger than L2 (3 rotating X copies of 67 MB + 2 rotating W copies of 132 MB)"}
    elif args.workload == "policy":
        roof = None
        cfg = {"workload": "policy_stack AUTO: 8 x [2048,4096]x[4096,4096]^T, 2 W4A8 layers", "global_batch": 2048}
    elif args.workload == "macro":
        ach = r["gemm_tflops"]
        roof = {"bound": "tensor", "achieved": ach, "peak": fp4_peak, "unit": "TFLOP/s", "frac": ach / fp4_peak,
                "traffic": None, "kernel": "macro_kernel", "peak_source": "measured in this run (fp4_peak)"}
        cfg = {"workload": "prefill_macro: X[4096,8192] x W[8192,8192]^T, FP16 macro-scales per 256",
               "global_batch": 4096, "l2": "2 rotating weight copies"}
    else:
        roof = None
        cfg = {"workload": "moe_grouped: 2048 tokens, 128 experts top-8, up [768,2048] + down [2048,768]",
               "global_batch": 2048}

    if rank == 0:
        line = {"metric": metric, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "fp4 (e2m1 x e4m3-scaled, fp32 accumulate)", "data": "synthetic",
                "config": cfg, "gpu_launches": r.get("launches_per_step", 0) * args.steps,
                "clocks": clocks, "device_status": r.get("device_status")}
        if roof is not None:
            line["roofline"] = roof
        if cpu is not None:
            line["cpu_baseline"] = cpu
        if "e2e" in r:
            line["e2e"] = r["e2e"]
        if "scale_stats" in r:
            line["scale_stats"] = r["scale_stats"]
        if extras:
            line["workloads"] = extras
        line["fp4_peak"] = fp4_info
        print(json.dumps(line))
    sampler.stop()
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
