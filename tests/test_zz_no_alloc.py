"""The no-allocation W4A4 entry point, for callers that cannot allocate device
memory at call time (a framework that owns all device memory in its own pool,
a plugin without allocation rights, a serving loop that must not reach the
allocator).  Its output must match the CPU oracle's FP64 product of the same
NVFP4 operands, within the GEMM tolerance of the other tests, on two calls in
a row (the calls share the library's fixed scratch array, so the second call
checks that the first left nothing behind that changes the result), for BF16
and FP32 outputs, and when two streams take turns ordered by an event.
This file runs last so that a failure here comes after every other test."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_common import dev_bf16, nv, quantize_pinned, y_np
from helpers import row_tolerance_ok

pytestmark = pytest.mark.gpu


def _operands(M, N, K, seed):
    """Device NVFP4 operands (GPU encodes checked bit for bit against the
    oracle's) and the oracle's FP64 product of the oracle's encodes."""
    xb = synth.activations(9, seed, M, K, 0.005, 100.0)
    wb = synth.weights(9, seed + 1, N, K)
    a_q, ac, as_, ag = quantize_pinned(xb)
    w, wc, ws, wg = quantize_pinned(wb)
    ref = oracle.gemm_w4a4((ac, as_, ag[0]), (wc, ws, wg[0]))
    return a_q, w, ref


@pytest.mark.parametrize("M,N,K", [(8, 4096, 8192), (16, 2944, 8192), (16, 28672, 8192), (200, 512, 1024)])
@pytest.mark.parametrize("out_dtype", [nv.OUT_BF16, nv.OUT_FP32])
def test_noalloc_matches_oracle_twice(M, N, K, out_dtype):
    a_q, w, ref = _operands(M, N, K, 40)
    dt = torch.bfloat16 if out_dtype == nv.OUT_BF16 else torch.float32
    for _ in range(2):
        y = torch.full((M, N), float("nan"), dtype=dt, device="cuda")
        nv.gemm_w4a4_noalloc(a_q, w, y, out_dtype=out_dtype)
        assert nv.noalloc_status() == nv.OK
        ok, worst = row_tolerance_ok(y_np(y), ref, out_bf16=out_dtype == nv.OUT_BF16)
        assert ok, f"{M}x{N}x{K}: worst row error ratio {worst:.3e}"


def test_noalloc_two_streams_ordered_by_an_event():
    # two streams take turns on the shared scratch; the event orders them,
    # as the header asks of callers on several streams
    a_q, w, ref = _operands(16, 2944, 8192, 44)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    y1 = torch.empty((16, 2944), dtype=torch.float32, device="cuda")
    y2 = torch.empty_like(y1)
    torch.cuda.synchronize()
    ev = torch.cuda.Event()
    nv.gemm_w4a4_noalloc(a_q, w, y1, out_dtype=nv.OUT_FP32, stream=s1)
    ev.record(s1)
    s2.wait_event(ev)
    nv.gemm_w4a4_noalloc(a_q, w, y2, out_dtype=nv.OUT_FP32, stream=s2)
    assert nv.noalloc_status(stream=s2) == nv.OK
    torch.cuda.synchronize()
    for y in (y1, y2):
        ok, worst = row_tolerance_ok(y_np(y), ref, out_bf16=False)
        assert ok, f"worst row error ratio {worst:.3e}"


def test_noalloc_rejects_shapes_beyond_its_scratch():
    # a narrow stream-K shape (16 N tiles) whose partial tiles (128 rows x
    # 256 columns of FP32 per SM) exceed 4 MiB
    a_q, w, _ = _operands(128, 4096, 8192, 50)
    y = torch.empty((128, 4096), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(nv.NVFP4Error) as e:
        nv.gemm_w4a4_noalloc(a_q, w, y)
    assert e.value.status == nv.ERR_WORKSPACE


def test_noalloc_rejects_a_wrong_output_before_launch():
    a_q, w, _ = _operands(8, 4096, 8192, 52)
    with pytest.raises(ValueError):   # BF16 output expected, FP32 given
        nv.gemm_w4a4_noalloc(a_q, w, torch.empty((8, 4096), dtype=torch.float32, device="cuda"))
    with pytest.raises(ValueError):   # FP32 output expected, BF16 given
        nv.gemm_w4a4_noalloc(a_q, w, torch.empty((8, 4096), dtype=torch.bfloat16, device="cuda"),
                             out_dtype=nv.OUT_FP32)
    with pytest.raises(ValueError):   # too few columns
        nv.gemm_w4a4_noalloc(a_q, w, torch.empty((8, 4000), dtype=torch.bfloat16, device="cuda"))
