"""The no-allocation W4A4 entry point, for callers that cannot allocate device
memory at call time (a framework that owns all device memory in its own pool,
a plugin without allocation rights, a serving loop that must not reach the
allocator).  Its output must match the workspace entry point nvfp4_gemm on
the same operands, within the GEMM tolerance of the other tests, on two calls
in a row (the calls share the library's fixed scratch array, so the second
call checks that the first left nothing behind that changes the result).
This file runs last so that a failure here comes after every other test."""
import ctypes

import numpy as np
import pytest
import torch

import synth
from gpu_common import dev_bf16, nv, y_np
from helpers import row_tolerance_ok

pytestmark = pytest.mark.gpu


def _operands(M, N, K, seed):
    x = dev_bf16(synth.activations(9, seed, M, K, 0.005, 100.0))
    w = nv.quantize(dev_bf16(synth.weights(9, seed + 1, N, K)))
    a_q = nv.quantize(x)
    return a_q, w


@pytest.mark.parametrize("M,N,K", [(8, 4096, 8192), (16, 2944, 8192), (16, 28672, 8192), (200, 512, 1024)])
def test_noalloc_matches_workspace_entry_point_twice(M, N, K):
    a_q, w = _operands(M, N, K, 40)
    y_ref = y_np(nv.gemm(w, a_q=a_q, out_dtype=nv.OUT_FP32))
    for _ in range(2):
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        ad, wd = a_q.desc(), w.desc()
        st = nv.lib().nvfp4_gemm_w4a4_noalloc(ctypes.byref(ad), ctypes.byref(wd), y.data_ptr(), y.stride(0),
                                              nv.OUT_FP32, torch.cuda.current_stream().cuda_stream)
        assert st == nv.OK
        ok, worst = row_tolerance_ok(y_np(y), y_ref)
        assert ok, f"{M}x{N}x{K}: worst row error ratio {worst:.3e}"


def test_noalloc_rejects_shapes_beyond_its_scratch():
    # a narrow stream-K shape (16 N tiles) whose partial tiles (128 rows x
    # 256 columns of FP32 per SM) exceed 4 MiB
    a_q, w = _operands(128, 4096, 8192, 50)
    y = torch.empty((128, 4096), dtype=torch.bfloat16, device="cuda")
    ad, wd = a_q.desc(), w.desc()
    st = nv.lib().nvfp4_gemm_w4a4_noalloc(ctypes.byref(ad), ctypes.byref(wd), y.data_ptr(), y.stride(0),
                                          nv.OUT_BF16, torch.cuda.current_stream().cuda_stream)
    assert st == nv.ERR_WORKSPACE
