"""Device-side failure detection without a GPU fault: a stream-K CTA is told
(test-only flag) never to raise its ready flag, so the owner of its tile
waits on a flag that nothing sets.  The bounded wait must give up after the
requested limit, record TIMEOUT in the workspace status word and let the
kernel exit; the context stays usable and, after nvfp4_workspace_init, the
same workspace gives the oracle's result again."""
import ctypes
import time

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_common import nv, nvfp4_device, y_np
from helpers import row_tolerance_ok

pytestmark = pytest.mark.gpu


def test_skipped_streamk_flag_times_out_and_recovers():
    M, N, K = 8, 4096, 8192
    xb = synth.activations(9, 70, M, K, 0.01, 50.0)
    wb = synth.weights(9, 71, N, K)
    ac, as_, ag = oracle.nvfp4_encode(xb)
    wc, ws, wg = oracle.nvfp4_encode(wb)
    a = nvfp4_device(ac, as_, ag, M, K)
    w = nvfp4_device(wc, ws, wg, N, K)
    work = nv.Workspace(nv.workspace_size(nv.OP_GEMM, M, N, K))
    y = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    ad, wd = a.desc(), w.desc()
    stream = torch.cuda.current_stream()
    t0 = time.time()
    st = nv.lib().nvfp4_diag_streamk_skip_flag(ctypes.byref(ad), ctypes.byref(wd), y.data_ptr(), y.stride(0),
                                               nv.OUT_FP32, 1, 50_000_000, work.ptr, work.nbytes,
                                               stream.cuda_stream)
    assert st == nv.OK
    assert work.status() == nv.ERR_TIMEOUT          # synchronises, reads and clears the word
    assert time.time() - t0 < 10.0
    # the context is still usable; re-initialised, the workspace works again
    assert nv.lib().nvfp4_workspace_init(work.ptr, work.nbytes, stream.cuda_stream) == nv.OK
    y2 = y_np(nv.gemm(w, a_q=a, out_dtype=nv.OUT_FP32, ws=work))
    assert work.status() == nv.OK
    ok, worst = row_tolerance_ok(y2, oracle.gemm_w4a4((ac, as_, ag), (wc, ws, wg)))
    assert ok, worst


def test_skip_flag_needs_a_streamk_shape():
    M, N, K = 256, 512, 512                           # whole tiles: no stream-K
    ac, as_ = np.zeros((M, K // 2), np.uint8), np.full((M, K // 16), 0x38, np.uint8)
    wc, ws = np.zeros((N, K // 2), np.uint8), np.full((N, K // 16), 0x38, np.uint8)
    a, w = nvfp4_device(ac, as_, 1.0, M, K), nvfp4_device(wc, ws, 1.0, N, K)
    work = nv.Workspace(nv.workspace_size(nv.OP_GEMM, M, N, K))
    y = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    ad, wd = a.desc(), w.desc()
    st = nv.lib().nvfp4_diag_streamk_skip_flag(ctypes.byref(ad), ctypes.byref(wd), y.data_ptr(), y.stride(0),
                                               nv.OUT_FP32, 1, 50_000_000, work.ptr, work.nbytes,
                                               torch.cuda.current_stream().cuda_stream)
    assert st == nv.ERR_UNSUPPORTED_SHAPE
