"""The measuring instruments the bench divides by: the dense FP4
tensor-core rate (nvfp4_diag_fp4_mma_rate, the prefill roofline's peak) and
the copy engine's streaming rate with the GEMM's weight boxes
(nvfp4_diag_tma_stream, the decode roofline's practical ceiling).  Each must
run to completion without a timeout and report rates inside what the
hardware can do: the FP4 rate at most one M = 128, N = 256, K = 64
block-scaled FP4 MMA per 128 cycles and SM, steady from run to run."""
import pytest
import torch

import nvfp4_block_scaled_30_b300 as nv

pytestmark = pytest.mark.gpu


def test_fp4_mma_rate_is_steady_and_at_most_one_mma_per_128_cycles():
    # as the bench runs it: long launches (~0.1 s each), three of them.
    # 2 * 128 * 256 * 64 FLOP per 128 cycles = 32768 FLOP per cycle and SM is
    # the tensor core's rate; the loop includes its fill and drain, so a
    # little below.  On most boxes it reads 32768; two fresh boxes read
    # exactly 15463 (every run, to 7 digits), so the floor here is loose and
    # the bench takes its peak from event time on the box it runs on
    nv.fp4_mma_rate(200)
    runs = [nv.fp4_mma_rate(400000) for _ in range(3)]
    assert all(r[2] == nv.sm_count() and r[1] > 0 for r in runs)
    info = [(round(r[0]), round(r[1], 3), round(400000 * 4 * nv.FP4_MMA_FLOP / r[0] / (r[1] * 1e-3) / 1e9, 3))
            for r in runs]   # FLOP/cycle/SM, ms, implied clock GHz
    print("fp4 mma rate:", info)
    rates = [r[0] for r in runs]
    assert max(rates) <= 1.001 * 32768 and min(rates) >= 0.4 * 32768, info
    assert max(rates) <= 1.02 * min(rates), info   # the cycle count is steady from run to run


def test_tma_stream_runs_and_stays_under_the_copy_peak():
    rows, row_bytes = 28672, 4096
    w = torch.randint(0, 255, (rows, row_bytes), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for grid in (1, 7, rows // 256, nv.sm_count()):
        nv.tma_stream(w, grid, status)
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        nv.tma_stream(w, grid, status)
        e.record()
        e.synchronize()
        gbs = rows * row_bytes / (s.elapsed_time(e) * 1e-3) / 1e9
        assert int(status.item()) == 0, f"grid {grid}: a bounded wait ran out"
        assert 0 < gbs < 8000, gbs   # below HBM3e's nominal 7.7 TB/s (and L2 holds only part of 117 MB)


def test_tma_stream_argument_checks():
    w = torch.zeros((256, 4096), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for bad in (torch.zeros((255, 4096), dtype=torch.uint8, device="cuda"),    # rows not a multiple of 256
                torch.zeros((256, 4000), dtype=torch.uint8, device="cuda")):   # row bytes not a multiple of 128
        with pytest.raises(nv.NVFP4Error) as e:
            nv.tma_stream(bad, 4, status)
        assert e.value.status == nv.ERR_INVALID_ARG
    with pytest.raises(nv.NVFP4Error):
        nv.tma_stream(w, 0, status)
