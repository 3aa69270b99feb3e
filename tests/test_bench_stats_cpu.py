"""bench.py's scale statistics (logged beside the timings): the E4M3 byte
table against torch's float8_e4m3fn, and the statistics of a small tensor
with hand-picked scale bytes and zero padding."""
import numpy as np
import torch

import bench
import nvfp4_block_scaled_30_b300 as nv


def test_e4m3_table_matches_torch():
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = bench.E4M3_VALUES
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])


def test_scale_stats_of_a_small_tensor():
    # 2 rows x 64 columns = 8 blocks; 8 more zero bytes stand for tiled padding
    sb = torch.tensor([0x38, 0x01, 0x7E, 0x00, 0x38, 0x38, 0x38, 0x38] + [0] * 8, dtype=torch.uint8)
    q = nv.NVFP4Tensor(torch.zeros(2, 32, dtype=torch.uint8), sb, torch.tensor([0.5]), 2, 64)
    st = bench.scale_stats(q)
    assert st["tensor_scale"] == 0.5
    assert st["block_scale_min"] == 2.0 ** -9      # 0x01: the smallest subnormal
    assert st["block_scale_max"] == 448.0          # 0x7E: the largest finite value
    assert st["zero_block_frac"] == 1 / 8          # one real block has scale 0
