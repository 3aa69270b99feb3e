"""Exhaustive check of the kernels' own element conversions: every one of the
2^32 binary32 bit patterns (NaNs excluded from the comparison) through the
device E2M1 and E4M3 conversions used by the quantisers, against the
oracle's round-to-nearest-even, saturating encoders."""
import numpy as np
import pytest
import torch

import oracle
from gpu_common import nv

pytestmark = pytest.mark.gpu

CHUNK = 1 << 28


@pytest.mark.parametrize("chunk", range((1 << 32) // CHUNK))
def test_all_float_bit_patterns(chunk):
    start = chunk * CHUNK
    bits = torch.arange(start, start + CHUNK, dtype=torch.int64, device="cuda")
    v = ((bits + (1 << 31)) % (1 << 32) - (1 << 31)).to(torch.int32).view(torch.float32)
    g2, g3 = nv.probe_convert(v)
    torch.cuda.synchronize()
    hv = np.arange(start, start + CHUNK, dtype=np.uint64).astype(np.uint32).view(np.float32)
    finite_or_inf = ~np.isnan(hv)
    o2 = oracle.e2m1_encode_array(hv)
    o3 = oracle.e4m3_encode_array(hv)
    d2 = g2.cpu().numpy()
    d3 = g3.cpu().numpy()
    bad2 = np.flatnonzero((d2 != o2) & finite_or_inf)
    bad3 = np.flatnonzero((d3 != o3) & finite_or_inf)
    assert bad2.size == 0, f"E2M1: {bad2.size} mismatches, e.g. {[(hex(int(start + i)), d2[i], o2[i]) for i in bad2[:4]]}"
    assert bad3.size == 0, f"E4M3: {bad3.size} mismatches, e.g. {[(hex(int(start + i)), d3[i], o3[i]) for i in bad3[:4]]}"
