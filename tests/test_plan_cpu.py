"""The W4A4 launch plan, host logic only (nvfp4_gemm_kernel_path: no launch;
without a GPU the library plans for 148 SMs, the B300's count).  Stream-K
only for M <= 128 when the N tiles cover under 60% of the SMs and there are
at least two 256-element K steps per SM to share; several M tiles always run
whole tiles (both rules measured on B300; the reasons are recorded beside
the plan in gemm_w4a4.cu)."""
import pytest

import nvfp4_block_scaled_30_b300 as nv


def _sms_or_skip():
    n = nv.lib().nvfp4_sm_count()
    if n not in (0, 148):
        pytest.skip(f"planned for 148 SMs, this device has {n}")


@pytest.mark.parametrize("M,N,K,path", [
    (1, 28672, 8192, nv.PATH_WHOLE_TILES),    # decode: 112 tiles keep HBM busy
    (8, 28672, 8192, nv.PATH_WHOLE_TILES),
    (16, 28672, 8192, nv.PATH_WHOLE_TILES),
    (8, 4096, 8192, nv.PATH_STREAMK),         # 16 tiles x 32 K steps
    (128, 4096, 8192, nv.PATH_STREAMK),
    (129, 4096, 8192, nv.PATH_WHOLE_TILES),   # two M tiles
    (8, 4096, 1024, nv.PATH_WHOLE_TILES),     # 16 x 4 K steps: too little to share
    (8, 22528, 8192, nv.PATH_STREAMK),        # 88 tiles: under 60 % of 148
    (8, 22784, 8192, nv.PATH_WHOLE_TILES),    # 89 tiles: not under 60 %
    (2048, 4096, 4096, nv.PATH_WHOLE_TILES),  # policy-stack layer
    (4096, 8192, 8192, nv.PATH_WHOLE_TILES),  # prefill
])
def test_kernel_path(M, N, K, path):
    _sms_or_skip()
    assert nv.gemm_kernel_path(M, N, K) == path


def test_rejected_sizes_have_no_path():
    assert nv.gemm_kernel_path(8, 4096, 100) == -1      # K not a multiple of 64
    assert nv.gemm_kernel_path(0, 4096, 8192) == -1


def test_streamk_workspace_holds_one_partial_tile_per_sm():
    _sms_or_skip()
    whole = nv.workspace_size(nv.OP_GEMM, 8, 28672, 8192)
    sk = nv.workspace_size(nv.OP_GEMM, 8, 4096, 8192)
    # 148 FP32 slots of 8 rows x 256 columns, plus one ready flag per CTA
    assert sk >= 148 * 8 * 256 * 4 + 148 * 4
    assert whole < 148 * 8 * 256 * 4
