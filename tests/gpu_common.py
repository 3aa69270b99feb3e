"""Shared plumbing for the GPU tests: host <-> device moves through the
binding (which calls the C ABI).  No method arithmetic here."""
import numpy as np
import torch

import nvfp4_block_scaled_30_b300 as nv
import oracle
from helpers import tile_scales, untile_scales


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits, np.uint16).view(np.int16)).cuda().view(torch.bfloat16)


def host(t: torch.Tensor) -> np.ndarray:
    torch.cuda.synchronize()
    return t.cpu().numpy()


def quantize_gpu(bits: np.ndarray, mode=nv.SCALE_TENSOR_FP32, layout=nv.LAYOUT_MMA_TILED, ws=None):
    """GPU NVFP4 encode of BF16 bits; returns (NVFP4Tensor, codes, row-major
    scales, second) with the numpy copies for comparison."""
    x = dev_bf16(bits)
    t = nv.quantize(x, mode=mode, layout=layout, ws=ws)
    rows, K = bits.shape
    codes = host(t.codes)
    sc = host(t.scales)
    scales = untile_scales(sc, rows, K) if layout == nv.LAYOUT_MMA_TILED else sc.reshape(rows, K // 16)
    second = host(t.second)
    if mode == nv.SCALE_MACRO_FP16:
        second = second.view(np.uint16)
    return t, codes, scales, second


def quantize_pinned(bits: np.ndarray, mode=nv.SCALE_TENSOR_FP32, ws=None):
    """GPU NVFP4 encode (MMA-tiled scales) of BF16 bits, checked bit for bit
    against the oracle's encode of the same bits.  Returns the device tensor
    and the ORACLE's (codes, row-major scales, second), so that every
    reference a test computes from them starts from oracle values only."""
    t, codes, scales, second = quantize_gpu(bits, mode, nv.LAYOUT_MMA_TILED, ws)
    if mode == nv.SCALE_TENSOR_FP32:
        oc, os_, og = oracle.nvfp4_encode(bits)
        osec = np.array([og], np.float32)
        assert second.view(np.uint32)[0] == osec.view(np.uint32)[0], "tensor scale differs from the oracle's"
    else:
        oc, os_, osec = oracle.nvfp4_encode_macro(bits)
        np.testing.assert_array_equal(second, osec)
    np.testing.assert_array_equal(codes, oc)
    np.testing.assert_array_equal(scales, os_)
    return t, oc, os_, osec


def nvfp4_device(codes: np.ndarray, scales_rm: np.ndarray, second, rows: int, K: int,
                 mode=nv.SCALE_TENSOR_FP32) -> nv.NVFP4Tensor:
    """Device NVFP4 tensor with MMA-tiled scales from host arrays."""
    c = torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).cuda()
    s = torch.from_numpy(tile_scales(np.asarray(scales_rm, np.uint8), rows, K)).cuda()
    if mode == nv.SCALE_TENSOR_FP32:
        sec = torch.from_numpy(np.atleast_1d(np.asarray(second, np.float32)).copy()).cuda()
    else:
        sec = torch.from_numpy(np.ascontiguousarray(second, np.uint16).view(np.int16)).cuda()
    return nv.NVFP4Tensor(c, s, sec, rows, K, mode, nv.LAYOUT_MMA_TILED)


def y_np(y: torch.Tensor) -> np.ndarray:
    return host(y.float()).astype(np.float64)
