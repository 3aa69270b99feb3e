"""Host-side checks of the C ABI that need no GPU: the library builds for
sm_103a and loads, it exports every function include/nvfp4.h declares, the
policy routing rule, the sizing helpers and the argument checks that fail
before anything is enqueued."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "nvfp4.h")


@pytest.fixture(scope="module")
def nv():
    from nvfp4_block_scaled_30_b300 import build
    build.build()
    import nvfp4_block_scaled_30_b300 as nv
    nv.lib()
    return nv


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(nvfp4_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_function(nv):
    names = header_functions()
    assert len(names) >= 12
    L = nv.lib()
    for n in names:
        assert hasattr(L, n), n
    assert sorted(nv.EXPORTED) == names


def test_policy_route(nv):
    r = nv.policy_route
    assert r(nv.POLICY_AUTO, 0) == 4 and r(nv.POLICY_AUTO, 1) == 8
    assert r(nv.POLICY_Q4, 0) == 4 and r(nv.POLICY_Q4, 1) == 4
    assert r(nv.POLICY_Q8, 0) == 8 and r(nv.POLICY_Q8, 1) == 8
    assert nv.lib().nvfp4_policy_route(7, 0) == -1


def test_scale_bytes(nv):
    assert nv.scale_bytes(128, 512, nv.LAYOUT_ROW_MAJOR) == 128 * 32
    assert nv.scale_bytes(1, 8192, nv.LAYOUT_MMA_TILED) == 128 * 512
    assert nv.scale_bytes(130, 320, nv.LAYOUT_MMA_TILED) == 256 * 20
    with pytest.raises(nv.NVFP4Error) as e:
        nv.scale_bytes(4, 48, nv.LAYOUT_MMA_TILED)
    assert e.value.status == nv.ERR_UNSUPPORTED_SHAPE
    with pytest.raises(nv.NVFP4Error) as e:
        nv.scale_bytes(4, 40, nv.LAYOUT_ROW_MAJOR)
    assert e.value.status == nv.ERR_UNSUPPORTED_SHAPE


def test_workspace_size(nv):
    q = nv.workspace_size(nv.OP_QUANTIZE, 4096, 0, 8192)
    g = nv.workspace_size(nv.OP_GEMM, 4096, 8192, 8192)
    assert q >= 256 + 4096 and g > 4096 * 4096  # on-the-fly codes fit
    small = nv.workspace_size(nv.OP_GEMM, 16, 4096, 8192)
    # stream-K (16 N tiles): one FP32 partial tile (16 rows x 256 columns) per SM
    assert small >= 148 * 16 * 256 * 4


def _desc(nv, **kw):
    d = dict(codes=0x10000, scales=0x20000, second=0x30000, rows=128, K=512, mode=0, layout=1)
    d.update(kw)
    return nv.TensorDesc(d["codes"], d["scales"], d["second"], d["rows"], d["K"], d["mode"], d["layout"])


def test_argument_errors_fail_before_any_launch(nv):
    L = nv.lib()
    ws = ctypes.c_void_p(0x40000)
    big = 1 << 30
    # quantize: null output tensor, mismatched rows, bad K
    assert L.nvfp4_quantize(0x1000, 128, 512, 512, None, ws, big, None) == nv.ERR_INVALID_ARG
    d = _desc(nv, rows=64)
    assert L.nvfp4_quantize(0x1000, 128, 512, 512, ctypes.byref(d), ws, big, None) == nv.ERR_INVALID_ARG
    d = _desc(nv, K=96)
    assert L.nvfp4_quantize(0x1000, 128, 96, 96, ctypes.byref(d), ws, big, None) == nv.ERR_UNSUPPORTED_SHAPE
    d = _desc(nv, mode=1, K=320, layout=0)
    assert L.nvfp4_quantize(0x1000, 128, 320, 320, ctypes.byref(d), ws, big, None) == nv.ERR_UNSUPPORTED_SHAPE
    d = _desc(nv)
    assert L.nvfp4_quantize(0x1001, 128, 512, 512, ctypes.byref(d), ws, big, None) == nv.ERR_INVALID_ARG
    assert L.nvfp4_quantize(0x1000, 128, 512, 512, ctypes.byref(d), ctypes.c_void_p(0x40010), big,
                            None) == nv.ERR_WORKSPACE
    assert L.nvfp4_quantize(0x1000, 128, 512, 512, ctypes.byref(d), ws, 16, None) == nv.ERR_WORKSPACE
    # gemm: both or neither activation form, bad policy, row-major weights
    w = _desc(nv, rows=256)
    a = _desc(nv)
    args = (ctypes.c_void_p(0x50000), 256, 0, 128, 0, 0, ws, big, None)
    assert L.nvfp4_gemm(None, 0, None, ctypes.byref(w), *args) == nv.ERR_INVALID_ARG
    assert L.nvfp4_gemm(0x1000, 512, ctypes.byref(a), ctypes.byref(w), *args) == nv.ERR_INVALID_ARG
    assert L.nvfp4_gemm(0x1000, 512, None, ctypes.byref(w), ctypes.c_void_p(0x50000), 256, 0, 128, 9, 0, ws,
                        big, None) == nv.ERR_INVALID_ARG
    wr = _desc(nv, rows=256, layout=0)
    assert L.nvfp4_gemm(0x1000, 512, None, ctypes.byref(wr), *args) == nv.ERR_INVALID_ARG
    # W4A8 route from pre-quantised NVFP4 activations is not a thing
    assert L.nvfp4_gemm(None, 0, ctypes.byref(a), ctypes.byref(w), ctypes.c_void_p(0x50000), 256, 0, 128,
                        nv.POLICY_Q8, 0, ws, big, None) == nv.ERR_UNSUPPORTED
    # output stride below N
    assert L.nvfp4_gemm(0x1000, 512, None, ctypes.byref(w), ctypes.c_void_p(0x50000), 100, 0, 128, 0, 0, ws, big,
                        None) == nv.ERR_INVALID_ARG
    # grouped: E out of range, N not a multiple of 128, W4A8 route
    ga = _desc(nv, rows=2048, K=2048)
    gw = _desc(nv, rows=128 * 768, K=2048)
    off = ctypes.c_void_p(0x60000)
    gargs = (ctypes.c_void_p(0x50000), 768, 0, 16384)
    assert L.nvfp4_grouped_gemm(ctypes.byref(ga), None, off, 0, ctypes.byref(gw), 768, *gargs, 0, 0, ws, big,
                                None) == nv.ERR_INVALID_ARG
    gw2 = _desc(nv, rows=128 * 700, K=2048)
    assert L.nvfp4_grouped_gemm(ctypes.byref(ga), ctypes.c_void_p(0x70000), off, 128, ctypes.byref(gw2), 700,
                                ctypes.c_void_p(0x50000), 700, 0, 16384, 0, 0, ws, big, None) == nv.ERR_UNSUPPORTED_SHAPE
    assert L.nvfp4_grouped_gemm(ctypes.byref(ga), ctypes.c_void_p(0x70000), off, 128, ctypes.byref(gw), 768,
                                *gargs, nv.POLICY_AUTO, 1, ws, big, None) == nv.ERR_UNSUPPORTED
    # fp8 quantiser shape check
    assert L.nvfp4_quantize_fp8(0x1000, 4, 40, 40, 0x2000, 0x3000, ws, big, None) == nv.ERR_UNSUPPORTED_SHAPE
    assert L.nvfp4_workspace_size(9, 1, 1, 1, 0, ctypes.byref(ctypes.c_size_t())) == nv.ERR_INVALID_ARG


def test_kv_argument_errors_fail_before_any_launch(nv):
    L = nv.lib()
    ws, big = ctypes.c_void_p(0x40000), 1 << 30

    def cache(**kw):
        d = dict(pages=0x100000, k_scale=0x2000, v_scale=0x2004, num_pages=64, num_kv_heads=8, head_dim=128,
                 page_tokens=64, format=nv.KV_NVFP4)
        d.update(kw)
        return nv.KvCacheDesc(d["pages"], d["k_scale"], d["v_scale"], d["num_pages"], d["num_kv_heads"],
                              d["head_dim"], d["page_tokens"], d["format"])

    def attn(c, H=64, B=4, max_ctx=4096, out_dtype=0, sm_scale=0.088):
        return L.nvfp4_kv_decode_attention(ctypes.byref(c), 0x3000, H, 0x4000, 0x5000, 65, B, max_ctx, sm_scale,
                                           0x6000, out_dtype, ws, big, None)

    assert attn(cache(format=7)) == nv.ERR_INVALID_ARG
    assert attn(cache(head_dim=64)) == nv.ERR_UNSUPPORTED_SHAPE
    assert attn(cache(pages=0x100008)) == nv.ERR_INVALID_ARG            # pages not 16-byte aligned
    assert attn(cache(), H=60) == nv.ERR_INVALID_ARG                     # not a multiple of the KV heads
    assert attn(cache(), H=8 * 17) == nv.ERR_UNSUPPORTED_SHAPE          # 17 query heads per KV head
    assert attn(cache(), B=65536) == nv.ERR_UNSUPPORTED_SHAPE           # beyond the grid's z limit
    assert attn(cache(num_kv_heads=65536), H=65536) == nv.ERR_UNSUPPORTED_SHAPE
    assert attn(cache(), out_dtype=5) == nv.ERR_INVALID_ARG
    assert attn(cache(), sm_scale=float("nan")) == nv.ERR_INVALID_ARG
    assert L.nvfp4_kv_decode_attention(ctypes.byref(cache()), 0x3000, 64, 0x4000, 0x5000, 65, 4, 4096, 0.088,
                                       0x6000, 0, ctypes.c_void_p(0x40000), 16, None) == nv.ERR_WORKSPACE
    assert L.nvfp4_kv_append(ctypes.byref(cache()), 0x3000, 0x3100, 0x4000, 0x5000, 0, 4, None) == nv.ERR_INVALID_ARG
    assert L.nvfp4_kv_append(None, 0x3000, 0x3100, 0x4000, 0x5000, 65, 4, None) == nv.ERR_INVALID_ARG


def test_output_checks_reject_before_launch(nv):
    # the bindings check an output tensor before its pointer reaches the C ABI
    import torch
    with pytest.raises(ValueError):
        nv._out(torch.empty((8, 16)), 8, 16, nv.OUT_BF16, None)       # not on a GPU
    with pytest.raises(ValueError):
        nv._out(None, 8, 16, 7, None)                                 # no such output type


def test_checked_variant_loads_and_says_so(nv):
    """The bounds-checked build exports the same functions and reports itself;
    the normal build reports that it is not checked and refuses the record
    query.  Host calls only."""
    from nvfp4_block_scaled_30_b300 import build
    path = build.build(checked=True)
    C = ctypes.CDLL(path)
    for n in header_functions():
        assert hasattr(C, n), n
    assert C.nvfp4_diag_bounds_checked() == 1
    L = ctypes.CDLL(build.LIB)
    assert L.nvfp4_diag_bounds_checked() == 0
    n = ctypes.c_uint64(0)
    assert L.nvfp4_diag_bounds_record(ctypes.byref(n), None, 0, None, None, 0) == nv.ERR_UNSUPPORTED
    # argument checks of the self-test come before any launch
    assert C.nvfp4_diag_bounds_selftest(None, ctypes.c_uint64(4160), ctypes.c_uint64(4096), None) == nv.ERR_INVALID_ARG
    assert C.nvfp4_diag_bounds_selftest(ctypes.c_void_p(0x1000), ctypes.c_uint64(4100), ctypes.c_uint64(4096),
                                        None) == nv.ERR_INVALID_ARG
