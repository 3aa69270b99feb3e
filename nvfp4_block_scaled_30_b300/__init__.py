"""Python binding of libnvfp4 (the NVFP4 W4A4 / W4A8 inference-GEMM hot path
for B300, sm_103a).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels behind the C ABI declared in include/nvfp4.h.  PyTorch supplies
device memory and the current CUDA stream.  If libnvfp4.so is missing or a
call fails, the functions raise; there is no fallback implementation.
"""
import ctypes
import dataclasses
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# NVFP4_LIB=checked loads the bounds-checked build (libnvfp4_checked.so:
# every kernel access tested first, failures recorded; see bounds_record)
LIB_VARIANT = os.environ.get("NVFP4_LIB", "")
if LIB_VARIANT not in ("", "checked"):
    raise RuntimeError(f"NVFP4_LIB={LIB_VARIANT!r}: expected unset or 'checked'")
LIB_NAME = "libnvfp4_checked.so" if LIB_VARIANT == "checked" else "libnvfp4.so"
LIB_PATH = os.path.join(_HERE, LIB_NAME)

# ---- enums (include/nvfp4.h) -----------------------------------------------------
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED_SHAPE, ERR_NONFINITE_INPUT, ERR_TIMEOUT, ERR_CUDA, \
    ERR_WORKSPACE, ERR_UNSUPPORTED = range(8)
STATUS_NAMES = {OK: "OK", ERR_INVALID_ARG: "INVALID_ARG", ERR_UNSUPPORTED_SHAPE: "UNSUPPORTED_SHAPE",
                ERR_NONFINITE_INPUT: "NONFINITE_INPUT", ERR_TIMEOUT: "TIMEOUT", ERR_CUDA: "CUDA",
                ERR_WORKSPACE: "WORKSPACE", ERR_UNSUPPORTED: "UNSUPPORTED"}
POLICY_AUTO, POLICY_Q4, POLICY_Q8 = 0, 1, 2
SCALE_TENSOR_FP32, SCALE_MACRO_FP16 = 0, 1
LAYOUT_ROW_MAJOR, LAYOUT_MMA_TILED = 0, 1
OUT_BF16, OUT_FP32 = 0, 1
OP_QUANTIZE, OP_QUANTIZE_FP8, OP_GEMM, OP_W4A8_GEMM, OP_GROUPED_GEMM, OP_GROUPED_GEMM_X, OP_KV_DECODE = range(7)

EXPORTED = ["nvfp4_scale_bytes", "nvfp4_workspace_size", "nvfp4_workspace_init", "nvfp4_device_status",
            "nvfp4_policy_route", "nvfp4_quantize", "nvfp4_quantize_fp8", "nvfp4_gemm", "nvfp4_w4a8_gemm",
            "nvfp4_grouped_gemm", "nvfp4_probe_convert", "nvfp4_sm_count", "nvfp4_version",
            "nvfp4_gemm_w4a4_noalloc", "nvfp4_gemm_nvfp4_out", "nvfp4_moe_up_swiglu",
            "nvfp4_moe_down_combine", "nvfp4_grouped_w4a8_gemm", "nvfp4_grouped_gemm_x",
            "nvfp4_diag_streamk_skip_flag", "nvfp4_kv_append", "nvfp4_kv_decode_attention",
            "nvfp4_gemm_kernel_path", "nvfp4_diag_fp4_mma_rate", "nvfp4_gemm_w4a4_noalloc_status",
            "nvfp4_diag_bounds_checked", "nvfp4_diag_bounds_record", "nvfp4_diag_bounds_selftest",
            "nvfp4_diag_tma_stream"]


def _require(ok: bool, what: str) -> None:
    """Argument check of the bindings (kept under python -O, unlike assert):
    a wrong dtype or layout must not reach the C ABI as a raw pointer."""
    if not ok:
        raise ValueError(what)


class NVFP4Error(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}")
        self.status = status


class TensorDesc(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("second", ctypes.c_void_p),
                ("rows", ctypes.c_int64), ("K", ctypes.c_int64), ("mode", ctypes.c_int32),
                ("layout", ctypes.c_int32)]


class KvCacheDesc(ctypes.Structure):
    _fields_ = [("pages", ctypes.c_void_p), ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
                ("num_pages", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("page_tokens", ctypes.c_int32), ("format", ctypes.c_int32)]


_LIB = None
_I64, _I32, _VP, _SZ = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t
_PT = ctypes.POINTER(TensorDesc)


def lib():
    """Load libnvfp4.so, or libnvfp4_checked.so under NVFP4_LIB=checked
    (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            flag = " --checked" if LIB_VARIANT == "checked" else ""
            raise RuntimeError(f"{LIB_NAME} not built ({LIB_PATH}); run "
                               f"python -m nvfp4_block_scaled_30_b300.build{flag}")
        L = ctypes.CDLL(LIB_PATH)
        sig = {
            "nvfp4_scale_bytes": (_I32, [_I64, _I64, _I32, ctypes.POINTER(_SZ)]),
            "nvfp4_workspace_size": (_I32, [_I32, _I64, _I64, _I64, _I32, ctypes.POINTER(_SZ)]),
            "nvfp4_workspace_init": (_I32, [_VP, _SZ, _VP]),
            "nvfp4_device_status": (_I32, [_VP, _VP, ctypes.POINTER(_I32)]),
            "nvfp4_policy_route": (_I32, [_I32, _I32]),
            "nvfp4_quantize": (_I32, [_VP, _I64, _I64, _I64, _PT, _VP, _SZ, _VP]),
            "nvfp4_quantize_fp8": (_I32, [_VP, _I64, _I64, _I64, _VP, _VP, _VP, _SZ, _VP]),
            "nvfp4_gemm": (_I32, [_VP, _I64, _PT, _PT, _VP, _I64, _I32, _I64, _I32, _I32, _VP, _SZ, _VP]),
            "nvfp4_w4a8_gemm": (_I32, [_VP, _VP, _PT, _VP, _I64, _I32, _I64, _VP, _SZ, _VP]),
            "nvfp4_grouped_gemm": (_I32, [_PT, _VP, _VP, _I32, _PT, _I64, _VP, _I64, _I32, _I64, _I32, _I32,
                                          _VP, _SZ, _VP]),
            "nvfp4_probe_convert": (_I32, [_VP, _I64, _VP, _VP, _VP]),
            "nvfp4_diag_streamk_skip_flag": (_I32, [_PT, _PT, _VP, _I64, _I32, _I32, ctypes.c_uint64, _VP, _SZ,
                                                    _VP]),
            "nvfp4_gemm_w4a4_noalloc": (_I32, [_PT, _PT, _VP, _I64, _I32, _VP]),
            "nvfp4_gemm_w4a4_noalloc_status": (_I32, [_VP, ctypes.POINTER(_I32)]),
            "nvfp4_gemm_nvfp4_out": (_I32, [_VP, _I64, _PT, _PT, _PT, _VP, _I64, _VP, _SZ, _VP]),
            "nvfp4_grouped_w4a8_gemm": (_I32, [_VP, _VP, _I64, _VP, _VP, _I32, _PT, _I64, _VP, _I64, _I32, _I64,
                                               _VP, _SZ, _VP]),
            "nvfp4_grouped_gemm_x": (_I32, [_VP, _I64, _I64, _VP, _VP, _I32, _PT, _I64, _VP, _I64, _I32, _I64,
                                            _I32, _I32, _VP, _SZ, _VP]),
            "nvfp4_kv_append": (_I32, [ctypes.POINTER(KvCacheDesc), _VP, _VP, _VP, _VP, _I32, _I32, _VP]),
            "nvfp4_kv_decode_attention": (_I32, [ctypes.POINTER(KvCacheDesc), _VP, _I32, _VP, _VP, _I32, _I32,
                                                 _I32, ctypes.c_float, _VP, _I32, _VP, _SZ, _VP]),
            "nvfp4_moe_up_swiglu": (_I32, [_PT, _VP, _VP, _I32, _PT, _I64, _VP, _I64, _I32, _PT, _VP, _I64,
                                           _VP, _SZ, _VP]),
            "nvfp4_moe_down_combine": (_I32, [_PT, _VP, _I32, _PT, _I64, _VP, _VP, _VP, _I64, _I64, _I64,
                                              _VP, _SZ, _VP]),
            "nvfp4_sm_count": (_I32, []),
            "nvfp4_gemm_kernel_path": (_I32, [_I64, _I64, _I64]),
            "nvfp4_diag_fp4_mma_rate": (_I32, [_I32, _VP, _VP]),
            "nvfp4_diag_bounds_checked": (_I32, []),
            "nvfp4_diag_bounds_record": (_I32, [ctypes.POINTER(ctypes.c_uint64), ctypes.c_char_p, _I32,
                                                ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(ctypes.c_uint64),
                                                _I32]),
            "nvfp4_diag_bounds_selftest": (_I32, [_VP, ctypes.c_uint64, ctypes.c_uint64, _VP]),
            "nvfp4_diag_tma_stream": (_I32, [_VP, _I64, _I64, _I32, _VP, _VP]),
            "nvfp4_version": (ctypes.c_char_p, []),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _LIB = L
    return _LIB


def _check(status: int, where: str):
    if status != OK:
        raise NVFP4Error(status, where)


def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


# ---- tensors and workspaces ----------------------------------------------------------

@dataclasses.dataclass
class NVFP4Tensor:
    """Device NVFP4 tensor [rows, K]: packed E2M1 codes uint8 [rows, K/2],
    E4M3 scale bytes (row-major [rows, K/16] or MMA-tiled), and the second
    level (float32 [1] or [E] tensor scale, or binary16 [rows, K/256] macro)."""
    codes: torch.Tensor
    scales: torch.Tensor
    second: torch.Tensor
    rows: int
    K: int
    mode: int = SCALE_TENSOR_FP32
    layout: int = LAYOUT_MMA_TILED

    def desc(self) -> TensorDesc:
        return TensorDesc(self.codes.data_ptr(), self.scales.data_ptr(), self.second.data_ptr(),
                          self.rows, self.K, self.mode, self.layout)


def scale_bytes(rows: int, K: int, layout: int = LAYOUT_MMA_TILED) -> int:
    n = _SZ(0)
    _check(lib().nvfp4_scale_bytes(rows, K, layout, ctypes.byref(n)), "nvfp4_scale_bytes")
    return n.value


def workspace_size(op: int, M: int = 0, N: int = 0, K: int = 0, E: int = 0) -> int:
    n = _SZ(0)
    _check(lib().nvfp4_workspace_size(op, M, N, K, E, ctypes.byref(n)), "nvfp4_workspace_size")
    return n.value


class Workspace:
    """Caller-owned device scratch (holds the sticky device status word)."""

    def __init__(self, nbytes: int, device="cuda", stream=None):
        self.buf = torch.empty(max(nbytes, 256) + 256, dtype=torch.uint8, device=device)
        off = (-self.buf.data_ptr()) % 256
        self.ptr = self.buf.data_ptr() + off
        self.nbytes = self.buf.numel() - off
        _check(lib().nvfp4_workspace_init(self.ptr, self.nbytes, _stream(stream)), "nvfp4_workspace_init")

    def ensure(self, nbytes: int, stream=None) -> "Workspace":
        return self if nbytes <= self.nbytes else Workspace(nbytes, self.buf.device, stream)

    def status(self, stream=None) -> int:
        out = _I32(0)
        _check(lib().nvfp4_device_status(self.ptr, _stream(stream), ctypes.byref(out)), "nvfp4_device_status")
        return out.value


def _ws(ws: Optional[Workspace], need: int, device) -> Workspace:
    if ws is None:
        return Workspace(need, device)
    if ws.nbytes < need:
        raise NVFP4Error(ERR_WORKSPACE, f"workspace of {ws.nbytes} bytes < {need}")
    return ws


def empty_nvfp4(rows: int, K: int, mode: int = SCALE_TENSOR_FP32, layout: int = LAYOUT_MMA_TILED,
                device="cuda", n_second: int = 1) -> NVFP4Tensor:
    codes = torch.empty((rows, K // 2), dtype=torch.uint8, device=device)
    scales = torch.empty(scale_bytes(rows, K, layout), dtype=torch.uint8, device=device)
    if mode == SCALE_TENSOR_FP32:
        second = torch.empty(n_second, dtype=torch.float32, device=device)
    else:
        second = torch.empty((rows, K // 256), dtype=torch.int16, device=device)
    return NVFP4Tensor(codes, scales, second, rows, K, mode, layout)


# ---- the hot path ----------------------------------------------------------------------

PATH_WHOLE_TILES, PATH_STREAMK = 1, 2


def gemm_kernel_path(M: int, N: int, K: int) -> int:
    """nvfp4_gemm_kernel_path: whole tiles or stream-K for the W4A4 shape."""
    return lib().nvfp4_gemm_kernel_path(M, N, K)


def sm_count() -> int:
    """nvfp4_sm_count: streaming multiprocessors of the current device."""
    return lib().nvfp4_sm_count()


FP4_MMA_FLOP = 2 * 128 * 256 * 64  # one kind::mxf4nvf4 M=128 N=256 K=64 instruction


def fp4_mma_rate(iters: int = 20000, stream=None):
    """nvfp4_diag_fp4_mma_rate: returns (FLOP per cycle and SM, elapsed ms of the
    launch, SM count).  The rate is the slowest CTA's; ms is CUDA-event time
    on the launching stream."""
    n = sm_count()
    cyc = torch.zeros(n, dtype=torch.int64, device="cuda")
    s = stream if stream is not None else torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    _check(lib().nvfp4_diag_fp4_mma_rate(iters, cyc.data_ptr(), s.cuda_stream), "nvfp4_diag_fp4_mma_rate")
    e1.record(s)
    e1.synchronize()
    c = cyc.cpu()
    worst = int(c.max()) if int(c.min()) >= 0 else -1  # ~0 (a wait that ran out) reads as -1
    if worst <= 0:
        raise NVFP4Error(ERR_TIMEOUT, "nvfp4_diag_fp4_mma_rate: a CTA's wait ran out")
    return iters * 4 * FP4_MMA_FLOP / worst, e0.elapsed_time(e1), n


def policy_route(policy: int, sensitive: int) -> int:
    return lib().nvfp4_policy_route(policy, int(bool(sensitive)))


def quantize(x: torch.Tensor, mode: int = SCALE_TENSOR_FP32, layout: int = LAYOUT_MMA_TILED,
             out: Optional[NVFP4Tensor] = None, ws: Optional[Workspace] = None, stream=None) -> NVFP4Tensor:
    """nvfp4_quantize of a BF16 [rows, K] tensor (row stride x.stride(0))."""
    _require(x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1,
             "quantize: x must be a 2-D BF16 tensor with unit column stride")
    rows, K = x.shape
    if out is None:
        out = empty_nvfp4(rows, K, mode, layout, x.device)
    ws = _ws(ws, workspace_size(OP_QUANTIZE, rows, 0, K), x.device)
    d = out.desc()
    _check(lib().nvfp4_quantize(_ptr(x), rows, K, x.stride(0), ctypes.byref(d), ws.ptr, ws.nbytes,
                                _stream(stream)), "nvfp4_quantize")
    return out


def quantize_fp8(x: torch.Tensor, ws: Optional[Workspace] = None, stream=None):
    """nvfp4_quantize_fp8: returns (E4M3 bytes uint8 [rows, K], s_t float32 [rows])."""
    _require(x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1,
             "quantize_fp8: x must be a 2-D BF16 tensor with unit column stride")
    rows, K = x.shape
    a = torch.empty((rows, K), dtype=torch.uint8, device=x.device)
    st = torch.empty(rows, dtype=torch.float32, device=x.device)
    ws = _ws(ws, workspace_size(OP_QUANTIZE_FP8, rows, 0, K), x.device)
    _check(lib().nvfp4_quantize_fp8(_ptr(x), rows, K, x.stride(0), _ptr(a), _ptr(st), ws.ptr, ws.nbytes,
                                    _stream(stream)), "nvfp4_quantize_fp8")
    return a, st


def _out(y, M, N, out_dtype, device):
    """The output tensor of a [M, N] product: allocated when y is None, else
    checked before any pointer reaches the C ABI (a wrong dtype or shape would
    make the kernel write past the buffer): a 2-D CUDA tensor of out_dtype,
    at least [M, N], unit column stride."""
    _require(out_dtype in (OUT_BF16, OUT_FP32), "out_dtype must be OUT_BF16 or OUT_FP32")
    dt = torch.bfloat16 if out_dtype == OUT_BF16 else torch.float32
    if y is None:
        return torch.empty((M, N), dtype=dt, device=device)
    _require(y.is_cuda and y.dim() == 2, "output y must be a 2-D CUDA tensor")
    _require(y.dtype == dt, f"output y must be {dt} for out_dtype {out_dtype}")
    _require(y.shape[0] >= M and y.shape[1] >= N, f"output y {tuple(y.shape)} is smaller than [{M}, {N}]")
    _require(y.stride(1) == 1, "output y must have unit column stride")
    return y


def gemm(w: NVFP4Tensor, x: Optional[torch.Tensor] = None, a_q: Optional[NVFP4Tensor] = None,
         out_dtype: int = OUT_BF16, policy: int = POLICY_AUTO, sensitive: int = 0,
         y: Optional[torch.Tensor] = None, ws: Optional[Workspace] = None, stream=None) -> torch.Tensor:
    """nvfp4_gemm: Y = X W^T for one layer under the precision policy."""
    N, K = w.rows, w.K
    M = x.shape[0] if x is not None else a_q.rows
    device = w.codes.device
    y = _out(y, M, N, out_dtype, device)
    if M == 0:
        return y
    ws = _ws(ws, workspace_size(OP_GEMM, M, N, K), device)
    wd = w.desc()
    ad = a_q.desc() if a_q is not None else None
    _check(lib().nvfp4_gemm(_ptr(x), x.stride(0) if x is not None else 0,
                            ctypes.byref(ad) if ad is not None else None, ctypes.byref(wd), _ptr(y),
                            y.stride(0), out_dtype, M, policy, int(bool(sensitive)), ws.ptr, ws.nbytes,
                            _stream(stream)), "nvfp4_gemm")
    return y


def gemm_nvfp4_out(w: NVFP4Tensor, s_y: torch.Tensor, x: Optional[torch.Tensor] = None,
                   a_q: Optional[NVFP4Tensor] = None, y_amax: Optional[torch.Tensor] = None,
                   out: Optional[NVFP4Tensor] = None, ws: Optional[Workspace] = None,
                   stream=None) -> NVFP4Tensor:
    """nvfp4_gemm_nvfp4_out: the W4A4 product encoded straight to NVFP4 under
    the device tensor scale s_y (float32 [1]); y_amax (float32 [1], optional)
    accumulates max|Y|."""
    N, K = w.rows, w.K
    M = x.shape[0] if x is not None else a_q.rows
    device = w.codes.device
    _require(s_y.dtype == torch.float32 and s_y.numel() == 1 and s_y.device == device,
             "gemm_nvfp4_out: s_y must be one FP32 value on the GEMM's device")
    _require(y_amax is None or (y_amax.dtype == torch.float32 and y_amax.device == device),
             "gemm_nvfp4_out: y_amax must be FP32 on the GEMM's device")
    if out is None:
        out = empty_nvfp4(M, N, SCALE_TENSOR_FP32, LAYOUT_MMA_TILED, device)
    out.second = s_y
    if M == 0:
        return out
    ws = _ws(ws, workspace_size(OP_GEMM, M, N, K), device)
    wd, yd = w.desc(), out.desc()
    ad = a_q.desc() if a_q is not None else None
    _check(lib().nvfp4_gemm_nvfp4_out(_ptr(x), x.stride(0) if x is not None else 0,
                                      ctypes.byref(ad) if ad is not None else None, ctypes.byref(wd),
                                      ctypes.byref(yd), _ptr(y_amax), M, ws.ptr, ws.nbytes, _stream(stream)),
           "nvfp4_gemm_nvfp4_out")
    return out


def w4a8_gemm(a_fp8: torch.Tensor, s_t: torch.Tensor, w: NVFP4Tensor, out_dtype: int = OUT_BF16,
              y: Optional[torch.Tensor] = None, ws: Optional[Workspace] = None, stream=None) -> torch.Tensor:
    M = a_fp8.shape[0]
    y = _out(y, M, w.rows, out_dtype, a_fp8.device)
    if M == 0:
        return y
    ws = _ws(ws, workspace_size(OP_W4A8_GEMM, M, w.rows, w.K), a_fp8.device)
    wd = w.desc()
    _check(lib().nvfp4_w4a8_gemm(_ptr(a_fp8), _ptr(s_t), ctypes.byref(wd), _ptr(y), y.stride(0), out_dtype, M,
                                 ws.ptr, ws.nbytes, _stream(stream)), "nvfp4_w4a8_gemm")
    return y


def grouped_gemm(a: NVFP4Tensor, offsets: torch.Tensor, w: NVFP4Tensor, N: int, total_rows: int,
                 row_idx: Optional[torch.Tensor] = None, out_dtype: int = OUT_BF16,
                 policy: int = POLICY_AUTO, sensitive: int = 0, y: Optional[torch.Tensor] = None,
                 ws: Optional[Workspace] = None, stream=None) -> torch.Tensor:
    """nvfp4_grouped_gemm over E = offsets.numel() - 1 experts stacked in w."""
    _require(offsets.dtype == torch.int64 and (row_idx is None or row_idx.dtype == torch.int32),
             "grouped_gemm: offsets must be int64 and row_idx int32")
    E = offsets.numel() - 1
    y = _out(y, total_rows, N, out_dtype, a.codes.device)
    if total_rows == 0:
        return y
    ws = _ws(ws, workspace_size(OP_GROUPED_GEMM, total_rows, N, a.K, E), a.codes.device)
    ad, wd = a.desc(), w.desc()
    _check(lib().nvfp4_grouped_gemm(ctypes.byref(ad), _ptr(row_idx), _ptr(offsets), E, ctypes.byref(wd), N,
                                    _ptr(y), y.stride(0), out_dtype, total_rows, policy, int(bool(sensitive)),
                                    ws.ptr, ws.nbytes, _stream(stream)), "nvfp4_grouped_gemm")
    return y


def gemm_w4a4_noalloc(a_q: NVFP4Tensor, w: NVFP4Tensor, y: torch.Tensor, out_dtype: int = OUT_BF16,
                      stream=None) -> torch.Tensor:
    """nvfp4_gemm_w4a4_noalloc: the W4A4 product for callers that cannot
    allocate; takes no workspace (its scratch is a fixed array inside the
    library, shared by all calls).  y must be provided by the caller."""
    _require(y is not None, "gemm_w4a4_noalloc: y must be provided by the caller")
    y = _out(y, a_q.rows, w.rows, out_dtype, None)
    ad, wd = a_q.desc(), w.desc()
    _check(lib().nvfp4_gemm_w4a4_noalloc(ctypes.byref(ad), ctypes.byref(wd), _ptr(y), y.stride(0), out_dtype,
                                         _stream(stream)), "nvfp4_gemm_w4a4_noalloc")
    return y


def noalloc_status(stream=None) -> int:
    """nvfp4_gemm_w4a4_noalloc_status: OK, ERR_TIMEOUT or ERR_NONFINITE_INPUT
    for the most recent no-allocation calls (waits for the stream; clears)."""
    out = _I32(0)
    _check(lib().nvfp4_gemm_w4a4_noalloc_status(_stream(stream), ctypes.byref(out)), "nvfp4_gemm_w4a4_noalloc_status")
    return out.value


def tma_stream(w: torch.Tensor, grid: int, status: torch.Tensor, stream=None) -> None:
    """nvfp4_diag_tma_stream over a contiguous 2-D uint8 CUDA tensor (rows a
    multiple of 256, row bytes a multiple of 128); status: an int32 CUDA word."""
    _require(w.dtype == torch.uint8 and w.is_cuda and w.dim() == 2 and w.is_contiguous(),
             "tma_stream: w must be a contiguous 2-D uint8 CUDA tensor")
    _require(status.dtype == torch.int32 and status.is_cuda and status.numel() >= 1,
             "tma_stream: status must be an int32 CUDA tensor")
    _check(lib().nvfp4_diag_tma_stream(_ptr(w), w.shape[0], w.shape[1], grid, _ptr(status), _stream(stream)),
           "nvfp4_diag_tma_stream")


def bounds_checked() -> bool:
    """Whether the loaded library is the bounds-checked build."""
    return bool(lib().nvfp4_diag_bounds_checked())


def bounds_record(clear: bool = True):
    """Bounds-checked build: (failures, where, value, limit) of the failed
    address tests since the last clear (synchronises the device); where is
    "unit.cu:line" of the first one, or "" when there was none."""
    n, v, lim = ctypes.c_uint64(0), ctypes.c_uint64(0), ctypes.c_uint64(0)
    buf = ctypes.create_string_buffer(128)
    _check(lib().nvfp4_diag_bounds_record(ctypes.byref(n), buf, len(buf), ctypes.byref(v), ctypes.byref(lim),
                                          1 if clear else 0), "nvfp4_diag_bounds_record")
    return n.value, buf.value.decode(), v.value, lim.value


def bounds_selftest(buf: torch.Tensor, span_bytes: int, stream=None) -> None:
    """nvfp4_diag_bounds_selftest on a uint8 CUDA tensor of at least
    span_bytes + 64 bytes."""
    _require(buf.dtype == torch.uint8 and buf.is_cuda and buf.is_contiguous(),
             "bounds_selftest: buf must be a contiguous uint8 CUDA tensor")
    _check(lib().nvfp4_diag_bounds_selftest(_ptr(buf), buf.numel(), span_bytes, _stream(stream)),
           "nvfp4_diag_bounds_selftest")


def probe_convert(v: torch.Tensor, stream=None):
    """The kernels' own E2M1 / E4M3 conversions applied to float32 values."""
    _require(v.dtype == torch.float32 and v.is_contiguous(), "probe_convert: v must be a contiguous FP32 tensor")
    o2 = torch.empty(v.shape, dtype=torch.uint8, device=v.device)
    o3 = torch.empty(v.shape, dtype=torch.uint8, device=v.device)
    _check(lib().nvfp4_probe_convert(_ptr(v), v.numel(), _ptr(o2), _ptr(o3), _stream(stream)),
           "nvfp4_probe_convert")
    return o2, o3


def version() -> str:
    return lib().nvfp4_version().decode()


def grouped_w4a8_gemm(a_fp8: torch.Tensor, s_t: torch.Tensor, offsets: torch.Tensor, w: NVFP4Tensor, N: int,
                      total_rows: int, row_idx: Optional[torch.Tensor] = None, out_dtype: int = OUT_BF16,
                      y: Optional[torch.Tensor] = None, ws: Optional[Workspace] = None,
                      stream=None) -> torch.Tensor:
    """nvfp4_grouped_w4a8_gemm: grouped W4A8 of FP8 activations [T, K] with
    per-token scales s_t [T]."""
    _require(offsets.dtype == torch.int64 and (row_idx is None or row_idx.dtype == torch.int32),
             "grouped_w4a8_gemm: offsets must be int64 and row_idx int32")
    E = offsets.numel() - 1
    y = _out(y, total_rows, N, out_dtype, a_fp8.device)
    if total_rows == 0:
        return y
    ws = _ws(ws, workspace_size(OP_GROUPED_GEMM, total_rows, N, w.K, E), a_fp8.device)
    wd = w.desc()
    _check(lib().nvfp4_grouped_w4a8_gemm(_ptr(a_fp8), _ptr(s_t), a_fp8.shape[0], _ptr(row_idx), _ptr(offsets), E,
                                         ctypes.byref(wd), N, _ptr(y), y.stride(0), out_dtype, total_rows, ws.ptr,
                                         ws.nbytes, _stream(stream)), "nvfp4_grouped_w4a8_gemm")
    return y


def grouped_gemm_x(x: torch.Tensor, offsets: torch.Tensor, w: NVFP4Tensor, N: int, total_rows: int,
                   row_idx: Optional[torch.Tensor] = None, out_dtype: int = OUT_BF16, policy: int = POLICY_AUTO,
                   sensitive: int = 0, y: Optional[torch.Tensor] = None, ws: Optional[Workspace] = None,
                   stream=None) -> torch.Tensor:
    """nvfp4_grouped_gemm_x: grouped GEMM of BF16 activations under the
    precision policy (W4A4 or W4A8 route)."""
    _require(x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1,
             "grouped_gemm_x: x must be a 2-D BF16 tensor with unit column stride")
    _require(offsets.dtype == torch.int64 and (row_idx is None or row_idx.dtype == torch.int32),
             "grouped_gemm_x: offsets must be int64 and row_idx int32")
    E = offsets.numel() - 1
    y = _out(y, total_rows, N, out_dtype, x.device)
    if total_rows == 0:
        return y
    ws = _ws(ws, workspace_size(OP_GROUPED_GEMM_X, x.shape[0], N, w.K, E), x.device)
    wd = w.desc()
    _check(lib().nvfp4_grouped_gemm_x(_ptr(x), x.stride(0), x.shape[0], _ptr(row_idx), _ptr(offsets), E,
                                      ctypes.byref(wd), N, _ptr(y), y.stride(0), out_dtype, total_rows, policy,
                                      int(bool(sensitive)), ws.ptr, ws.nbytes, _stream(stream)),
           "nvfp4_grouped_gemm_x")
    return y


def moe_up_swiglu(a: NVFP4Tensor, offsets: torch.Tensor, w_gate_up: NVFP4Tensor, I: int, total_rows: int,
                  row_idx: Optional[torch.Tensor] = None, out_dtype: int = OUT_BF16,
                  h: Optional[torch.Tensor] = None, s_h: Optional[torch.Tensor] = None,
                  h_amax: Optional[torch.Tensor] = None, h_q: Optional[NVFP4Tensor] = None,
                  ws: Optional[Workspace] = None, stream=None):
    """nvfp4_moe_up_swiglu: SiLU(gate) * up of the routed rows.  With s_h
    (float32 [1] device tensor scale) the output is NVFP4 (returned as an
    NVFP4Tensor); otherwise a BF16/FP32 [total_rows, I] tensor."""
    _require(offsets.dtype == torch.int64 and (row_idx is None or row_idx.dtype == torch.int32),
             "moe_up_swiglu: offsets must be int64 and row_idx int32")
    E = offsets.numel() - 1
    dev = a.codes.device
    hd = None
    if s_h is not None:
        if h_q is None:
            h_q = empty_nvfp4(total_rows, I, device=dev)
        h_q.second = s_h
        result = h_q
    else:
        h = _out(h, total_rows, I, out_dtype, dev)
        result = h
    if total_rows == 0:
        return result
    ws = _ws(ws, workspace_size(OP_GROUPED_GEMM, total_rows, 2 * I, a.K, E), dev)
    ad, wd = a.desc(), w_gate_up.desc()
    if s_h is not None:
        hd = h_q.desc()
    _check(lib().nvfp4_moe_up_swiglu(ctypes.byref(ad), _ptr(row_idx), _ptr(offsets), E, ctypes.byref(wd), I,
                                     _ptr(h), h.stride(0) if h is not None else 0, out_dtype,
                                     ctypes.byref(hd) if hd is not None else None, _ptr(h_amax), total_rows,
                                     ws.ptr, ws.nbytes, _stream(stream)), "nvfp4_moe_up_swiglu")
    return result


def moe_down_combine(h: NVFP4Tensor, offsets: torch.Tensor, w_down: NVFP4Tensor, N: int,
                     token_idx: torch.Tensor, gate_w: torch.Tensor, y: torch.Tensor,
                     ws: Optional[Workspace] = None, stream=None) -> torch.Tensor:
    """nvfp4_moe_down_combine: y[token_idx[j]] += gate_w[j] * (h[j] W_e^T) into
    the FP32 [T, N] tensor y (which holds zeros or the residual)."""
    _require(offsets.dtype == torch.int64 and token_idx.dtype == torch.int32 and gate_w.dtype == torch.float32,
             "moe_down_combine: offsets must be int64, token_idx int32 and gate_w FP32")
    _require(y.dtype == torch.float32 and y.stride(1) == 1, "moe_down_combine: y must be FP32 with unit column stride")
    E = offsets.numel() - 1
    R = h.rows
    ws = _ws(ws, workspace_size(OP_GROUPED_GEMM, R, N, h.K, E), h.codes.device)
    hd, wd = h.desc(), w_down.desc()
    _check(lib().nvfp4_moe_down_combine(ctypes.byref(hd), _ptr(offsets), E, ctypes.byref(wd), N,
                                        _ptr(token_idx), _ptr(gate_w), _ptr(y), y.stride(0), y.shape[0], R,
                                        ws.ptr, ws.nbytes, _stream(stream)), "nvfp4_moe_down_combine")
    return y


# ---- NVFP4 paged KV cache --------------------------------------------------------------

KV_PAGE = 64
KV_HEAD_DIM = 128
KV_NVFP4, KV_FP8 = 0, 1


KV_PAGE_BYTES = {KV_NVFP4: 9216, KV_FP8: 16384}


@dataclasses.dataclass
class KvCache:
    """Device paged KV cache (layouts in include/nvfp4.h): `pages` uint8
    [num_pages, num_kv_heads, page block], one contiguous block per page and
    KV head (NVFP4: key codes, key scales, value codes dim-major, value
    scales; FP8: two 32-token halves of keys then dim-major values); static
    tensor scales k_scale / v_scale (float32 [1])."""
    pages: torch.Tensor
    k_scale: torch.Tensor
    v_scale: torch.Tensor
    fmt: int = KV_NVFP4

    @property
    def num_pages(self) -> int:
        return self.pages.shape[0]

    @property
    def num_kv_heads(self) -> int:
        return self.pages.shape[1]

    @staticmethod
    def empty(num_pages: int, num_kv_heads: int, k_scale: torch.Tensor, v_scale: torch.Tensor,
              device="cuda", fmt: int = KV_NVFP4) -> "KvCache":
        pages = torch.zeros((num_pages, num_kv_heads, KV_PAGE_BYTES[fmt]), dtype=torch.uint8, device=device)
        return KvCache(pages, k_scale, v_scale, fmt)

    def desc(self) -> KvCacheDesc:
        _require(self.pages.is_contiguous() and self.pages.shape[2] == KV_PAGE_BYTES[self.fmt],
                 "desc: pages must be contiguous page blocks of the cache format's size")
        return KvCacheDesc(self.pages.data_ptr(), self.k_scale.data_ptr(), self.v_scale.data_ptr(),
                           self.num_pages, self.num_kv_heads, KV_HEAD_DIM, KV_PAGE, self.fmt)


def kv_append(cache: KvCache, k_new: torch.Tensor, v_new: torch.Tensor, positions: torch.Tensor,
              block_table: torch.Tensor, stream=None):
    """nvfp4_kv_append: one new token per sequence (BF16 [B][H_kv][128])."""
    _require(k_new.dtype == torch.bfloat16 and v_new.dtype == torch.bfloat16 and k_new.is_contiguous(),
             "kv_append: k_new and v_new must be BF16, k_new contiguous")
    _require(positions.dtype == torch.int32 and block_table.dtype == torch.int32 and block_table.is_contiguous(),
             "kv_append: positions and block_table must be int32, block_table contiguous")
    B = k_new.shape[0]
    d = cache.desc()
    _check(lib().nvfp4_kv_append(ctypes.byref(d), _ptr(k_new), _ptr(v_new.contiguous()), _ptr(positions),
                                 _ptr(block_table), block_table.shape[1], B, _stream(stream)), "nvfp4_kv_append")


def kv_decode_attention(cache: KvCache, q: torch.Tensor, ctx_lens: torch.Tensor, block_table: torch.Tensor,
                        max_ctx: int, sm_scale: float, out_dtype: int = OUT_BF16,
                        out: Optional[torch.Tensor] = None, ws: Optional[Workspace] = None,
                        stream=None) -> torch.Tensor:
    """nvfp4_kv_decode_attention: q BF16 [B][H][128] -> out [B][H][128]."""
    _require(q.dtype == torch.bfloat16 and q.is_contiguous() and q.shape[2] == KV_HEAD_DIM,
             "kv_decode_attention: q must be contiguous BF16 [B][H][128]")
    _require(ctx_lens.dtype == torch.int32 and block_table.dtype == torch.int32 and block_table.is_contiguous(),
             "kv_decode_attention: ctx_lens and block_table must be int32, block_table contiguous")
    B, H, D = q.shape
    if out is None:
        out = torch.empty((B, H, D), dtype=torch.bfloat16 if out_dtype == OUT_BF16 else torch.float32,
                          device=q.device)
    ws = _ws(ws, workspace_size(OP_KV_DECODE, B, H, max_ctx, cache.num_kv_heads), q.device)
    d = cache.desc()
    _check(lib().nvfp4_kv_decode_attention(ctypes.byref(d), _ptr(q), H, _ptr(ctx_lens), _ptr(block_table),
                                           block_table.shape[1], B, max_ctx, float(sm_scale), _ptr(out),
                                           out_dtype, ws.ptr, ws.nbytes, _stream(stream)),
           "nvfp4_kv_decode_attention")
    return out
