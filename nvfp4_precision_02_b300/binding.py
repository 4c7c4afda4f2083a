"""Python binding of libnvfp4.so: argument marshalling only.

Every function here allocates outputs with PyTorch (device memory), passes raw
pointers and sizes to the C entry point of the same name, and raises
``Nvfp4Error`` on a non-OK status.  No arithmetic of the method happens in
Python.  The library must exist (``python -m nvfp4_precision_02_b300.build``);
there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libnvfp4.so")

RNE, SR = 0, 1
OUT_BF16, OUT_FP32 = 0, 1
DEV_TIMEOUT, DEV_BAD_OFFSETS = 1, 2
MAX_GROUPS = 1024

STATIC_MAX_BATCH = 4096

STATUS = {0: "NVFP4_OK", 1: "NVFP4_ERR_NULL", 2: "NVFP4_ERR_SHAPE", 3: "NVFP4_ERR_ALIGN",
          4: "NVFP4_ERR_DEVICE", 5: "NVFP4_ERR_CUDA", 6: "NVFP4_ERR_TIMEOUT", 7: "NVFP4_ERR_LIMIT"}

EXPORTS = ["nvfp4_sf_bytes", "nvfp4_sf_bytes_grouped", "nvfp4_sf_offset", "nvfp4_amax", "nvfp4_quantize_1d",
           "nvfp4_quantize_1d_grouped", "nvfp4_quantize_2d", "nvfp4_quantize_2d_fused_workspace",
           "nvfp4_quantize_2d_fused", "nvfp4_quantize_2d_fused_static", "nvfp4_rht_amax",
           "nvfp4_rht_quantize", "nvfp4_dual_amax", "nvfp4_dual_sr_quantize", "nvfp4_count_zero_codes",
           "nvfp4_quantize_1d_mse",
           "nvfp4_sr_fp16", "nvfp4_group_k_capacity", "nvfp4_rht_quantize_grouped", "nvfp4_gemm",
           "nvfp4_grouped_gemm", "nvfp4_grouped_gemm_k", "nvfp4_status_string", "nvfp4_last_error",
           "nvfp4_device_status", "nvfp4_launch_count", "nvfp4_debug_inject", "nvfp4_debug_wait_timeout"]


class Nvfp4Error(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


class CTensor(ctypes.Structure):
    """Mirror of nvfp4_tensor."""
    _fields_ = [("codes", ctypes.c_void_p), ("sf", ctypes.c_void_p), ("amax", ctypes.c_void_p),
                ("rows", ctypes.c_int64), ("cols", ctypes.c_int64)]


_lib = None


def lib():
    """Load libnvfp4.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m nvfp4_precision_02_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        P, i64, i32, u64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint64
        st = ctypes.c_int
        TP = ctypes.POINTER(CTensor)
        sig = {
            "nvfp4_sf_bytes": (ctypes.c_size_t, [i64, i64]),
            "nvfp4_sf_bytes_grouped": (ctypes.c_size_t, [i64, i64, i32]),
            "nvfp4_sf_offset": (i64, [i64, i64, i64]),
            "nvfp4_amax": (st, [P, i64, i64, i64, i64, P, P]),
            "nvfp4_quantize_1d": (st, [P, i64, i64, i64, ctypes.c_int, u64, P, TP, P]),
            "nvfp4_quantize_1d_grouped": (st, [P, i64, i64, i64, P, i32, ctypes.c_int, u64, P, TP, P]),
            "nvfp4_quantize_2d": (st, [P, i64, i64, i64, i64, P, TP, TP, P, P]),
            "nvfp4_quantize_2d_fused_workspace": (ctypes.c_size_t, [i64]),
            "nvfp4_quantize_2d_fused": (st, [P, i64, i64, i64, i64, P, ctypes.c_size_t, TP, P, P]),
            "nvfp4_quantize_2d_fused_static": (st, [P, i64, i64, i64, i64, TP, P, P]),
            "nvfp4_rht_amax": (st, [P, i64, i64, i64, ctypes.c_uint16, P, P]),
            "nvfp4_rht_quantize": (st, [P, i64, i64, i64, ctypes.c_uint16, ctypes.c_int, u64, P, TP, P]),
            "nvfp4_gemm": (st, [TP, TP, P, i64, ctypes.c_int, P, P]),
            "nvfp4_grouped_gemm": (st, [TP, P, i32, TP, i64, P, i64, ctypes.c_int, P, P]),
            "nvfp4_group_k_capacity": (i64, [i64, i32]),
            "nvfp4_sr_fp16": (st, [P, i64, ctypes.c_uint64, P, P]),
            "nvfp4_quantize_1d_mse": (st, [P, i64, i64, i64, P, TP, P]),
            "nvfp4_dual_amax": (st, [P, i64, i64, i64, ctypes.c_uint16, P, P, P]),
            "nvfp4_count_zero_codes": (st, [TP, P, P]),
            "nvfp4_dual_sr_quantize": (st, [P, i64, i64, i64, ctypes.c_uint16, u64, u64, P, P, TP, TP, P, P]),
            "nvfp4_rht_quantize_grouped": (st, [P, i64, i64, i64, P, i32, i64, ctypes.c_uint16, ctypes.c_int,
                                                ctypes.c_uint64, P, TP, P]),
            "nvfp4_grouped_gemm_k": (st, [TP, TP, P, i32, P, i64, ctypes.c_int, P, P]),
            "nvfp4_status_string": (ctypes.c_char_p, [st]),
            "nvfp4_last_error": (ctypes.c_char_p, []),
            "nvfp4_device_status": (st, [ctypes.POINTER(ctypes.c_int32)]),
            "nvfp4_launch_count": (ctypes.c_uint64, []),
            "nvfp4_debug_inject": (None, [st]),
            "nvfp4_debug_wait_timeout": (st, [i64, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _check(status: int):
    if status != 0:
        raise Nvfp4Error(status, lib().nvfp4_last_error().decode())


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _rows2d(x: torch.Tensor):
    assert x.dim() == 2 and x.dtype == torch.bfloat16 and x.stride(1) == 1, "bf16 [rows, cols] with unit column stride"
    return x.shape[0], x.shape[1], x.stride(0)


@dataclass
class QTensor:
    """A quantised operand: packed E2M1 codes, swizzled E4M3 scales, FP32 amax."""
    codes: torch.Tensor      # uint8 [rows, cols/2] (or [batch, rows, cols/2])
    sf: torch.Tensor         # uint8, swizzled
    amax: torch.Tensor       # float32 [1] / [groups] / [batch]
    rows: int
    cols: int

    def c(self) -> CTensor:
        return CTensor(self.codes.data_ptr(), self.sf.data_ptr(), self.amax.data_ptr(), self.rows, self.cols)


# ------------------------------------------------------------------ layout
def sf_bytes(rows: int, cols: int) -> int:
    return lib().nvfp4_sf_bytes(rows, cols)


def sf_bytes_grouped(rows: int, cols: int, groups: int) -> int:
    return lib().nvfp4_sf_bytes_grouped(rows, cols, groups)


def sf_offset(r: int, c: int, cols: int) -> int:
    return lib().nvfp4_sf_offset(r, c, cols)


def empty_qtensor(rows: int, cols: int, device, batch: int = 1, n_amax: int = 1,
                  sf_size: Optional[int] = None) -> QTensor:
    shape = (rows, cols // 2) if batch == 1 else (batch, rows, cols // 2)
    return QTensor(torch.empty(shape, dtype=torch.uint8, device=device),
                   torch.empty(sf_size if sf_size is not None else batch * sf_bytes(rows, cols),
                               dtype=torch.uint8, device=device),
                   torch.empty(n_amax, dtype=torch.float32, device=device), rows, cols)


# ------------------------------------------------------------------ entry points
def amax(x: torch.Tensor, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """x: bf16 [rows, cols] or [batch, rows, cols] -> float32 [batch]."""
    if x.dim() == 2:
        x3 = x.unsqueeze(0)
    else:
        x3 = x
    batch, rows, cols = x3.shape
    assert x3.stride(2) == 1 and (batch == 1 or x3.stride(0) == rows * x3.stride(1))
    out = torch.empty(batch, dtype=torch.float32, device=x.device) if out is None else out
    _check(lib().nvfp4_amax(_ptr(x3), batch, rows, cols, x3.stride(1), _ptr(out), _stream(stream)))
    return out


def quantize_1d(x: torch.Tensor, mode: int = RNE, seed: int = 0, amax_in: Optional[torch.Tensor] = None,
                out: Optional[QTensor] = None, stream=None) -> QTensor:
    rows, cols, ld = _rows2d(x)
    out = empty_qtensor(rows, cols, x.device) if out is None else out
    co = out.c()
    _check(lib().nvfp4_quantize_1d(_ptr(x), rows, cols, ld, mode, seed, _ptr(amax_in), ctypes.byref(co),
                                   _stream(stream)))
    return out


def quantize_1d_grouped(x: torch.Tensor, offsets: torch.Tensor, mode: int = RNE, seed: int = 0,
                        amax_in: Optional[torch.Tensor] = None, out: Optional[QTensor] = None,
                        stream=None) -> QTensor:
    rows, cols, ld = _rows2d(x)
    assert offsets.dtype == torch.int64 and offsets.is_cuda
    groups = offsets.numel() - 1
    out = (empty_qtensor(rows, cols, x.device, n_amax=groups, sf_size=sf_bytes_grouped(rows, cols, groups))
           if out is None else out)
    co = out.c()
    _check(lib().nvfp4_quantize_1d_grouped(_ptr(x), rows, cols, ld, _ptr(offsets), groups, mode, seed,
                                           _ptr(amax_in), ctypes.byref(co), _stream(stream)))
    return out


def quantize_2d(w: torch.Tensor, want_t: bool = True, want_tile_sf: bool = False,
                amax_in: Optional[torch.Tensor] = None, out: Optional[QTensor] = None,
                out_t: Optional[QTensor] = None, stream=None):
    """w: bf16 [rows, cols] or [batch, rows, cols] -> (W, W^T or None, tile_sf or None)."""
    w3 = w.unsqueeze(0) if w.dim() == 2 else w
    batch, rows, cols = w3.shape
    assert w3.dtype == torch.bfloat16 and w3.stride(2) == 1 and (batch == 1 or w3.stride(0) == rows * w3.stride(1))
    dev = w.device
    if out is None:
        out = empty_qtensor(rows, cols, dev, batch=batch, n_amax=batch)
    if want_t and out_t is None:
        out_t = empty_qtensor(cols, rows, dev, batch=batch, n_amax=1)
    tile = torch.empty(batch, rows // 16, cols // 16, dtype=torch.uint8, device=dev) if want_tile_sf else None
    co = out.c()
    ct = out_t.c() if want_t else None
    _check(lib().nvfp4_quantize_2d(_ptr(w3), batch, rows, cols, w3.stride(1), _ptr(amax_in), ctypes.byref(co),
                                   ctypes.byref(ct) if ct is not None else None, _ptr(tile), _stream(stream)))
    if want_t:
        out_t.amax = out.amax
    return out, (out_t if want_t else None), tile


def quantize_2d_fused_workspace(batch: int) -> int:
    return lib().nvfp4_quantize_2d_fused_workspace(batch)


def quantize_2d_fused(w: torch.Tensor, want_tile_sf: bool = False, workspace: Optional[torch.Tensor] = None,
                      out: Optional[QTensor] = None, stream=None):
    """Per-entry amax and 2D quantisation (W only) in one HBM pass, for
    entries that fit in L2.  w: bf16 [rows, cols] or [batch, rows, cols]
    -> (W, tile_sf or None)."""
    w3 = w.unsqueeze(0) if w.dim() == 2 else w
    batch, rows, cols = w3.shape
    assert w3.dtype == torch.bfloat16 and w3.stride(2) == 1 and (batch == 1 or w3.stride(0) == rows * w3.stride(1))
    dev = w.device
    if out is None:
        out = empty_qtensor(rows, cols, dev, batch=batch, n_amax=batch)
    if workspace is None:
        workspace = torch.empty(quantize_2d_fused_workspace(batch), dtype=torch.uint8, device=dev)
    tile = torch.empty(batch, rows // 16, cols // 16, dtype=torch.uint8, device=dev) if want_tile_sf else None
    co = out.c()
    _check(lib().nvfp4_quantize_2d_fused(_ptr(w3), batch, rows, cols, w3.stride(1), _ptr(workspace),
                                         workspace.numel() * workspace.element_size(), ctypes.byref(co),
                                         _ptr(tile), _stream(stream)))
    return out, tile


def quantize_2d_fused_static(w: torch.Tensor, want_tile_sf: bool = False, out: Optional[QTensor] = None,
                             stream=None):
    """quantize_2d_fused with the library's own fixed scratch instead of a
    workspace (for callers that cannot allocate at the call); at most
    STATIC_MAX_BATCH entries, and calls must not overlap on the GPU."""
    w3 = w.unsqueeze(0) if w.dim() == 2 else w
    batch, rows, cols = w3.shape
    assert w3.dtype == torch.bfloat16 and w3.stride(2) == 1 and (batch == 1 or w3.stride(0) == rows * w3.stride(1))
    dev = w.device
    if out is None:
        out = empty_qtensor(rows, cols, dev, batch=batch, n_amax=batch)
    tile = torch.empty(batch, rows // 16, cols // 16, dtype=torch.uint8, device=dev) if want_tile_sf else None
    co = out.c()
    _check(lib().nvfp4_quantize_2d_fused_static(_ptr(w3), batch, rows, cols, w3.stride(1), ctypes.byref(co),
                                                _ptr(tile), _stream(stream)))
    return out, tile


def rht_amax(x: torch.Tensor, sign_mask: int, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    tokens, cols, ld = _rows2d(x)
    out = torch.empty(1, dtype=torch.float32, device=x.device) if out is None else out
    _check(lib().nvfp4_rht_amax(_ptr(x), tokens, cols, ld, sign_mask, _ptr(out), _stream(stream)))
    return out


def rht_quantize(x: torch.Tensor, sign_mask: int, mode: int = RNE, seed: int = 0,
                 amax_in: Optional[torch.Tensor] = None, out: Optional[QTensor] = None, stream=None) -> QTensor:
    """x: bf16 [tokens, cols] -> transposed operand [cols, tokens]."""
    tokens, cols, ld = _rows2d(x)
    out = empty_qtensor(cols, tokens, x.device) if out is None else out
    co = out.c()
    _check(lib().nvfp4_rht_quantize(_ptr(x), tokens, cols, ld, sign_mask, mode, seed, _ptr(amax_in),
                                    ctypes.byref(co), _stream(stream)))
    return out


def dual_amax(x: torch.Tensor, sign_mask: int, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """x: bf16 [tokens, cols] -> float32 [2]: (max |x|, max |RHT(x)|) from one read."""
    tokens, cols, ld = _rows2d(x)
    out = torch.empty(2, dtype=torch.float32, device=x.device) if out is None else out
    assert out.dtype == torch.float32 and out.numel() >= 2
    _check(lib().nvfp4_dual_amax(_ptr(x), tokens, cols, ld, sign_mask, _ptr(out), ctypes.c_void_p(out.data_ptr() + 4),
                                 _stream(stream)))
    return out


def dual_sr_quantize(dy: torch.Tensor, sign_mask: int, seed_row: int, seed_rht: int, amax: torch.Tensor,
                     out_row: Optional[QTensor] = None, out_t: Optional[QTensor] = None,
                     zero_count: Optional[torch.Tensor] = None, stream=None):
    """Both stochastically rounded operands of a gradient from one read:
    dy bf16 [tokens, cols], amax float32 [2] = (max |dy|, max |RHT(dy)|) as
    dual_amax gives -> (row operand [tokens, cols] as quantize_1d(SR,
    seed_row), RHT operand [cols, tokens] as rht_quantize(SR, seed_rht));
    zero_count (int64 [1], optional) receives the row operand's zero-code
    count."""
    tokens, cols, ld = _rows2d(dy)
    dev = dy.device
    out_row = empty_qtensor(tokens, cols, dev) if out_row is None else out_row
    out_t = empty_qtensor(cols, tokens, dev) if out_t is None else out_t
    assert amax.dtype == torch.float32 and amax.numel() >= 2
    cr, ct = out_row.c(), out_t.c()
    _check(lib().nvfp4_dual_sr_quantize(_ptr(dy), tokens, cols, ld, sign_mask, seed_row, seed_rht, _ptr(amax),
                                        ctypes.c_void_p(amax.data_ptr() + 4), ctypes.byref(cr), ctypes.byref(ct),
                                        _ptr(zero_count), _stream(stream)))
    return out_row, out_t


def count_zero_codes(q: QTensor, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Number of zero-magnitude codes of a quantised tensor (int64 [1], on the device)."""
    out = torch.empty(1, dtype=torch.int64, device=q.codes.device) if out is None else out
    cq = q.c()
    _check(lib().nvfp4_count_zero_codes(ctypes.byref(cq), _ptr(out), _stream(stream)))
    return out


def quantize_1d_mse(x: torch.Tensor, amax_in: Optional[torch.Tensor] = None, out: Optional[QTensor] = None,
                    stream=None) -> QTensor:
    """1x16 RNE quantisation with block scales chosen by minimum squared error (PTQ weights)."""
    rows, cols, ld = _rows2d(x)
    out = empty_qtensor(rows, cols, x.device) if out is None else out
    co = out.c()
    _check(lib().nvfp4_quantize_1d_mse(_ptr(x), rows, cols, ld, _ptr(amax_in), ctypes.byref(co), _stream(stream)))
    return out


def sr_fp16(x: torch.Tensor, seed: int, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """FP32 tensor -> FP16 tensor with stochastic rounding (Philox-5 word of each element)."""
    assert x.dtype == torch.float32 and x.is_cuda and x.is_contiguous()
    if out is None:
        out = torch.empty(x.shape, dtype=torch.float16, device=x.device)
    _check(lib().nvfp4_sr_fp16(_ptr(x), x.numel(), seed, _ptr(out), _stream(stream)))
    return out


def group_k_capacity(rows: int, groups: int) -> int:
    """Columns of an expert-segmented RHT operand for any split of `rows` tokens."""
    return lib().nvfp4_group_k_capacity(rows, groups)


def rht_quantize_grouped(x: torch.Tensor, offsets: torch.Tensor, sign_mask: int, mode: int = RNE, seed: int = 0,
                         kt: Optional[int] = None, amax_in: Optional[torch.Tensor] = None,
                         out: Optional[QTensor] = None, stream=None) -> QTensor:
    """x: bf16 [rows, cols], expert-sorted -> transposed operand [cols, kt] with every
    expert's tokens zero-padded to a multiple of 64 (amax per expert)."""
    rows, cols, ld = _rows2d(x)
    assert offsets.dtype == torch.int64 and offsets.is_cuda
    groups = offsets.numel() - 1
    if kt is None:
        kt = group_k_capacity(rows, groups) if out is None else out.cols
    out = empty_qtensor(cols, kt, x.device, n_amax=groups) if out is None else out
    co = out.c()
    _check(lib().nvfp4_rht_quantize_grouped(_ptr(x), rows, cols, ld, _ptr(offsets), groups, kt, sign_mask, mode,
                                            seed, _ptr(amax_in), ctypes.byref(co), _stream(stream)))
    return out


def grouped_gemm_k(a: QTensor, b: QTensor, offsets: torch.Tensor, out_dtype: int = OUT_FP32,
                   out: Optional[torch.Tensor] = None, stream=None,
                   c_amax: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Groups along K (expert wgrad): C[g*M:(g+1)*M] = alpha_g * A[:, slice_g] . B[:, slice_g]^T
    for a [M, KT], b [N, KT] from rht_quantize_grouped with the same offsets."""
    groups = offsets.numel() - 1
    if out is None:
        out = torch.empty(groups * a.rows, b.rows, dtype=torch.float32 if out_dtype == OUT_FP32 else torch.bfloat16,
                          device=a.codes.device)
    ca, cb = a.c(), b.c()
    _check(lib().nvfp4_grouped_gemm_k(ctypes.byref(ca), ctypes.byref(cb), _ptr(offsets), groups, _ptr(out),
                                      out.stride(0), out_dtype, _ptr(c_amax), _stream(stream)))
    return out


def gemm(a: QTensor, b: QTensor, out_dtype: int = OUT_BF16, out: Optional[torch.Tensor] = None,
         stream=None, c_amax: Optional[torch.Tensor] = None) -> torch.Tensor:
    """C[M, N] = alpha * A[M, K] . B[N, K]^T (both quantised, K-major); c_amax
    (float32 [1], optional) receives max |C|."""
    M, N = a.rows, b.rows
    if out is None:
        out = torch.empty(M, N, dtype=torch.float32 if out_dtype == OUT_FP32 else torch.bfloat16,
                          device=a.codes.device)
    ca, cb = a.c(), b.c()
    _check(lib().nvfp4_gemm(ctypes.byref(ca), ctypes.byref(cb), _ptr(out), out.stride(0), out_dtype,
                            _ptr(c_amax), _stream(stream)))
    return out


def grouped_gemm(a: QTensor, offsets: torch.Tensor, b: QTensor, n: int, out_dtype: int = OUT_BF16,
                 out: Optional[torch.Tensor] = None, stream=None,
                 c_amax: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Per expert g: C[o_g:o_{g+1}] = alpha_g * A_g . W_g^T; b is the batched [E, n, K] weight;
    c_amax (float32 [groups], optional) receives each group's max |C|."""
    groups = offsets.numel() - 1
    if out is None:
        out = torch.empty(a.rows, n, dtype=torch.float32 if out_dtype == OUT_FP32 else torch.bfloat16,
                          device=a.codes.device)
    ca, cb = a.c(), b.c()
    _check(lib().nvfp4_grouped_gemm(ctypes.byref(ca), _ptr(offsets), groups, ctypes.byref(cb), n, _ptr(out),
                                    out.stride(0), out_dtype, _ptr(c_amax), _stream(stream)))
    return out


def device_status() -> int:
    flags = ctypes.c_int32(0)
    st = lib().nvfp4_device_status(ctypes.byref(flags))
    if st not in (0, 6):
        _check(st)
    return int(flags.value)


def launch_count() -> int:
    return int(lib().nvfp4_launch_count())


def debug_inject(status: int):
    lib().nvfp4_debug_inject(status)


def debug_wait_timeout(timeout_ns: int, stream=None):
    _check(lib().nvfp4_debug_wait_timeout(timeout_ns, _stream(stream)))
