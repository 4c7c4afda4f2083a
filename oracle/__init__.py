"""CPU oracle for the NVFP4 training linear-layer path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The oracle is
plain C (``oracle.c``) compiled with ``gcc -ffp-contract=off`` and called
through ctypes; it shares no code with the CUDA library and never imports it.

Every function here only marshals numpy arrays into the C routines; the
arithmetic lives in ``oracle.c`` (see its header for the sources and the
readings taken where the pages are silent).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

RNE = 0
SR = 1


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (in-tree)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
               "-fopenmp", "-shared", "-fPIC", "-o", _LIB + ".tmp", _SRC, "-lm"]
        subprocess.check_call(cmd)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i64, u64, i32, u32, f32, f64 = (ctypes.c_int64, ctypes.c_uint64, ctypes.c_int32,
                                        ctypes.c_uint32, ctypes.c_float, ctypes.c_double)
        sig = {
            "oracle_e2m1_value": (f64, [ctypes.c_int]),
            "oracle_e4m3_value": (f64, [ctypes.c_int]),
            "oracle_e4m3_encode": (ctypes.c_uint8, [f32]),
            "oracle_e2m1_rne": (ctypes.c_int, [f32]),
            "oracle_e2m1_sr": (ctypes.c_int, [f32, u32]),
            "oracle_philox4x32": (None, [P, P, ctypes.c_int, P]),
            "oracle_sr_word": (u32, [u64, u64]),
            "oracle_tensor_scale": (f32, [f32]),
            "oracle_tensor_decode_scale": (f32, [f32]),
            "oracle_block_scale": (ctypes.c_uint8, [f32, f32]),
            "oracle_encode_block": (None, [P, ctypes.c_int, f32, ctypes.c_int, u64, u64, P, P]),
            "oracle_sf_offset": (i64, [i64, i64, i64]),
            "oracle_sf_bytes": (ctypes.c_size_t, [i64, i64]),
            "oracle_sf_bytes_grouped": (ctypes.c_size_t, [i64, i64, i32]),
            "oracle_group_sf_row": (i64, [P, i32]),
            "oracle_amax_bf16": (f32, [P, i64, i64, i64]),
            "oracle_quantize_1d": (None, [P, i64, i64, i64, ctypes.c_int, u64, P, P, P, P]),
            "oracle_quantize_1d_grouped": (None, [P, i64, i64, i64, P, i32, ctypes.c_int, u64,
                                                  P, P, P, P]),
            "oracle_quantize_2d": (None, [P, i64, i64, i64, i64, P, P, P, P, P, P, P]),
            "oracle_rht16": (None, [P, ctypes.c_uint16, P]),
            "oracle_rht_amax": (f32, [P, i64, i64, i64, ctypes.c_uint16]),
            "oracle_rht_quantize": (None, [P, i64, i64, i64, ctypes.c_uint16, ctypes.c_int, u64,
                                           P, P, P, P]),
            "oracle_group_k_offset": (i64, [P, i32]),
            "oracle_fp16_sr": (ctypes.c_uint16, [f32, u32]),
            "oracle_quantize_1d_mse": (None, [P, i64, i64, i64, P, P, P, P]),
            "oracle_sr_fp16": (None, [P, i64, u64, P]),
            "oracle_rht_quantize_grouped": (None, [P, i64, i64, i64, P, i32, i64, ctypes.c_uint16, ctypes.c_int,
                                                   u64, P, P, P, P]),
            "oracle_dequantize_rows": (None, [P, P, i64, i64, f32, P, i64, P]),
            "oracle_gemm": (None, [P, P, i64, i64, i64, P, P]),
            "oracle_num_threads": (ctypes.c_int, []),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _p(a: Optional[np.ndarray]):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _bf16_bits(x) -> np.ndarray:
    """Accept a torch bf16 tensor or a uint16 numpy array of bf16 bits."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16
        return np.ascontiguousarray(x)
    import torch
    assert x.dtype == torch.bfloat16
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


# ----------------------------------------------------------------- scalars
def e2m1_value(code: int) -> float:
    return lib().oracle_e2m1_value(code)


def e4m3_value(byte: int) -> float:
    return lib().oracle_e4m3_value(byte)


def e4m3_encode(x: float) -> int:
    return lib().oracle_e4m3_encode(x)


def e2m1_rne(v: float) -> int:
    return lib().oracle_e2m1_rne(v)


def e2m1_sr(v: float, u: int) -> int:
    return lib().oracle_e2m1_sr(v, u)


def philox4x32(ctr, key, rounds: int = 5):
    c = np.asarray(ctr, dtype=np.uint32)
    k = np.asarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    lib().oracle_philox4x32(_p(c), _p(k), rounds, _p(out))
    return [int(v) for v in out]


def sr_word(seed: int, e: int) -> int:
    return lib().oracle_sr_word(seed, e)


def tensor_scale(amax: float) -> float:
    return lib().oracle_tensor_scale(amax)


def decode_scale(amax: float) -> float:
    return lib().oracle_tensor_decode_scale(amax)


def block_scale(bamax: float, s_enc: float) -> int:
    return lib().oracle_block_scale(bamax, s_enc)


def encode_block(x, s_enc: float, mode: int = RNE, seed: int = 0, e0: int = 0):
    """Encode one block (<=16 float32 values) -> (scale byte, list of 4-bit codes)."""
    xs = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    sf = np.zeros(1, dtype=np.uint8)
    codes = np.zeros(len(xs), dtype=np.uint8)
    lib().oracle_encode_block(_p(xs), len(xs), s_enc, mode, seed, e0, _p(sf), _p(codes))
    return int(sf[0]), [int(c) for c in codes]


def sf_offset(r: int, c: int, cols: int) -> int:
    return lib().oracle_sf_offset(r, c, cols)


def sf_bytes(rows: int, cols: int) -> int:
    return lib().oracle_sf_bytes(rows, cols)


def sf_bytes_grouped(rows: int, cols: int, groups: int) -> int:
    return lib().oracle_sf_bytes_grouped(rows, cols, groups)


def group_sf_row(offsets: np.ndarray, g: int) -> int:
    o = np.ascontiguousarray(offsets, dtype=np.int64)
    return lib().oracle_group_sf_row(_p(o), g)


def rht16(x, sign_mask: int):
    xs = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    assert xs.size == 16
    out = np.zeros(16, dtype=np.float32)
    lib().oracle_rht16(_p(xs), sign_mask, _p(out))
    return out


# ----------------------------------------------------------------- tensors
def amax(x) -> float:
    xb = _bf16_bits(x)
    rows, cols = xb.shape
    return lib().oracle_amax_bf16(_p(xb), rows, cols, cols)


def quantize_1d(x, mode: int = RNE, seed: int = 0, amax_in: Optional[float] = None):
    """x: bf16 [rows, cols] -> dict(codes [rows, cols/2] u8, sf swizzled u8, amax)."""
    xb = _bf16_bits(x)
    rows, cols = xb.shape
    codes = np.zeros((rows, cols // 2), dtype=np.uint8)
    sf = np.zeros(sf_bytes(rows, cols), dtype=np.uint8)
    am = np.zeros(1, dtype=np.float32)
    ain = None if amax_in is None else np.array([amax_in], dtype=np.float32)
    lib().oracle_quantize_1d(_p(xb), rows, cols, cols, mode, seed, _p(ain), _p(codes), _p(sf), _p(am))
    return {"codes": codes, "sf": sf, "amax": float(am[0])}


def quantize_1d_grouped(x, offsets, mode: int = RNE, seed: int = 0, amax_in=None):
    xb = _bf16_bits(x)
    rows, cols = xb.shape
    off = np.ascontiguousarray(np.asarray(offsets, dtype=np.int64))
    groups = off.size - 1
    codes = np.zeros((rows, cols // 2), dtype=np.uint8)
    sf = np.zeros(sf_bytes_grouped(rows, cols, groups), dtype=np.uint8)
    am = np.zeros(groups, dtype=np.float32)
    ain = None if amax_in is None else np.ascontiguousarray(np.asarray(amax_in, dtype=np.float32))
    lib().oracle_quantize_1d_grouped(_p(xb), rows, cols, cols, _p(off), groups, mode, seed,
                                     _p(ain), _p(codes), _p(sf), _p(am))
    return {"codes": codes, "sf": sf, "amax": am}


def quantize_2d(w, want_t: bool = True, amax_in=None):
    """w: bf16 [rows, cols] or [batch, rows, cols]."""
    wb = _bf16_bits(w)
    if wb.ndim == 2:
        wb = wb[None]
    batch, rows, cols = wb.shape
    wb = np.ascontiguousarray(wb)
    codes = np.zeros((batch, rows, cols // 2), dtype=np.uint8)
    sf = np.zeros(batch * sf_bytes(rows, cols), dtype=np.uint8)
    codes_t = np.zeros((batch, cols, rows // 2), dtype=np.uint8) if want_t else None
    sf_t = np.zeros(batch * sf_bytes(cols, rows), dtype=np.uint8) if want_t else None
    tile = np.zeros((batch, rows // 16, cols // 16), dtype=np.uint8)
    am = np.zeros(batch, dtype=np.float32)
    ain = None if amax_in is None else np.ascontiguousarray(np.asarray(amax_in, dtype=np.float32))
    lib().oracle_quantize_2d(_p(wb), batch, rows, cols, cols, _p(ain), _p(codes), _p(sf),
                             _p(codes_t), _p(sf_t), _p(tile), _p(am))
    return {"codes": codes, "sf": sf, "codes_t": codes_t, "sf_t": sf_t, "tile_sf": tile, "amax": am}


def rht_amax(x, sign_mask: int) -> float:
    xb = _bf16_bits(x)
    tokens, cols = xb.shape
    return lib().oracle_rht_amax(_p(xb), tokens, cols, cols, sign_mask)


def rht_quantize(x, sign_mask: int, mode: int = RNE, seed: int = 0, amax_in: Optional[float] = None):
    """x: bf16 [tokens, cols] -> transposed operand [cols, tokens]."""
    xb = _bf16_bits(x)
    tokens, cols = xb.shape
    codes = np.zeros((cols, tokens // 2), dtype=np.uint8)
    sf = np.zeros(sf_bytes(cols, tokens), dtype=np.uint8)
    am = np.zeros(1, dtype=np.float32)
    ain = None if amax_in is None else np.array([amax_in], dtype=np.float32)
    lib().oracle_rht_quantize(_p(xb), tokens, cols, cols, sign_mask, mode, seed, _p(ain),
                              _p(codes), _p(sf), _p(am))
    return {"codes": codes, "sf": sf, "amax": float(am[0])}


def quantize_1d_mse(x, amax_in=None):
    """1x16 RNE quantisation with each block's E4M3 scale chosen by minimum
    squared error over all finite positive codes (R16)."""
    xb = _bf16_bits(x)
    rows, cols = xb.shape
    codes = np.zeros((rows, cols // 2), dtype=np.uint8)
    sf = np.zeros(sf_bytes(rows, cols), dtype=np.uint8)
    am = np.zeros(1, dtype=np.float32)
    ain = None if amax_in is None else np.array([amax_in], dtype=np.float32)
    lib().oracle_quantize_1d_mse(_p(xb), rows, cols, cols, _p(ain), _p(codes), _p(sf), _p(am))
    return {"codes": codes, "sf": sf, "amax": float(am[0])}


def fp16_sr(x: float, u: int) -> int:
    """FP16 bits of x stochastically rounded with the 32-bit word u (R15)."""
    return lib().oracle_fp16_sr(x, u)


def sr_fp16(x, seed: int) -> np.ndarray:
    """FP32 array -> FP16 bits (uint16) with SR, word of element e from (seed, e) (R4, R15)."""
    xs = np.ascontiguousarray(np.asarray(x, dtype=np.float32)).reshape(-1)
    out = np.zeros(xs.size, dtype=np.uint16)
    lib().oracle_sr_fp16(_p(xs), xs.size, seed, _p(out))
    return out


def group_k_offset(offsets, g: int) -> int:
    """Column where expert g's 64-padded token segment starts (R14)."""
    o = np.ascontiguousarray(np.asarray(offsets, dtype=np.int64))
    return lib().oracle_group_k_offset(_p(o), g)


def rht_quantize_grouped(x, offsets, kt: int, sign_mask: int, mode: int = RNE, seed: int = 0, amax_in=None):
    """x: bf16 [rows, cols], expert-sorted -> transposed operand [cols, kt]
    with every expert's segment padded to 64 tokens (R14)."""
    xb = _bf16_bits(x)
    rows, cols = xb.shape
    off = np.ascontiguousarray(np.asarray(offsets, dtype=np.int64))
    groups = off.size - 1
    codes = np.zeros((cols, kt // 2), dtype=np.uint8)
    sf = np.zeros(sf_bytes(cols, kt), dtype=np.uint8)
    am = np.zeros(groups, dtype=np.float32)
    ain = None if amax_in is None else np.ascontiguousarray(np.asarray(amax_in, dtype=np.float32))
    lib().oracle_rht_quantize_grouped(_p(xb), rows, cols, cols, _p(off), groups, kt, sign_mask, mode, seed,
                                      _p(ain), _p(codes), _p(sf), _p(am))
    return {"codes": codes, "sf": sf, "amax": am}


def dequantize_rows(codes: np.ndarray, sf: np.ndarray, cols: int, amax: float,
                    rows, sf_row0: int = 0) -> np.ndarray:
    """FP64 dequantisation of the listed rows of a quantised [*, cols] tensor."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    sf = np.ascontiguousarray(sf, dtype=np.uint8)
    idx = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    out = np.zeros((idx.size, cols), dtype=np.float64)
    lib().oracle_dequantize_rows(_p(codes), _p(sf), sf_row0, cols, amax, _p(idx), idx.size, _p(out))
    return out


def dequantize(q: dict, rows: int, cols: int) -> np.ndarray:
    return dequantize_rows(q["codes"].reshape(rows, cols // 2), q["sf"], cols,
                           float(np.asarray(q["amax"]).reshape(-1)[0]), np.arange(rows))


def gemm(A: np.ndarray, B: np.ndarray):
    """ref = A @ B^T and absum = |A| @ |B|^T elementwise-product sums, FP64 loops."""
    A = np.ascontiguousarray(A, dtype=np.float64)
    B = np.ascontiguousarray(B, dtype=np.float64)
    M, K = A.shape
    N = B.shape[0]
    ref = np.zeros((M, N), dtype=np.float64)
    absum = np.zeros((M, N), dtype=np.float64)
    lib().oracle_gemm(_p(A), _p(B), M, N, K, _p(ref), _p(absum))
    return ref, absum


def num_threads() -> int:
    return lib().oracle_num_threads()
