"""Shared helpers of the GPU parity tests (no method arithmetic here: the
expected values always come from the oracle)."""
import numpy as np
import torch


def np_u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().numpy()


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(x), np.float64(2.0) ** -126)
    return np.float64(2.0) ** (np.floor(np.log2(ax)) - 7)


def gemm_within_bound(out: np.ndarray, ref: np.ndarray, absum: np.ndarray, bf16: bool):
    """The GEMM acceptance rule: |gpu - ref| <= 1e-5 * sum_k |a_k b_k| per
    element against the FP64 reference on the dequantised operands; a bf16
    output may also carry its one rounding (half a bf16 ulp of the larger of
    |ref| and |gpu|).  Returns (ok mask, worst error / tolerance)."""
    out = out.astype(np.float64)
    tol = 1e-5 * absum
    if bf16:
        tol = tol + 0.5 * bf16_ulp(np.maximum(np.abs(ref), np.abs(out)))
    err = np.abs(out - ref)
    ok = err <= tol
    ratio = np.where(tol > 0, err / np.where(tol > 0, tol, 1), np.where(err > 0, np.inf, 0))
    return ok, float(ratio.max()) if ratio.size else 0.0


def sf_rows_region(sf: np.ndarray, scale_rows: int, cols: int) -> np.ndarray:
    """Bytes of the first `scale_rows` (a multiple of 128) scale rows."""
    catoms = ((cols // 16) + 3) // 4
    return sf[: (scale_rows // 128) * catoms * 512]
