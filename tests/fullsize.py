"""Helpers of the full-size parity tests (no method arithmetic here).

At the full workload sizes the oracle cannot quantise whole operands in a
test's time, so it quantises only sampled rows.  Each helper composes the
oracle's own whole-tensor steps for those rows: the tensor amax of the whole
operand (computed by the oracle over all of it), the block encoder with the
element index the block has in the whole output (the SR word depends on it),
the 2D quantiser on the 16-row slab that holds a row, and the 16-point RHT on
the token chunks of a column.  CPU tests check every helper against the
oracle's whole-tensor quantisers on small operands, so a full-size test
compares the GPU with exactly the bytes the oracle would give for the whole
operand."""
import numpy as np
import torch


def bits(x) -> np.ndarray:
    """bf16 tensor (any device) -> host uint16 array of its bits."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16
        return x
    return x.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def f32(b: np.ndarray) -> np.ndarray:
    """bf16 bits -> float32 values (exact)."""
    return (b.astype(np.uint32) << 16).view(np.float32)


def pack(codes) -> np.ndarray:
    """4-bit codes (even count) -> bytes, element 2j in the low nibble."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[0::2] | (c[1::2] << 4)).astype(np.uint8)


def scale_rows(orc, sf: np.ndarray, rows, cols: int, base: int = 0, b0: int = 0, b1=None) -> np.ndarray:
    """Block scales [len(rows), b1-b0] (blocks b0 .. b1-1, all by default) of
    the listed scale rows of a swizzled buffer (atoms laid out for a
    [*, cols] operand, starting at byte `base`)."""
    b1 = cols // 16 if b1 is None else b1
    out = np.zeros((len(rows), b1 - b0), dtype=np.uint8)
    for i, r in enumerate(rows):
        for b in range(b0, b1):
            out[i, b - b0] = sf[base + orc.sf_offset(int(r), b, cols)]
    return out


class OracleRows:
    """The oracle's codes [n, cols/2], block scales [n, cols/16] and tensor
    amax for n sampled rows of an operand."""

    def __init__(self, n: int, cols: int, amax: float):
        self.codes = np.zeros((n, cols // 2), dtype=np.uint8)
        self.scales = np.zeros((n, cols // 16), dtype=np.uint8)
        self.cols = cols
        self.amax = float(amax)

    def local_sf(self, orc) -> np.ndarray:
        """The scales in a swizzled buffer of an [n, cols] operand (row i at scale row i)."""
        n = self.codes.shape[0]
        sf = np.zeros(orc.sf_bytes(n, self.cols), dtype=np.uint8)
        for i in range(n):
            for b in range(self.cols // 16):
                sf[orc.sf_offset(i, b, self.cols)] = self.scales[i, b]
        return sf

    def dequantized(self, orc) -> np.ndarray:
        """FP64 values of the rows (the oracle's dequantisation)."""
        n = self.codes.shape[0]
        return orc.dequantize_rows(self.codes, self.local_sf(orc), self.cols, self.amax, np.arange(n))


def rows_1d(orc, x_rows: np.ndarray, row_ids, cols: int, amax: float, mode: int, seed: int = 0,
            index_rows=None) -> OracleRows:
    """1x16 quantisation of rows `row_ids` of a [*, cols] operand with tensor
    amax `amax`; x_rows: bf16 bits [n, cols] of those rows.  The SR index of
    element (r, c) is index_row * cols + c, index_row = row_ids[i] unless
    index_rows gives it."""
    out = OracleRows(len(row_ids), cols, amax)
    s_enc = orc.tensor_scale(amax)
    xf = f32(x_rows)
    idx = row_ids if index_rows is None else index_rows
    for i in range(len(row_ids)):
        e_row = int(idx[i]) * cols
        for b in range(cols // 16):
            sfb, cd = orc.encode_block(xf[i, 16 * b:16 * b + 16], s_enc, mode, seed, e_row + 16 * b)
            out.scales[i, b] = sfb
            out.codes[i, 8 * b:8 * b + 8] = pack(cd)
    return out


def rows_2d(orc, slab, row_ids, cols: int, amax: float) -> OracleRows:
    """16x16 quantisation of rows `row_ids` of a weight with tensor amax
    `amax`; slab(n0) returns the bf16 bits [16, cols] of rows n0 .. n0+15."""
    out = OracleRows(len(row_ids), cols, amax)
    cache = {}
    for i, n in enumerate(row_ids):
        n0 = int(n) // 16 * 16
        if n0 not in cache:
            cache[n0] = orc.quantize_2d(np.ascontiguousarray(slab(n0)), want_t=False,
                                        amax_in=np.array([amax], dtype=np.float32))
        q = cache[n0]
        out.codes[i] = q["codes"][0][int(n) - n0]
        out.scales[i] = scale_rows(orc, q["sf"], [int(n) - n0], cols)[0]
    return out


def rows_rht(orc, x_cols: np.ndarray, col_ids, tokens: int, amax: float, sign_mask: int, mode: int,
             seed: int = 0, index_stride: int = 0, index_offset: int = 0) -> OracleRows:
    """Rows `col_ids` of the RHT operand [cols, tokens] of x [tokens, cols]
    with RHT amax `amax`; x_cols: bf16 bits [tokens, n] of those columns.
    Each 16-token chunk is transformed and encoded as one block; the SR index
    of output element (c, t) is c * tokens + t, or c * index_stride +
    index_offset + t for an expert segment placed at column index_offset of
    an operand index_stride tokens wide."""
    out = OracleRows(len(col_ids), tokens, amax)
    s_enc = orc.tensor_scale(amax)
    xf = f32(x_cols)
    stride = index_stride if index_stride else tokens
    for i, c in enumerate(col_ids):
        col = np.ascontiguousarray(xf[:, i])
        for t0 in range(0, tokens, 16):
            y = orc.rht16(col[t0:t0 + 16], sign_mask)
            sfb, cd = orc.encode_block(y, s_enc, mode, seed, int(c) * stride + index_offset + t0)
            out.scales[i, t0 // 16] = sfb
            out.codes[i, t0 // 2:t0 // 2 + 8] = pack(cd)
    return out


def padded_segment(x_bits: np.ndarray, o0: int, o1: int, pad: int = 64) -> np.ndarray:
    """Rows o0 .. o1-1 of x (bf16 bits) followed by zero rows up to a multiple of `pad`."""
    n = o1 - o0
    kp = (n + pad - 1) // pad * pad
    seg = np.zeros((kp, x_bits.shape[1]), dtype=np.uint16)
    seg[:n] = x_bits[o0:o1]
    return seg


def assert_rows_equal(name: str, orc_rows: OracleRows, gpu_codes: np.ndarray, gpu_scales: np.ndarray, row_ids):
    """Codes and block scales of the sampled rows, bit for bit."""
    bad_sf = np.argwhere(gpu_scales != orc_rows.scales)
    assert bad_sf.size == 0, (f"{name}: {len(bad_sf)} block scales differ, first (row, block) "
                              f"{[(int(row_ids[i]), int(b)) for i, b in bad_sf[:4]]}")
    bad = np.argwhere(gpu_codes != orc_rows.codes)
    assert bad.size == 0, (f"{name}: {len(bad)} code bytes differ, first (row, byte) "
                           f"{[(int(row_ids[i]), int(b)) for i, b in bad[:4]]}")


def sample_ids(n: int, k: int, seed: int, must=()) -> np.ndarray:
    """k sorted distinct indices in [0, n): the `must` ones, the first and
    the last, and seeded random others."""
    rng = np.random.default_rng(seed)
    ids = set(int(m) for m in must if 0 <= m < n) | {0, n - 1}
    while len(ids) < min(k, n):
        ids.add(int(rng.integers(0, n)))
    return np.array(sorted(ids), dtype=np.int64)
