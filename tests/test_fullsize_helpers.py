"""The sampled-row helpers of the full-size parity tests give the same bytes
as the oracle's whole-tensor quantisers (small operands, CPU), and the row
checks they feed reject a planted mistake."""
import numpy as np
import pytest
import torch

import fullsize as fs


def _bf16(rows, cols, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(rows, cols, generator=g) * std).to(torch.bfloat16)


def _whole_scales(orc, sf, rows, cols, sf_row0=0):
    return fs.scale_rows(orc, sf, [sf_row0 + r for r in rows], cols)


@pytest.mark.parametrize("mode", [0, 1])
def test_rows_1d_equal_whole_tensor(orc, mode):
    x = _bf16(70, 96, 1)
    xb = fs.bits(x)
    q = orc.quantize_1d(x, mode=mode, seed=123)
    ids = fs.sample_ids(70, 9, 2, must=[31, 32, 63])
    rows = fs.rows_1d(orc, xb[ids], ids, 96, orc.amax(xb), mode, 123)
    assert rows.amax == q["amax"]
    fs.assert_rows_equal("1d", rows, q["codes"][ids], _whole_scales(orc, q["sf"], ids, 96), ids)
    # dequantised rows equal the oracle's dequantisation of the whole tensor
    whole = orc.dequantize(q, 70, 96)
    assert (rows.dequantized(orc) == whole[ids]).all()


def test_rows_1d_grouped_equal_whole_tensor(orc):
    """Grouped operands: rows of expert g use its own amax and scale rows
    from P_g; the SR index is the row's index in the whole output."""
    x = _bf16(300, 64, 3)
    xb = fs.bits(x)
    offsets = np.array([0, 5, 5, 140, 141, 300], dtype=np.int64)
    for mode in (0, 1):
        q = orc.quantize_1d_grouped(x, offsets, mode=mode, seed=9)
        for g in (0, 2, 3, 4):
            o0, o1 = int(offsets[g]), int(offsets[g + 1])
            ids = fs.sample_ids(o1 - o0, 6, g) + o0
            am = orc.amax(xb[o0:o1])
            assert am == q["amax"][g]
            rows = fs.rows_1d(orc, xb[ids], ids, 64, am, mode, 9)
            p = orc.group_sf_row(offsets, g)
            fs.assert_rows_equal(f"grouped g{g}", rows, q["codes"][ids],
                                 _whole_scales(orc, q["sf"], ids - o0, 64, p), ids)


def test_rows_2d_and_transposed_equal_whole_tensor(orc):
    w = _bf16(64, 160, 4, std=0.02)
    wb = fs.bits(w)
    q = orc.quantize_2d(w, want_t=True)
    am = orc.amax(wb)
    assert am == q["amax"][0]
    ids = fs.sample_ids(64, 7, 5, must=[15, 16])
    rows = fs.rows_2d(orc, lambda n0: wb[n0:n0 + 16], ids, 160, am)
    fs.assert_rows_equal("2d", rows, q["codes"][0][ids], _whole_scales(orc, q["sf"], ids, 160), ids)
    # rows of W^T: 16-column slabs of W, transposed
    tid = fs.sample_ids(160, 7, 6, must=[47, 48])
    trows = fs.rows_2d(orc, lambda k0: np.ascontiguousarray(wb[:, k0:k0 + 16].T), tid, 64, am)
    fs.assert_rows_equal("2d^T", trows, q["codes_t"][0][tid], _whole_scales(orc, q["sf_t"], tid, 64), tid)


def test_rows_2d_batched_equal_whole_tensor(orc):
    w = torch.stack([_bf16(32, 64, 7 + e, std=0.02 * (e + 1)) for e in range(3)])
    q = orc.quantize_2d(w, want_t=False)
    nsf = orc.sf_bytes(32, 64)
    for e in range(3):
        wb = fs.bits(w[e])
        am = orc.amax(wb)
        assert am == q["amax"][e]
        ids = np.array([0, 17, 31])
        rows = fs.rows_2d(orc, lambda n0: wb[n0:n0 + 16], ids, 64, am)
        fs.assert_rows_equal(f"batched e{e}", rows, q["codes"][e][ids],
                             fs.scale_rows(orc, q["sf"], ids, 64, base=e * nsf), ids)


@pytest.mark.parametrize("mode", [0, 1])
def test_rows_rht_equal_whole_tensor(orc, mode):
    x = _bf16(96, 40, 8)
    xb = fs.bits(x)
    mask = 0x6A5C
    q = orc.rht_quantize(x, mask, mode=mode, seed=77)
    am = orc.rht_amax(xb, mask)
    assert am == q["amax"]
    ids = fs.sample_ids(40, 6, 9, must=[33])
    rows = fs.rows_rht(orc, np.ascontiguousarray(xb[:, ids]), ids, 96, am, mask, mode, 77)
    fs.assert_rows_equal("rht", rows, q["codes"][ids], _whole_scales(orc, q["sf"], ids, 96), ids)


@pytest.mark.parametrize("mode", [0, 1])
def test_rows_rht_of_expert_segments_equal_whole_tensor(orc, mode):
    """Expert-segmented RHT operand [cols, kt]: expert g's zero-padded
    segment at column ko_g, its own RHT amax, SR index c * kt + ko_g + t."""
    x = _bf16(230, 24, 11)
    xb = fs.bits(x)
    offsets = np.array([0, 30, 30, 100, 229, 230], dtype=np.int64)
    counts = np.diff(offsets)
    kt = int(((counts + 63) // 64 * 64).sum()) + 64
    mask = 0x0F0F
    q = orc.rht_quantize_grouped(x, offsets, kt, mask, mode=mode, seed=31)
    for g in (0, 2, 3, 4):
        o0, o1 = int(offsets[g]), int(offsets[g + 1])
        seg = fs.padded_segment(xb, o0, o1)
        kp, ko = seg.shape[0], orc.group_k_offset(offsets, g)
        am = orc.rht_amax(seg, mask)
        assert am == q["amax"][g]
        ids = np.array([0, 5, 23])
        rows = fs.rows_rht(orc, np.ascontiguousarray(seg[:, ids]), ids, kp, am, mask, mode, 31,
                           index_stride=kt, index_offset=ko)
        codes = q["codes"][ids][:, ko // 2:(ko + kp) // 2]
        scales = fs.scale_rows(orc, q["sf"], ids, kt)[:, ko // 16:(ko + kp) // 16]
        fs.assert_rows_equal(f"segment g{g}", rows, codes, scales, ids)


def test_row_check_rejects_a_planted_mistake(orc):
    """A wrong SR index (the row's local index instead of its index in the
    whole output) or one flipped code is caught."""
    x = _bf16(40, 64, 10)
    xb = fs.bits(x)
    q = orc.quantize_1d(x, mode=1, seed=5)
    ids = np.array([3, 20, 39])
    sc = _whole_scales(orc, q["sf"], ids, 64)
    wrong = fs.rows_1d(orc, xb[ids], ids, 64, orc.amax(xb), 1, 5, index_rows=np.arange(3))
    with pytest.raises(AssertionError):
        fs.assert_rows_equal("local index", wrong, q["codes"][ids], sc, ids)
    right = fs.rows_1d(orc, xb[ids], ids, 64, orc.amax(xb), 1, 5)
    codes = q["codes"][ids].copy()
    codes[1, 7] ^= 0x10
    with pytest.raises(AssertionError):
        fs.assert_rows_equal("flipped", right, codes, sc, ids)


def test_sample_ids():
    ids = fs.sample_ids(1000, 10, 0, must=[500, 2000])
    assert len(ids) == 10 and ids[0] == 0 and ids[-1] == 999 and 500 in ids
    assert (np.diff(ids) > 0).all()
    assert list(fs.sample_ids(3, 10, 0)) == [0, 1, 2]
