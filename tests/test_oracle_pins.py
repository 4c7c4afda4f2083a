"""Pins of the CPU oracle against things other than itself: format tables from
their definitions, a library conversion (torch float8_e4m3fn), hand-worked
blocks, published Philox known-answer values, Hadamard algebra checked
against scipy, SR unbiasedness, brute force on tiny inputs, and invariants.
No GPU is needed."""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import scipy.linalg
import torch

from nvfp4_precision_02_b300 import workloads as wl

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ------------------------------------------------------------ format tables
def test_e2m1_table_from_bit_fields(orc):
    # OCP MX E2M1: 1 sign, 2 exponent (bias 1), 1 mantissa bit; exponent 0 is
    # subnormal with value m * 2^-1.
    for code in range(16):
        s, e, m = code >> 3, (code >> 1) & 3, code & 1
        mag = Fraction(m, 2) if e == 0 else Fraction(2) ** (e - 1) * (1 + Fraction(m, 2))
        want = -float(mag) if s else float(mag)
        got = orc.e2m1_value(code)
        assert got == want and math.copysign(1, got) == math.copysign(1, want), code


def test_e4m3_decode_matches_torch_float8(orc):
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    got = np.array([orc.e4m3_value(b) for b in range(256)])
    nan = np.isnan(ref)
    assert (np.isnan(got) == nan).all()
    assert nan.sum() == 2                      # 0x7F and 0xFF only
    assert (got[~nan] == ref[~nan]).all()
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


def test_e4m3_encode_matches_torch_in_range(orc):
    # every representable value, every midpoint between neighbours, and a
    # dense random sweep: torch's float8 cast rounds to nearest-even.
    vals = sorted({orc.e4m3_value(b) for b in range(0x7F)})
    mids = [(a + b) / 2 for a, b in zip(vals, vals[1:])]
    rng = np.random.default_rng(0)
    sweep = list(np.exp(rng.uniform(np.log(1e-4), np.log(448.0), 20000)).astype(np.float32))
    xs = np.array(vals + mids + sweep + [0.0, 1e-30, 2.0 ** -10, 3 * 2.0 ** -11], dtype=np.float32)
    want = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.e4m3_encode(float(x)) for x in xs], dtype=np.uint8)
    assert (got == want).all(), np.nonzero(got != want)


def test_e4m3_encode_saturates(orc):
    # satfinite reading: anything at or above 448 encodes as 448 (0x7E)
    for x in [448.0, 449.0, 464.0, 470.0, 1e6, 3.4e38]:
        assert orc.e4m3_encode(x) == 0x7E


def test_e2m1_rne_grid_and_ties(orc):
    grid = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for i, g in enumerate(grid):
        assert orc.e2m1_rne(g) == i
        assert orc.e2m1_rne(-g) == 8 | i
    for v, code in [(0.25, 0), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6), (5.0, 6),
                    (0.2499, 0), (0.2501, 1), (5.001, 7), (6.5, 7), (1e9, 7), (-0.1, 8)]:
        assert orc.e2m1_rne(v) == code, v


def test_e2m1_rne_is_nearest_bruteforce(orc):
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    rng = np.random.default_rng(1)
    for v in rng.uniform(-7, 7, 3000).astype(np.float32):
        c = orc.e2m1_rne(float(v))
        d = np.abs(abs(float(v)) - grid)
        mag = grid[c & 7]
        if abs(v) <= 6:
            assert abs(abs(v) - mag) == d.min()
        else:
            assert mag == 6
        assert (c >> 3) == (1 if v < 0 or (v == 0 and math.copysign(1, v) < 0) else 0)


# ------------------------------------------------------------ scales
def test_tensor_scale_special_cases(orc):
    assert orc.tensor_scale(2688.0) == 1.0
    assert orc.tensor_scale(0.0) == 1.0                     # empty / all-zero tensor
    assert orc.tensor_scale(1.0) == 2688.0
    assert orc.tensor_scale(1e-38) == np.finfo(np.float32).max   # quotient overflows: clamp
    assert orc.decode_scale(2688.0) == 1.0


def test_element_multiplier_overflow_clamps(orc):
    """Reading R3 with R1's clamp, worked by hand.  Tensor amax 1e-37:
    2688 / amax overflows, so S_enc = FLT_MAX.  Block max 2^-132 (bf16
    0x0002): (2^-132 / 6) * FLT_MAX = 0.0104, E4M3 code 5 (5 * 2^-9, a
    subnormal scale).  FLT_MAX / (5 * 2^-9) overflows as well and clamps to
    FLT_MAX, so 2^-132 * FLT_MAX = 0.0625, +-2^-133 * FLT_MAX = +-0.03125 and
    +-0 stay +-0: every element rounds to zero, negative ones to code 0x8.
    Without the clamp the multiplier is inf: 2^-132 would encode as 6 (code
    7) and the zeros as NaN."""
    bits = np.zeros((1, 16), dtype=np.uint16)
    bits[0, :5] = [0x0000, 0x8000, 0x0002, 0x8001, 0x0001]
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
    ref = orc.quantize_1d(x, mode=0, amax_in=1e-37)
    assert ref["sf"][orc.sf_offset(0, 0, 16)] == 0x05
    assert list(ref["codes"][0]) == [0x80, 0x80] + [0] * 6


def test_block_scale_max_maps_to_448(orc):
    # the block holding the tensor amax gets scale 448 (largest E4M3) for any amax
    rng = np.random.default_rng(2)
    for amax in rng.uniform(1e-3, 1e3, 200).astype(np.float32):
        s = orc.block_scale(float(amax), orc.tensor_scale(float(amax)))
        assert s == 0x7E


# ------------------------------------------------------------ hand-worked blocks
@pytest.mark.parametrize("blk", _load("blocks.json")["blocks"], ids=lambda b: b["name"])
def test_hand_worked_blocks(orc, blk):
    sf, codes = orc.encode_block(np.array(blk["x"], dtype=np.float32), orc.tensor_scale(blk["amax"]))
    assert sf == blk["sf"]
    assert codes == blk["codes"]


# ------------------------------------------------------------ Philox / SR
def test_philox_known_answers(orc):
    kat = _load("philox4x32_kat.json")
    for v in kat["vectors"]:
        ctr = [int(x, 16) for x in v["ctr"]]
        key = [int(x, 16) for x in v["key"]]
        assert orc.philox4x32(ctr, key, kat["rounds"]) == [int(x, 16) for x in v["out"]]


def test_sr_word_counter_layout(orc):
    # element e uses word e & 3 of Philox5(ctr = (e >> 2) split lo/hi, key = seed lo/hi)
    seed = 0x0123456789ABCDEF
    for e in [0, 1, 2, 3, 4, 7, 1 << 33 | 5]:
        q = e >> 2
        out = orc.philox4x32([q & 0xFFFFFFFF, q >> 32, 0, 0], [seed & 0xFFFFFFFF, seed >> 32], 5)
        assert orc.sr_word(seed, e) == out[e & 3]


@pytest.mark.parametrize("case", _load("sr_cases.json")["cases"], ids=lambda c: f'{c["v"]}-{c["u"]}')
def test_sr_hand_cases(orc, case):
    assert orc.e2m1_sr(case["v"], case["u"]) == case["code"]


def test_sr_unbiased_rne_biased(orc):
    """Over many random words SR's mean equals the input (CLT 4-sigma bound);
    RTNE's error is systematic (Nemotron 3 Super summary, section 4.3)."""
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    n = 20000
    words = [orc.sr_word(99, e) for e in range(n)]
    for v in [0.1, 0.3, 0.625, 1.2, 2.7, 3.3, 4.9, 5.5]:
        vals = np.array([grid[orc.e2m1_sr(v, u) & 7] for u in words])
        lo = grid[grid <= v].max()
        hi = grid[grid > v].min()
        sigma = (hi - lo) * 0.5 / math.sqrt(n)
        assert abs(vals.mean() - v) < 4 * sigma, v
        assert set(np.unique(vals)) <= {lo, hi}
        rne = grid[orc.e2m1_rne(v) & 7]
        assert rne != v                 # RTNE is deterministic: error never averages out


# ------------------------------------------------------------ layout
def test_sf_layout_hand_offsets(orc):
    cols = 128    # 8 scale columns -> 2 column atoms
    assert orc.sf_offset(0, 0, cols) == 0
    assert orc.sf_offset(1, 0, cols) == 16
    assert orc.sf_offset(32, 0, cols) == 4
    assert orc.sf_offset(33, 3, cols) == 16 + 4 + 3
    assert orc.sf_offset(0, 4, cols) == 512
    assert orc.sf_offset(128, 0, cols) == 1024
    assert orc.sf_bytes(129, 128) == 256 * 8
    assert orc.sf_bytes(1, 16) == 128 * 4


@pytest.mark.parametrize("rows,cols", [(1, 16), (130, 48), (256, 256), (300, 1040)])
def test_sf_layout_is_a_bijection(orc, rows, cols):
    R = -(-rows // 128) * 128
    C = -(-(cols // 16) // 4) * 4
    offs = {orc.sf_offset(r, c, cols) for r in range(R) for c in range(C)}
    assert offs == set(range(orc.sf_bytes(rows, cols)))


# ------------------------------------------------------------ Hadamard
def test_rht_matrix_is_scaled_sylvester_hadamard(orc):
    H = scipy.linalg.hadamard(16).astype(np.float64)
    for mask in [0, 0xFFFF, 0xA5C3, 1]:
        s = np.array([-1.0 if (mask >> j) & 1 else 1.0 for j in range(16)])
        Q = np.stack([orc.rht16(np.eye(16)[j], mask) for j in range(16)], axis=1).astype(np.float64)
        assert (Q == 0.25 * H * s[None, :]).all()
        assert (Q @ Q.T == np.eye(16)).all()       # orthogonal for every sign pattern
    assert (H @ H.T == 16 * np.eye(16)).all()


def test_rht_preserves_dot_products_and_concentrates_constants(orc):
    rng = np.random.default_rng(3)
    for _ in range(50):
        a = rng.standard_normal(16).astype(np.float32)
        b = rng.standard_normal(16).astype(np.float32)
        mask = int(rng.integers(0, 1 << 16))
        qa = orc.rht16(a, mask).astype(np.float64)
        qb = orc.rht16(b, mask).astype(np.float64)
        assert abs(qa @ qb - a.astype(np.float64) @ b) < 1e-5 * (np.abs(a) @ np.abs(b) + 1)
    y = orc.rht16(np.full(16, 3.0), 0)
    assert y[0] == 12.0 and (y[1:] == 0).all()


# ------------------------------------------------------------ whole tensors
def _bf16(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)


def _unpack(codes, cols):
    lo = codes & 15
    hi = codes >> 4
    return np.stack([lo, hi], axis=-1).reshape(codes.shape[0], cols)


def test_quantize_1d_bruteforce(orc):
    """Tiny tensor: every block's scale and every code recomputed in numpy
    FP32 by brute force over the grids, read back through the layout."""
    rng = np.random.default_rng(4)
    rows, cols = 37, 64
    x = _bf16(rng.standard_normal((rows, cols)) * np.exp(rng.uniform(-6, 3, (rows, 1))))
    q = orc.quantize_1d(x)
    xf = x.float().numpy()
    amax = np.float32(np.abs(xf).max())
    assert q["amax"] == amax
    s_enc = np.float32(2688.0) / amax
    e4 = torch.arange(127, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], dtype=np.float64)
    codes = _unpack(q["codes"], cols)
    for r in range(rows):
        for b in range(cols // 16):
            blk = xf[r, b * 16:(b + 1) * 16]
            sf_f = np.float32(np.float32(np.abs(blk).max()) / np.float32(6.0)) * s_enc
            want_sf = torch.tensor([sf_f]).to(torch.float8_e4m3fn).view(torch.uint8).item()
            sf = q["sf"][orc.sf_offset(r, b, cols)]
            assert sf == want_sf
            cb = codes[r, b * 16:(b + 1) * 16]
            if sf == 0:
                assert (cb == 0).all()
                continue
            rr = np.float32(s_enc / np.float32(e4[sf]))
            v = (blk * rr).astype(np.float32)
            for j in range(16):
                d = np.abs(abs(float(v[j])) - grid)
                mag = grid[cb[j] & 7]
                assert abs(abs(float(v[j])) - mag) == d.min() or (abs(v[j]) > 6 and mag == 6)
                assert (cb[j] >> 3) == (1 if np.signbit(v[j]) else 0)


def test_quantize_1d_sr_matches_per_element_rule(orc):
    rng = np.random.default_rng(5)
    rows, cols, seed = 9, 48, 1234
    x = _bf16(rng.standard_normal((rows, cols)))
    q = orc.quantize_1d(x, mode=orc.SR, seed=seed)
    qr = orc.quantize_1d(x)
    assert (q["sf"] == qr["sf"]).all()               # scales are always RNE
    codes = _unpack(q["codes"], cols)
    s_enc = orc.tensor_scale(q["amax"])
    xf = x.float().numpy()
    for r in range(rows):
        for c in range(cols):
            sf = q["sf"][orc.sf_offset(r, c // 16, cols)]
            rr = np.float32(np.float32(s_enc) / np.float32(orc.e4m3_value(sf)))
            v = float(np.float32(xf[r, c]) * rr)
            assert codes[r, c] == orc.e2m1_sr(v, orc.sr_word(seed, r * cols + c))


def test_quantize_1d_supplied_amax(orc):
    rng = np.random.default_rng(6)
    x = _bf16(rng.standard_normal((16, 32)))
    q1 = orc.quantize_1d(x)
    q2 = orc.quantize_1d(x, amax_in=q1["amax"])
    assert (q1["codes"] == q2["codes"]).all() and (q1["sf"] == q2["sf"]).all()
    q3 = orc.quantize_1d(x, amax_in=4 * q1["amax"])
    assert q3["amax"] == 4 * q1["amax"]


def test_quantize_2d_transpose_invariant(orc):
    """W and W^T quantise identically (2D blocks; Nemotron 3 Ultra report, 2.2)."""
    rng = np.random.default_rng(7)
    w = _bf16(rng.standard_normal((48, 80)) * 0.02)
    a = orc.quantize_2d(w)
    b = orc.quantize_2d(w.t().contiguous())
    assert (a["codes_t"] == b["codes"]).all() and (a["codes"] == b["codes_t"]).all()
    assert (a["sf_t"] == b["sf"]).all() and (a["sf"] == b["sf_t"]).all()
    assert (a["tile_sf"][0] == b["tile_sf"][0].T).all()
    assert a["amax"][0] == b["amax"][0]


def test_quantize_2d_tile_scale_is_tile_amax(orc):
    rng = np.random.default_rng(8)
    w = _bf16(rng.standard_normal((32, 64)) * np.exp(rng.uniform(-4, 2, (32, 64))))
    q = orc.quantize_2d(w)
    wf = w.float().numpy()
    s_enc = orc.tensor_scale(q["amax"][0])
    for ti in range(2):
        for tj in range(4):
            t = wf[ti * 16:(ti + 1) * 16, tj * 16:(tj + 1) * 16]
            s = orc.block_scale(float(np.abs(t).max()), s_enc)
            assert q["tile_sf"][0, ti, tj] == s
            for i in range(16):
                assert q["sf"][orc.sf_offset(ti * 16 + i, tj, 64)] == s
                assert q["sf_t"][orc.sf_offset(tj * 16 + i, ti, 32)] == s


def test_quantize_2d_batched_equals_per_batch(orc):
    rng = np.random.default_rng(9)
    w = _bf16(rng.standard_normal((3, 32, 48)))
    qb = orc.quantize_2d(w)
    n = orc.sf_bytes(32, 48)
    for b in range(3):
        q = orc.quantize_2d(w[b])
        assert (qb["codes"][b] == q["codes"][0]).all()
        assert (qb["sf"][b * n:(b + 1) * n] == q["sf"]).all()
        assert qb["amax"][b] == q["amax"][0]


@pytest.mark.parametrize("mode", [0, 1])
def test_rht_quantize_equals_quantize_of_exact_transform(orc, mode):
    """Integer inputs make the FP32 butterfly exact, so the RHT output equals
    0.25*H*D*x from scipy's Hadamard in FP64, and it is bf16-representable:
    quantising it with the 1D quantiser along tokens must give the same bytes
    (same transpose, chunking, sign bit order, and SR index space)."""
    rng = np.random.default_rng(10 + mode)
    T, C, mask, seed = 64, 24, 0xB3E1, 77
    x = _bf16(rng.integers(-8, 9, (T, C)))
    H = scipy.linalg.hadamard(16).astype(np.float64)
    s = np.array([-1.0 if (mask >> j) & 1 else 1.0 for j in range(16)])
    xf = x.double().numpy()
    y = np.zeros((C, T))
    for t0 in range(0, T, 16):
        y[:, t0:t0 + 16] = (0.25 * H @ (s[:, None] * xf[t0:t0 + 16, :])).T
    yb = _bf16(y)
    assert (yb.double().numpy() == y).all()
    q = orc.rht_quantize(x, mask, mode=mode, seed=seed)
    ref = orc.quantize_1d(yb, mode=mode, seed=seed)
    assert q["amax"] == ref["amax"] == np.abs(y).max()
    assert orc.rht_amax(x, mask) == q["amax"]
    assert (q["codes"] == ref["codes"]).all() and (q["sf"] == ref["sf"]).all()


@pytest.mark.parametrize("mode", [0, 1])
def test_rht_quantize_grouped_is_per_expert_padded_rht(orc, mode):
    """Expert-segmented RHT quantisation (reading R14): expert g's tokens,
    padded with zero tokens to a multiple of 64, sit at columns ko_g (the sum
    of the earlier padded counts) of the transposed operand.  Checked against
    the plain RHT quantiser run on each zero-padded segment on its own (RNE:
    same bytes; SR: the same words once the index space is shifted by the
    segment's column, via single blocks), and one expert of a multiple of 64
    tokens spanning the operand is exactly the plain RHT quantiser."""
    rng = np.random.default_rng(30 + mode)
    cols, mask, seed = 24, 0x5A3C, 91
    offsets = np.array([0, 30, 30, 100, 164, 165], dtype=np.int64)      # 30, 0, 70, 64, 1 tokens
    counts = np.diff(offsets)
    kp = (counts + 63) // 64 * 64
    ko = np.concatenate([[0], np.cumsum(kp)])
    kt = int(ko[-1]) + 64                                                 # capacity past the last expert
    x = _bf16(rng.standard_normal((int(offsets[-1]), cols)) * np.repeat([1, 1, 5, 0.02, 3], counts)[:, None])
    q = orc.rht_quantize_grouped(x, offsets, kt, mask, mode=mode, seed=seed)
    for g in range(len(counts)):
        assert orc.group_k_offset(offsets, g) == ko[g]
        if counts[g] == 0:
            assert q["amax"][g] == 0
            continue
        xp = torch.zeros(int(kp[g]), cols, dtype=torch.bfloat16)
        xp[:counts[g]] = x[offsets[g]:offsets[g + 1]]
        ref = orc.rht_quantize(xp, mask, mode=orc.RNE)
        assert q["amax"][g] == ref["amax"]
        if mode == 0:
            assert (q["codes"][:, ko[g] // 2:(ko[g] + kp[g]) // 2] == ref["codes"]).all()
            for c in range(cols):
                for b in range(int(kp[g]) // 16):
                    assert q["sf"][orc.sf_offset(c, ko[g] // 16 + b, kt)] == ref["sf"][orc.sf_offset(c, b, kp[g])]
        else:
            # every SR block: the padded segment's transform, encoded with words c*kt + ko_g + t
            s_enc = orc.tensor_scale(q["amax"][g])
            xf = xp.float().numpy()
            codes = _unpack(q["codes"], kt)
            for c in range(0, cols, 7):
                for t in range(0, int(kp[g]), 16):
                    y = orc.rht16(xf[t:t + 16, c], mask)
                    sf_b, cd = orc.encode_block(y, s_enc, orc.SR, seed, c * kt + int(ko[g]) + t)
                    assert q["sf"][orc.sf_offset(c, (int(ko[g]) + t) // 16, kt)] == sf_b
                    assert (codes[c, int(ko[g]) + t:int(ko[g]) + t + 16] == cd).all()
    # nothing is written past the last expert
    assert (q["codes"][:, ko[-1] // 2:] == 0).all()
    # one expert of 128 tokens spanning the operand: the plain RHT quantiser
    one = orc.rht_quantize_grouped(x[:128], np.array([0, 128]), 128, mask, mode=mode, seed=seed)
    ref = orc.rht_quantize(x[:128], mask, mode=mode, seed=seed)
    assert one["amax"][0] == ref["amax"]
    assert (one["codes"] == ref["codes"]).all() and (one["sf"] == ref["sf"]).all()


def test_grouped_quantize_equals_per_group(orc):
    rng = np.random.default_rng(12)
    cols = 32
    offsets = np.array([0, 5, 5, 140, 141, 300], dtype=np.int64)     # one empty group
    x = _bf16(rng.standard_normal((300, cols)) * np.repeat([1, 1, 3, 0.01, 7], np.diff(offsets))[:, None])
    q = orc.quantize_1d_grouped(x, offsets)
    codes = q["codes"]
    for g in range(len(offsets) - 1):
        o, n = offsets[g], offsets[g + 1] - offsets[g]
        po = orc.group_sf_row(offsets, g)
        assert po % 128 == 0
        if n == 0:
            assert q["amax"][g] == 0
            continue
        ref = orc.quantize_1d(x[o:o + n])
        assert q["amax"][g] == ref["amax"]
        assert (codes[o:o + n] == ref["codes"]).all()
        for r in range(n):
            for b in range(cols // 16):
                assert q["sf"][orc.sf_offset(po + r, b, cols)] == ref["sf"][orc.sf_offset(r, b, cols)]
    # SR: one group covering everything is the plain 1D quantiser
    one = orc.quantize_1d_grouped(x, np.array([0, 300]), mode=orc.SR, seed=5)
    ref = orc.quantize_1d(x, mode=orc.SR, seed=5)
    assert (one["codes"] == ref["codes"]).all()


# ------------------------------------------------------------ GEMM definition
def test_gemm_matches_numpy_float64(orc):
    rng = np.random.default_rng(13)
    A = rng.standard_normal((17, 48))
    B = rng.standard_normal((9, 48))
    ref, absum = orc.gemm(A, B)
    assert np.allclose(ref, A @ B.T, rtol=1e-12, atol=1e-12)
    assert np.allclose(absum, np.abs(A) @ np.abs(B).T, rtol=1e-12)


def test_gemm_of_dequantised_one_hot_operands_is_exact(orc):
    """One nonzero per row whose sixth is an E4M3 value: the block scale is
    exact, the element encodes as 6, dequantisation returns the input, and
    every output is a single exactly representable product."""
    K = 64
    A = np.zeros((16, K), dtype=np.float32)
    B = np.zeros((16, K), dtype=np.float32)
    for i in range(16):
        A[i, (5 * i) % K] = [6, 3, 1.5, 0.75, 9, 4.5, 7.5, -10.5][i % 8]
        B[i, (5 * i) % K] = [12, -6, 3, 1.5, 7.5, 0.375, 24, 9][i % 8]
    qa = orc.quantize_1d(_bf16(A), amax_in=2688.0)
    qb = orc.quantize_1d(_bf16(B), amax_in=2688.0)
    Ah = orc.dequantize(qa, 16, K)
    Bh = orc.dequantize(qb, 16, K)
    assert (Ah == A).all() and (Bh == B).all()
    ref, _ = orc.gemm(Ah, Bh)
    assert (ref == A.astype(np.float64) @ B.astype(np.float64).T).all()


def test_dequantise_roundtrip_error_bound(orc):
    """RNE: |x_hat - x| is at most half a grid gap at the block scale
    (the gap at 6 is 2, so <= 1 * scale), plus saturation never applies to
    the block's own amax element (it maps to <= 6)."""
    rng = np.random.default_rng(14)
    x = _bf16(rng.standard_normal((64, 64)))
    q = orc.quantize_1d(x)
    xh = orc.dequantize(q, 64, 64)
    xf = x.double().numpy()
    dec = orc.decode_scale(q["amax"])
    for r in range(64):
        for b in range(4):
            s = orc.e4m3_value(q["sf"][orc.sf_offset(r, b, 64)]) * dec
            err = np.abs(xh[r, b * 16:(b + 1) * 16] - xf[r, b * 16:(b + 1) * 16])
            # 1.02: the E4M3 rounding of the scale can shrink it by up to 1/16
            assert (err <= 1.0 * s * 1.07 + 1e-12).all()


# ------------------------------------------------------------ routing metric
def test_maxvio_bound():
    """MaxVio <= N/k, equal when one expert receives every token (Ultra report 2.7)."""
    r = wl.zipf_routing(2048, 512, 22, seed=4)
    assert r.max_vio <= wl.max_vio_bound(512, 22) + 1e-12
    assert int(r.offsets[-1]) == 2048 * 22
    assert (r.counts <= 2048).all()
    counts = torch.zeros(512, dtype=torch.int64)
    counts[:22] = 100          # every one of 100 tokens picks the same 22 experts
    fake = wl.Routing(torch.zeros(0), torch.zeros(0), torch.zeros(513), counts, 22)
    assert abs(fake.max_vio - 512 / 22) < 1e-12


# ------------------------------------------------------------ FP16 SR (SSM cache, reading R15)
def test_fp16_sr_keeps_exact_fp16_values(orc):
    """Every finite FP16 value is its own rounding for any word (p = 0)."""
    h = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = h.view(np.float16)
    keep = np.isfinite(vals)
    xs = vals[keep].astype(np.float32)
    bits = h[keep]
    rng = np.random.default_rng(50)
    for x, b, u in zip(xs[::7], bits[::7], rng.integers(0, 1 << 32, size=len(xs[::7]), dtype=np.uint64)):
        assert orc.fp16_sr(float(x), int(u)) == b


def test_fp16_sr_brackets_and_is_unbiased(orc):
    """The result is one of the two FP16 neighbours of x, and over an even
    grid of 65536 words its mean is x to within 2^-16 of the local spacing."""
    rng = np.random.default_rng(51)
    xs = (rng.standard_normal(300) * np.exp(rng.uniform(-20, 10, 300))).astype(np.float32)
    us = (np.arange(65536, dtype=np.uint64) << 16) | 0x1234
    for x in xs[:40]:
        r = np.float16(x)                                   # RNE: one neighbour
        if float(r) == float(x):
            continue
        other = np.nextafter(r, np.float16(np.inf) if float(x) > float(r) else np.float16(-np.inf))
        lo, hi = sorted([abs(float(r)), abs(float(other))])
        assert lo < abs(float(x)) < hi
        got = np.array([orc.fp16_sr(float(x), int(u)) for u in us[::64]], dtype=np.uint16).view(np.float16)
        assert set(np.abs(got.astype(np.float64))) <= {lo, hi}
    for x in xs[:6]:
        got = np.array([orc.fp16_sr(float(x), int(u)) for u in us], dtype=np.uint16).view(np.float16)
        m = abs(float(x))
        r = np.float16(m)
        sp = abs(float(np.nextafter(r, np.float16(np.inf))) - float(r)) if float(r) <= m else \
            abs(float(r) - float(np.nextafter(r, np.float16(0))))
        assert abs(np.abs(got.astype(np.float64)).mean() - m) <= sp * 2.0 ** -16 + 1e-30


def test_fp16_sr_threshold_and_special_values(orc):
    """p = 3/4 rounds up for exactly the words below 3 * 2^30; saturation at
    65504, NaN kept (sign too), signed zero kept, the FP16 subnormal range."""
    x = 1.0 + 3 * 2.0 ** -12                                # 3/4 of the way from 1 to 1 + 2^-10
    assert orc.fp16_sr(x, 3 * (1 << 30) - 1) == 0x3C01
    assert orc.fp16_sr(x, 3 * (1 << 30)) == 0x3C00
    assert orc.fp16_sr(70000.0, 0) == 0x7BFF and orc.fp16_sr(-float("inf"), 0) == 0xFBFF
    assert orc.fp16_sr(float("nan"), 0) & 0x7FFF == 0x7E00
    assert orc.fp16_sr(-0.0, 0) == 0x8000 and orc.fp16_sr(0.0, 0) == 0
    t = 2.0 ** -24 * 0.25                                    # a quarter of the smallest subnormal
    assert orc.fp16_sr(t, (1 << 30) - 1) == 1 and orc.fp16_sr(t, 1 << 30) == 0
    # the word of element e is the R4 word of index e
    xs = np.linspace(-3, 3, 37).astype(np.float32) * 1.001
    got = orc.sr_fp16(xs, 99)
    assert all(got[e] == orc.fp16_sr(float(xs[e]), orc.sr_word(99, e)) for e in range(len(xs)))


# ------------------------------------------------------------ PTQ block scales (reading R16)
_E2M1 = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], dtype=np.float64)


def _e2m1_rne_np(v):
    """Nearest E2M1 magnitude code, ties to the even code, saturating at 6 (numpy, FP64)."""
    m = np.minimum(np.abs(v), 6.0)
    d = np.abs(m[..., None] - _E2M1[None, :])
    best = d.min(axis=-1, keepdims=True)
    cand = np.where(np.isclose(d, best, rtol=0, atol=0), np.arange(8)[None, :], 99)
    even = np.where(cand % 2 == 0, cand, 99).min(axis=-1)
    anyc = cand.min(axis=-1)
    return np.where((cand < 99).sum(axis=-1) > 1, even, anyc)


def test_mse_block_scales_minimise_the_error(orc):
    """Each block's scale has the least FP64 squared error over all 126
    finite positive E4M3 scales (to FP32 rounding of the oracle's sums), never
    more than the max-based scale's, its codes are the RNE codes at that scale,
    and all-zero blocks keep scale 0."""
    rng = np.random.default_rng(60)
    rows, cols = 6, 64
    xf = rng.standard_normal((rows, cols)) * np.exp(rng.uniform(-3, 3, (rows, 1)))
    xf[0, :16] = 0.0                                                  # an all-zero block
    xf[1, 16] = 40.0                                                  # an outlier block
    x = _bf16(xf)
    q = orc.quantize_1d_mse(x)
    ref = orc.quantize_1d(x)
    xv = x.double().numpy()
    amax = float(np.abs(xv).max())
    s_enc = orc.tensor_scale(amax)
    dec = orc.decode_scale(amax)
    e4m3 = torch.arange(127, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    codes = _unpack(q["codes"], cols)
    differs = 0
    for r in range(rows):
        for b in range(cols // 16):
            blk = xv[r, 16 * b:16 * b + 16]
            c = int(q["sf"][orc.sf_offset(r, b, cols)])
            if not blk.any():
                assert c == 0 and not codes[r, 16 * b:16 * b + 16].any()
                continue
            errs = {}
            for cc in range(1, 127):
                rq = np.float32(s_enc) / np.float32(e4m3[cc])
                k = _e2m1_rne_np(blk * float(rq))
                rec = np.sign(blk) * _E2M1[k] * (e4m3[cc] * dec)
                errs[cc] = float(((blk - rec) ** 2).sum())
            best = min(errs.values())
            assert errs[c] <= best * (1 + 1e-5) + 1e-30, (r, b, c, errs[c], best)
            c_max = int(ref["sf"][orc.sf_offset(r, b, cols)])
            assert errs[c] <= errs[c_max] * (1 + 1e-5) + 1e-30
            differs += c != c_max
            kk = _e2m1_rne_np(blk * float(np.float32(s_enc) / np.float32(e4m3[c])))
            assert ((codes[r, 16 * b:16 * b + 16] & 7) == kk).all()
    assert differs > 0                                               # the search does change scales


def test_mse_block_scale_ties_keep_the_largest(orc):
    """Hand-worked blocks where several E4M3 scales rebuild the block exactly
    (error 0 in FP32): the oracle keeps the largest of them (R16), not the
    smallest or the first found."""
    with open(os.path.join(GOLD, "mse_ties.json")) as f:
        gold = json.load(f)
    for blk in gold["blocks"]:
        x = _bf16(np.array([blk["x"]], dtype=np.float64))
        q = orc.quantize_1d_mse(x, amax_in=blk["amax"])
        sf = int(q["sf"][orc.sf_offset(0, 0, 16)])
        assert sf == blk["sf"] != blk["smallest_tied_sf"], (blk["name"], sf)
        assert _unpack(q["codes"], 16)[0].tolist() == blk["codes"], blk["name"]
