"""GPU parity of the quantisers against the CPU oracle, bit for bit: packed
codes, the whole swizzled scale buffer (padding included) and the FP32 amax.
Shapes span several warps and CTAs, ragged row counts (not multiples of 128),
scale-column padding (cols/16 not a multiple of 4), empty and one-row
groups, and the degenerate all-zero tensor."""
import numpy as np
import pytest
import torch

from parity import np_u8, sf_rows_region

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from nvfp4_precision_02_b300 import binding, build
    build.build()
    binding.lib()
    assert torch.cuda.is_available()
    return binding


def _x(rows, cols, seed, scale=1.0, spread=0.0):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, cols, generator=g) * scale
    if spread:
        x = x * torch.exp(torch.rand(rows, 1, generator=g) * spread - spread / 2)
    return x.to(torch.bfloat16)


def _same(gpu_q, ref, rows, cols, check_amax=True):
    assert (np_u8(gpu_q.codes).reshape(ref["codes"].shape) == ref["codes"]).all(), "codes differ"
    assert (np_u8(gpu_q.sf) == ref["sf"]).all(), "scales differ"
    if check_amax:
        assert np_u8(gpu_q.amax)[0] == np.float32(ref["amax"]), "amax differs"


SHAPES_1D = [(1, 16), (15, 32), (128, 64), (129, 1040), (300, 256), (257, 48), (1000, 2048)]


@pytest.mark.parametrize("rows,cols", SHAPES_1D)
@pytest.mark.parametrize("mode", [0, 1])
def test_quantize_1d(B, orc, rows, cols, mode):
    x = _x(rows, cols, seed=rows * 7 + cols, spread=8.0)
    seed = 0xDEADBEEF12345 + rows
    q = B.quantize_1d(x.cuda(), mode=mode, seed=seed)
    torch.cuda.synchronize()
    _same(q, orc.quantize_1d(x, mode=mode, seed=seed), rows, cols)


def test_quantize_1d_supplied_amax_and_ld(B, orc):
    x = _x(200, 96, seed=3)
    big = torch.zeros(200, 128, dtype=torch.bfloat16)
    big[:, :96] = x
    xg = big.cuda()[:, :96]                                  # ld = 128 > cols
    amax_in = torch.tensor([7.5], device="cuda")
    q = B.quantize_1d(xg, mode=1, seed=9, amax_in=amax_in)
    torch.cuda.synchronize()
    _same(q, orc.quantize_1d(x, mode=1, seed=9, amax_in=7.5), 200, 96)


def test_quantize_1d_zero_tensor_and_denormals(B, orc):
    z = torch.zeros(130, 64, dtype=torch.bfloat16)
    q = B.quantize_1d(z.cuda())
    torch.cuda.synchronize()
    _same(q, orc.quantize_1d(z), 130, 64)
    assert (np_u8(q.codes) == 0).all() and (np_u8(q.sf) == 0).all()
    # tiny (subnormal bf16) and large magnitudes in one tensor: underflowing blocks
    x = _x(64, 64, seed=5)
    x[:8] = (torch.randn(8, 64) * 1e-39).to(torch.bfloat16)
    x[8:16] = (torch.randn(8, 64) * 3e4).to(torch.bfloat16)
    for mode in (0, 1):
        q = B.quantize_1d(x.cuda(), mode=mode, seed=1)
        torch.cuda.synchronize()
        _same(q, orc.quantize_1d(x, mode=mode, seed=1), 64, 64)


@pytest.mark.parametrize("mode", [0, 1])
def test_quantize_1d_grouped(B, orc, mode):
    cols = 80
    offsets = np.array([0, 0, 5, 6, 140, 140, 400, 401, 700], dtype=np.int64)   # empty, 1-row groups
    scales = np.array([1, 1, 3, 0.01, 1, 7, 1e-3, 2.0])
    rows = int(offsets[-1])
    x = (_x(rows, cols, seed=11).float() * torch.from_numpy(np.repeat(scales, np.diff(offsets))).float()[:, None]).to(torch.bfloat16)
    off = torch.from_numpy(offsets).cuda()
    q = B.quantize_1d_grouped(x.cuda(), off, mode=mode, seed=77)
    torch.cuda.synchronize()
    ref = orc.quantize_1d_grouped(x, offsets, mode=mode, seed=77)
    assert (np_u8(q.codes) == ref["codes"]).all()
    used = orc.group_sf_row(offsets, len(offsets) - 1)
    assert (sf_rows_region(np_u8(q.sf), used, cols) == sf_rows_region(ref["sf"], used, cols)).all()
    assert (np_u8(q.amax) == ref["amax"]).all()


SHAPES_2D = [(1, 16, 16), (1, 48, 80), (1, 128, 256), (1, 144, 1040), (3, 32, 64), (2, 2688 // 8, 1024 // 8)]


@pytest.mark.parametrize("batch,rows,cols", SHAPES_2D)
def test_quantize_2d(B, orc, batch, rows, cols):
    g = torch.Generator().manual_seed(rows + cols + batch)
    w = (torch.randn(batch, rows, cols, generator=g) * 0.02 *
         torch.exp(torch.rand(batch, rows, cols, generator=g) * 6 - 3)).to(torch.bfloat16)
    qw, qt, tile = B.quantize_2d(w.cuda(), want_t=True, want_tile_sf=True)
    torch.cuda.synchronize()
    ref = orc.quantize_2d(w)
    assert (np_u8(qw.codes).reshape(ref["codes"].shape) == ref["codes"]).all()
    assert (np_u8(qw.sf) == ref["sf"]).all()
    assert (np_u8(qt.codes).reshape(ref["codes_t"].shape) == ref["codes_t"]).all()
    assert (np_u8(qt.sf) == ref["sf_t"]).all()
    assert (np_u8(tile) == ref["tile_sf"]).all()
    assert (np_u8(qw.amax) == ref["amax"]).all()


@pytest.mark.parametrize("tokens,cols", [(16, 1), (64, 24), (80, 130), (1024, 300), (48, 8), (1040, 520),
                                         (8192, 1536)])
@pytest.mark.parametrize("mode", [0, 1])
def test_rht_quantize(B, orc, tokens, cols, mode):
    """RHT + quantise and the RHT amax equal the oracle's; rows of 16-byte
    multiples (cols % 8 == 0) take the persistent streaming kernel (a last
    tile of 16 tokens and 8 channels at 1040 x 520; several tiles per CTA at
    8192 x 1536), others one CTA per tile."""
    x = _x(tokens, cols, seed=tokens * 3 + cols, spread=4.0)
    mask = 0xB5A3 ^ tokens
    q = B.rht_quantize(x.cuda(), mask, mode=mode, seed=1234567)
    a = B.rht_amax(x.cuda(), mask)
    torch.cuda.synchronize()
    ref = orc.rht_quantize(x, mask, mode=mode, seed=1234567)
    _same(q, ref, cols, tokens)
    assert np_u8(a)[0] == np.float32(ref["amax"])


def test_amax_batched(B, orc):
    w = _x(3 * 48, 64, seed=2).reshape(3, 48, 64)
    a = B.amax(w.cuda())
    torch.cuda.synchronize()
    for b in range(3):
        assert np_u8(a)[b] == np.float32(orc.amax(w[b]))


def test_device_status_clean(B):
    assert B.device_status() == 0


def test_quantize_1d_ties_signed_zeros_saturation(B, orc):
    """Blocks whose largest magnitude is 6 under a tensor amax of 2688 get
    scale 1.0 and element multiplier 1, so every value below reaches the E2M1
    rounding unchanged: the seven ties of the grid, negative values that
    round to zero (code 0x8), -0, and values beyond 6 that saturate."""
    rows = [
        [6, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.1, -0.25, -5, 5.5, 0.5, 1.0, -0.0, -6],
        [6, -0.75, -1.25, -1.75, -2.5, -3.5, -0.0001, 0.0001, -3, 4.5, 2.75, -0.3, 0.2, 1.4, -1.6, 6],
        [-6, 0.2499, 0.2501, 0.7499, 0.7501, 4.999, 5.001, -5.001, -0.2501, 3.49, 3.51, 1.74, 1.76, 0, 0, 0],
    ]
    x = torch.tensor(rows, dtype=torch.float32).repeat(5, 2).to(torch.bfloat16)   # 15 x 32
    amax_in = torch.tensor([2688.0], device="cuda")
    for mode in (0, 1):
        q = B.quantize_1d(x.cuda(), mode=mode, seed=5, amax_in=amax_in)
        torch.cuda.synchronize()
        _same(q, orc.quantize_1d(x, mode=mode, seed=5, amax_in=2688.0), 15, 32)
    # 2D tiles and the transposed copy take the same conversion
    w = torch.tensor(rows, dtype=torch.float32).repeat(6, 1)[:16].to(torch.bfloat16)    # 16 x 16
    qw, qt, _ = B.quantize_2d(w.cuda(), want_t=True, amax_in=amax_in)
    torch.cuda.synchronize()
    ref = orc.quantize_2d(w, amax_in=[2688.0])
    assert (np_u8(qw.codes).reshape(ref["codes"].shape) == ref["codes"]).all()
    assert (np_u8(qt.codes).reshape(ref["codes_t"].shape) == ref["codes_t"]).all()


@pytest.mark.parametrize("batch,rows,cols", SHAPES_2D + [(5, 64, 1040), (4, 16, 48), (7, 336, 2064)])
@pytest.mark.parametrize("supplied", [False, True])
def test_quantize_2d_w_only(B, orc, batch, rows, cols, supplied):
    """W without W^T (the expert-weight form): bytes, scales, tile scales and
    amax equal the oracle's, with the amax computed or supplied in another
    buffer (then copied into the output), and column counts that leave a
    partial 64-column block (1040, 2064) or fit in one (48)."""
    g = torch.Generator().manual_seed(rows * 3 + cols + batch)
    w = (torch.randn(batch, rows, cols, generator=g) * 0.02 *
         torch.exp(torch.rand(batch, 1, 1, generator=g) * 6 - 3)).to(torch.bfloat16)
    ref = orc.quantize_2d(w, want_t=False)
    am = torch.from_numpy(np.asarray(ref["amax"], dtype=np.float32).copy()).cuda() if supplied else None
    qw, qt, tile = B.quantize_2d(w.cuda(), want_t=False, want_tile_sf=True, amax_in=am)
    torch.cuda.synchronize()
    assert qt is None
    assert (np_u8(qw.codes).reshape(ref["codes"].shape) == ref["codes"]).all()
    assert (np_u8(qw.sf) == ref["sf"]).all()
    assert (np_u8(tile) == ref["tile_sf"]).all()
    assert (np_u8(qw.amax) == ref["amax"]).all()
    assert B.device_status() == 0


@pytest.mark.parametrize("batch,rows,cols", [(1, 48, 80), (2, 144, 1040), (5, 320, 256), (3, 64, 64),
                                             (7, 2688 // 8, 1024 // 8), (4, 16, 3072),
                                             (40, 512, 2048), (2, 2048, 8192), (1, 5120, 2048), (3, 5120, 2048)])
def test_quantize_2d_fused(B, orc, batch, rows, cols):
    """One-pass (amax in the same cooperative launch) 2D quantisation gives
    the oracle's bytes, for one entry and several, one 16-row strip per entry
    and many, column counts below one 256-column unit (64, 80, 128) and ones
    that leave a partial unit (1040), entries of fewer units than the grid
    has CTAs, Ultra expert weights (5120 x 2048: the largest entry kept on
    chip, 17 or 18 units per CTA) and an entry too large for that
    (2048 x 8192: the path that re-reads through L2)."""
    g = torch.Generator().manual_seed(batch * 1000 + rows + cols)
    w = (torch.randn(batch, rows, cols, generator=g) * 0.02 *
         torch.exp(torch.rand(batch, 1, 1, generator=g) * 6 - 3)).to(torch.bfloat16)
    ws = torch.full((B.quantize_2d_fused_workspace(batch),), 0xAB, dtype=torch.uint8, device="cuda")
    for _ in range(2):   # the call re-zeroes its workspace
        qw, tile = B.quantize_2d_fused(w.cuda(), want_tile_sf=True, workspace=ws)
        torch.cuda.synchronize()
        ref = orc.quantize_2d(w, want_t=False)
        assert (np_u8(qw.amax) == ref["amax"]).all()
        assert (np_u8(qw.codes).reshape(ref["codes"].shape) == ref["codes"]).all()
        assert (np_u8(qw.sf) == ref["sf"]).all()
        assert (np_u8(tile) == ref["tile_sf"]).all()
    assert B.device_status() == 0


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("cols", [48, 300])
def test_rht_quantize_grouped(B, orc, mode, cols):
    """Expert-segmented RHT + quantisation (wgrad inputs of the expert GEMMs):
    every expert's tokens zero-padded to a multiple of 64 at the running sum of
    padded counts, its own amax; bytes equal the oracle's on the used columns,
    with empty and one-token experts and a capacity larger than needed."""
    offsets = np.array([0, 0, 1, 70, 70, 200, 265], dtype=np.int64)
    counts = np.diff(offsets)
    rows = int(offsets[-1])
    g = torch.Generator().manual_seed(cols + mode)
    scale = torch.from_numpy(np.repeat([1, 1, 4, 1, 0.01, 2.0], counts)).float()[:, None]
    x = (torch.randn(rows, cols, generator=g) * scale).to(torch.bfloat16)
    off = torch.from_numpy(offsets).cuda()
    kt = B.group_k_capacity(rows, len(counts))
    assert kt % 64 == 0 and kt >= ((counts + 63) // 64 * 64).sum()
    q = B.rht_quantize_grouped(x.cuda(), off, 0x2D71, mode=mode, seed=4321)
    torch.cuda.synchronize()
    ref = orc.rht_quantize_grouped(x, offsets, kt, 0x2D71, mode=mode, seed=4321)
    used = orc.group_k_offset(offsets, len(counts))
    assert (np_u8(q.amax) == ref["amax"]).all()
    assert (np_u8(q.codes)[:, :used // 2] == ref["codes"][:, :used // 2]).all()
    sf = np_u8(q.sf)
    for c in range(cols):
        for b in range(used // 16):
            off_b = orc.sf_offset(c, b, kt)
            assert sf[off_b] == ref["sf"][off_b], (c, b)
    # the supplied-amax path gives the same bytes
    q2 = B.rht_quantize_grouped(x.cuda(), off, 0x2D71, mode=mode, seed=4321, amax_in=q.amax.clone())
    torch.cuda.synchronize()
    assert (np_u8(q2.codes)[:, :used // 2] == ref["codes"][:, :used // 2]).all()
    assert B.device_status() == 0


@pytest.mark.parametrize("n", [1, 7, 1000003])
def test_sr_fp16(B, orc, n):
    """FP32 -> FP16 stochastic rounding (SSM cache) equals the oracle bit for
    bit: wide exponent spread, the FP16 subnormal range, signed zeros,
    saturation, infinities and NaN; aligned (vector) and offset (element)
    paths."""
    rng = np.random.default_rng(n)
    x = (rng.standard_normal(n) * np.exp(rng.uniform(-25, 12, n))).astype(np.float32)
    special = np.array([0.0, -0.0, 65504.0, 70000.0, -np.inf, np.nan, 2.0 ** -25, -3e-7, 6e-8, 1.0 + 2.0 ** -11],
                       dtype=np.float32)
    x[:min(n, len(special))] = special[:min(n, len(special))]
    xt = torch.from_numpy(x).cuda()
    got = B.sr_fp16(xt, 0xC0FFEE)
    torch.cuda.synchronize()
    ref = orc.sr_fp16(x, 0xC0FFEE)
    assert (got.cpu().numpy().view(np.uint16) == ref).all()
    if n > 1:
        got1 = B.sr_fp16(xt[1:], 0xC0FFEE)                 # 4-byte offset: element path
        torch.cuda.synchronize()
        assert (got1.cpu().numpy().view(np.uint16) == orc.sr_fp16(x[1:], 0xC0FFEE)).all()
    assert B.device_status() == 0


@pytest.mark.parametrize("rows,cols", [(1, 16), (37, 64), (300, 1040)])
def test_quantize_1d_mse(B, orc, rows, cols):
    """PTQ block scales by minimum squared error: codes and scales equal the
    oracle's bytes (all 126 scales tried per block), including an all-zero
    block and outlier blocks; supplied amax gives the same bytes."""
    g = torch.Generator().manual_seed(rows * 13 + cols)
    x = torch.randn(rows, cols, generator=g) * torch.exp(torch.rand(rows, 1, generator=g) * 6 - 3)
    x[0, :16] = 0.0
    if cols >= 64:
        x[rows // 2, 20] = 50.0
    x = x.to(torch.bfloat16)
    q = B.quantize_1d_mse(x.cuda())
    torch.cuda.synchronize()
    ref = orc.quantize_1d_mse(x)
    _same(q, ref, rows, cols)
    q2 = B.quantize_1d_mse(x.cuda(), amax_in=q.amax.clone())
    torch.cuda.synchronize()
    _same(q2, ref, rows, cols)
    assert B.device_status() == 0


@pytest.mark.parametrize("tokens,cols", [(16, 1), (80, 130), (1024, 300), (1040, 520), (8192, 1536)])
def test_dual_amax_and_zero_code_count(B, orc, tokens, cols):
    """One read gives both tensor amaxes of a gradient (plain and after the
    RHT), each equal to the oracle's; the zero-code count of the SR-quantised
    gradient equals the count of zero-magnitude codes in the oracle's bytes."""
    x = _x(tokens, cols, seed=tokens + cols, scale=1e-3, spread=6.0)
    mask = 0x51C3
    a = B.dual_amax(x.cuda(), mask)
    torch.cuda.synchronize()
    got = np_u8(a)
    assert got[0] == np.float32(orc.amax(x)) and got[1] == np.float32(orc.rht_amax(x, mask))
    if cols % 16 == 0:
        q = B.quantize_1d(x.cuda(), mode=1, seed=3, amax_in=a[:1])
        n0 = B.count_zero_codes(q)
        torch.cuda.synchronize()
        ref = orc.quantize_1d(x, mode=1, seed=3, amax_in=float(got[0]))
        codes = ref["codes"]
        want = int(((codes & 7) == 0).sum() + (((codes >> 4) & 7) == 0).sum())
        assert int(n0.item()) == want
    assert B.device_status() == 0


@pytest.mark.parametrize("tokens,cols", [(16, 16), (64, 272), (80, 1040), (1040, 320), (208, 48)])
def test_dual_sr_quantize(B, orc, tokens, cols):
    """One read of a gradient gives both stochastically rounded operands: the
    row operand equals the oracle's 1x16 SR quantisation (seed_row, amax of
    |dy|) and the transposed operand the oracle's RHT + SR quantisation
    (seed_rht, amax of |RHT(dy)|), bytes and padding included; the zero count
    is the number of zero-magnitude codes of the row operand.  Shapes cover
    a partial 64-token tile, a partial 256-channel tile, rows and columns not
    multiples of 128 and a scale-column padding."""
    _dual_sr_case(B, orc, tokens, cols, 0)


@pytest.mark.parametrize("tokens,cols", [(80, 272), (1040, 48)])
def test_dual_sr_quantize_strided_rows(B, orc, tokens, cols):
    """The same with rows 8 bytes past a 16-byte multiple apart (ld = cols +
    4), which the per-tile kernel takes instead of the streaming one."""
    _dual_sr_case(B, orc, tokens, cols, 4)


@pytest.mark.parametrize("tokens,cols", [(80, 272), (1040, 528)])
def test_rht_paths_in_the_subnormal_range(B, orc, tokens, cols):
    """Inputs near the bottom of the FP32 range (|x| ~ 1e-38, some of them
    bf16 subnormals): the transform's sums and its factor 1/4 produce FP32
    subnormals, which every RHT path (amax, both amaxes, RNE, SR, the dual
    encoder) must round exactly as the oracle's FP32 arithmetic does."""
    x = _x(tokens, cols, seed=5 * tokens + cols, scale=2e-38, spread=3.0)
    assert (x.float().abs() < 1.1754944e-38).any()
    mask = 0x6A39
    a = B.dual_amax(x.cuda(), mask)
    r = B.rht_amax(x.cuda(), mask)
    torch.cuda.synchronize()
    got = np_u8(a)
    assert got[0] == np.float32(orc.amax(x)) and got[1] == np.float32(orc.rht_amax(x, mask))
    assert np_u8(r)[0] == got[1]
    for mode in (0, 1):
        q = B.rht_quantize(x.cuda(), mask, mode=mode, seed=99)
        torch.cuda.synchronize()
        _same(q, orc.rht_quantize(x, mask, mode=mode, seed=99), cols, tokens)
    _dual_sr_case(B, orc, tokens, cols, 0, scale=2e-38, spread=3.0)


def _dual_sr_case(B, orc, tokens, cols, pad, scale=1e-3, spread=6.0):
    x = _x(tokens, cols, seed=7 * tokens + cols, scale=scale, spread=spread)
    mask, s_row, s_rht = 0x2D96, 7, 7 ^ 0x9E3779B97F4A7C15
    xd = x.cuda()
    if pad:
        wide = torch.zeros(tokens, cols + pad, dtype=torch.bfloat16, device="cuda")
        wide[:, :cols] = xd
        xd = wide[:, :cols]
    a = B.dual_amax(xd, mask)
    zc = torch.full((1,), -1, dtype=torch.int64, device="cuda")
    qr, qt = B.dual_sr_quantize(xd, mask, s_row, s_rht, a, zero_count=zc)
    torch.cuda.synchronize()
    got = np_u8(a)
    ref_r = orc.quantize_1d(x, mode=1, seed=s_row, amax_in=float(got[0]))
    ref_t = orc.rht_quantize(x, mask, mode=1, seed=s_rht, amax_in=float(got[1]))
    _same(qr, ref_r, tokens, cols)
    _same(qt, ref_t, cols, tokens)
    codes = ref_r["codes"]
    assert int(zc.item()) == int(((codes & 7) == 0).sum() + (((codes >> 4) & 7) == 0).sum())
    assert B.device_status() == 0
