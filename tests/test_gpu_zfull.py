"""Full-size parity: one step of the Super-shaped and of the Ultra-shaped
workload, in exactly the launch configuration the benchmark times (its
Workload object, CTA-pair GEMMs), checked against the oracle on sampled rows
and outputs.  The Super step covers the Super in_proj fprop (X 8192 x 6144
with outlier channels, W 18560 x 6144), its backward (dY 8192 x 18560 with
SR, dgrad over K = 18560, RHT wgrad over 8192 tokens) and the Super LatentMoE
(latent 1024 -> expert hidden 2688 -> 1024, 180224 routed rows); the Ultra
step covers the same rows at the Ultra shapes.  Sampled rows and columns
include the 128-row and 256-row tile edges and the last, possibly partial,
tile of every axis (N = 18560 and 2688 end on half a 256-column tile).

- Tensor amaxes (X, W, dY, max |RHT(dY)|, RHT(X), every sampled expert) equal
  the oracle's over the whole operand.
- Codes and block scales of sampled rows of every quantised operand equal the
  oracle's bit for bit.  Those rows carry the whole-operand amax and their
  SR indices in the whole output.
- Sampled GEMM outputs lie within the bound: 1e-5 * sum |a b|, plus one bf16
  rounding for bf16 outputs.
- The per-expert amax that the up-projection's epilogue writes equals the
  largest stored |H| of every expert.
- The down-projection is checked on a seeded H of the same shape, so that
  none of the oracle's inputs comes from a GPU result."""
import types

import numpy as np
import pytest
import torch

import fullsize as fs
from parity import gemm_within_bound

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

RNE, SR = 0, 1
NS = 24            # sampled rows per operand of a dense GEMM
NS_E = 8           # sampled rows per operand of one expert
BOUNDARY = (127, 128, 255, 256, 257)     # rows at 128-row tile and 256-row pair-tile edges


def edges(n: int):
    """BOUNDARY plus the indices around the start of the last 128- and
    256-wide tile of an axis of length n, and its last index."""
    out = set(BOUNDARY) | {n - 1}
    for t in (128, 256):
        last = (n - 1) // t * t
        out |= {last - 1, last}
    return tuple(sorted(i for i in out if 0 <= i < n))


@pytest.fixture(scope="module", params=["super", "ultra"])
def run(orc, request):
    from nvfp4_precision_02_b300 import binding as B, build
    build.build()
    B.lib()
    assert torch.cuda.is_available()
    import bench
    wk = bench.Workload(request.param, torch.device("cuda", 0))
    wk.step()
    torch.cuda.synchronize()
    assert B.device_status() == 0
    r = types.SimpleNamespace(wk=wk, B=B, host={})
    yield r
    r.host.clear()
    del r.wk, wk
    torch.cuda.empty_cache()


def _host(run, name):
    if name not in run.host:
        run.host[name] = fs.bits(getattr(run.wk, name))
    return run.host[name]


def _gpu_rows(orc, q, ids, cols, batch=None, sf=None, sf_rows=None):
    """Codes and block scales of rows `ids` of a GPU-quantised operand."""
    idx = torch.as_tensor(ids, device=q.codes.device)
    codes = (q.codes[batch] if batch is not None else q.codes)[idx].cpu().numpy()
    sf = q.sf.cpu().numpy() if sf is None else sf
    return codes, fs.scale_rows(orc, sf, ids if sf_rows is None else sf_rows, cols)


def _check_rows(name, orc, orows, q, ids, cols, **kw):
    codes, scales = _gpu_rows(orc, q, ids, cols, **kw)
    fs.assert_rows_equal(name, orows, codes, scales, ids)


def _check_gemm(name, orc, out, m_ids, n_ids, arows, brows, bf16):
    mi = torch.as_tensor(m_ids, device=out.device)
    ni = torch.as_tensor(n_ids, device=out.device)
    sub = out[mi][:, ni].float().cpu().numpy()
    ref, absum = orc.gemm(arows.dequantized(orc), brows.dequantized(orc))
    ok, worst = gemm_within_bound(sub, ref, absum, bf16)
    bad = np.argwhere(~ok)
    assert ok.all(), (f"{name}: {len(bad)} of {ok.size} sampled outputs out of bound (worst ratio {worst:.3g}), "
                      f"first {[(int(m_ids[i]), int(n_ids[j])) for i, j in bad[:4]]}")
    assert np.abs(ref).max() > 0


def test_fprop_full_size(run, orc):
    wk = run.wk
    T, K, N = wk.dense.tokens, wk.dense.hidden, wk.dense.out
    xb, wb = _host(run, "x"), _host(run, "w")
    ax, aw = orc.amax(xb), orc.amax(wb)
    assert float(wk.qx.amax[0]) == ax and float(wk.qw.amax[0]) == aw
    m_ids = fs.sample_ids(T, NS, 1, must=edges(T))
    n_ids = fs.sample_ids(N, NS, 2, must=edges(N))
    xr = fs.rows_1d(orc, xb[m_ids], m_ids, K, ax, RNE)
    wr = fs.rows_2d(orc, lambda n0: wb[n0:n0 + 16], n_ids, K, aw)
    _check_rows("X (1x16 RNE)", orc, xr, wk.qx, m_ids, K)
    _check_rows("W (16x16)", orc, wr, wk.qw, n_ids, K)
    _check_gemm("fprop Y = X.W^T", orc, wk.y, m_ids, n_ids, xr, wr, bf16=True)


def test_dgrad_full_size(run, orc):
    wk = run.wk
    T, K, N = wk.dense.tokens, wk.dense.hidden, wk.dense.out
    dyb, wb = _host(run, "dy"), _host(run, "w")
    ady, aw = orc.amax(dyb), orc.amax(wb)
    assert float(wk.dy_amax[0]) == ady and float(wk.qdy.amax[0]) == ady
    m_ids = fs.sample_ids(T, NS, 3, must=edges(T))
    k_ids = fs.sample_ids(K, NS, 4, must=edges(K))
    dyr = fs.rows_1d(orc, dyb[m_ids], m_ids, N, ady, SR, wk.seed)
    wtr = fs.rows_2d(orc, lambda k0: np.ascontiguousarray(wb[:, k0:k0 + 16].T), k_ids, N, aw)
    _check_rows("dY (1x16 SR)", orc, dyr, wk.qdy, m_ids, N)
    _check_rows("W^T (16x16)", orc, wtr, wk.qwt, k_ids, N)
    _check_gemm("dgrad dX = dY.W", orc, wk.dx, m_ids, k_ids, dyr, wtr, bf16=True)


def test_wgrad_full_size(run, orc):
    wk = run.wk
    T, K, N = wk.dense.tokens, wk.dense.hidden, wk.dense.out
    dyb, xb = _host(run, "dy"), _host(run, "x")
    ardy, arx = orc.rht_amax(dyb, wk.mask), orc.rht_amax(xb, wk.mask)
    assert float(wk.dy_amax[1]) == ardy and float(wk.sdy.amax[0]) == ardy
    assert float(wk.sx.amax[0]) == arx
    n_ids = fs.sample_ids(N, NS, 5, must=edges(N))
    k_ids = fs.sample_ids(K, NS, 6, must=edges(K))
    sdyr = fs.rows_rht(orc, np.ascontiguousarray(dyb[:, n_ids]), n_ids, T, ardy, wk.mask, SR, wk.wseed)
    sxr = fs.rows_rht(orc, np.ascontiguousarray(xb[:, k_ids]), k_ids, T, arx, wk.mask, RNE, 0)
    _check_rows("RHT(dY)^T (SR)", orc, sdyr, wk.sdy, n_ids, T)
    _check_rows("RHT(X)^T (RNE)", orc, sxr, wk.sx, k_ids, T)
    _check_gemm("wgrad dW = RHT(dY)^T.RHT(X)", orc, wk.dw, n_ids, k_ids, sdyr, sxr, bf16=False)


def _experts(counts, seed):
    """The largest expert, the smallest non-empty one and three seeded others."""
    nz = np.flatnonzero(counts)
    rng = np.random.default_rng(seed)
    pick = {int(np.argmax(counts)), int(nz[np.argmin(counts[nz])])}
    pick |= set(int(g) for g in rng.choice(nz, size=min(3, len(nz)), replace=False))
    return sorted(pick)


def _expert_check(run, orc, name, x, qx, qx_sf, offsets, g, w_e, qw, out, seed):
    """Rows of expert g's activations (grouped 1x16 RNE, own amax), rows of
    its weight (16x16, own amax) and the sampled outputs of its GEMM.
    qx_sf: host copy of the activations' block scales."""
    B = run.B
    o0, o1 = int(offsets[g]), int(offsets[g + 1])
    cols = x.shape[1]
    xb = fs.bits(x[o0:o1])
    am = orc.amax(xb)
    assert float(qx.amax[g]) == am, (name, g)
    loc = fs.sample_ids(o1 - o0, NS_E, seed, must=edges(o1 - o0))
    rows = loc + o0
    xr = fs.rows_1d(orc, xb[loc], rows, cols, am, RNE)
    p = orc.group_sf_row(offsets, g)
    _check_rows(f"{name} activations, expert {g}", orc, xr, qx, rows, cols, sf=qx_sf, sf_rows=loc + p)
    wb = fs.bits(w_e[g])
    n_out = wb.shape[0]
    aw = orc.amax(wb)
    assert float(qw.amax[g]) == aw, (name, g)
    n_ids = fs.sample_ids(n_out, NS_E, seed + 1, must=edges(n_out))
    wr = fs.rows_2d(orc, lambda n0: wb[n0:n0 + 16], n_ids, cols, aw)
    nsf = B.sf_bytes(n_out, cols)
    _check_rows(f"{name} weight, expert {g}", orc, wr, qw, n_ids, cols, batch=g,
                sf=qw.sf[g * nsf:(g + 1) * nsf].cpu().numpy())
    _check_gemm(f"{name} GEMM, expert {g}", orc, out, rows, n_ids, xr, wr, bf16=True)


def test_moe_up_full_size(run, orc):
    wk = run.wk
    offsets = wk.routing.offsets.cpu().numpy().astype(np.int64)
    counts = np.diff(offsets)
    qa_sf = wk.qa.sf.cpu().numpy()
    for g in _experts(counts, 7):
        _expert_check(run, orc, "up", wk.a, wk.qa, qa_sf, offsets, g, wk.w_up, wk.qwu, wk.h, seed=10 + g)
    # the epilogue's per-expert amax of H is the largest stored |H| of each expert
    amax_h = wk.qh.amax.cpu().numpy()
    for g in np.flatnonzero(counts):
        o0, o1 = int(offsets[g]), int(offsets[g + 1])
        assert amax_h[g] == float(wk.h[o0:o1].abs().max()), g


def test_moe_down_full_size(run, orc):
    """The down-projection's grouped quantiser and GEMM on a seeded H of the
    step's shape and routing, with the step's quantised W_down."""
    from nvfp4_precision_02_b300 import workloads as wl
    wk, B = run.wk, run.B
    R, Hh, L = wk.R, wk.moe.expert_hidden, wk.moe.latent
    h = wl.normal_bf16((R, Hh), 0.5, 2024, device=wk.a.device)
    qh = B.quantize_1d_grouped(h, wk.offsets)
    o = B.grouped_gemm(qh, wk.offsets, wk.qwd, L, B.OUT_BF16)
    if o.is_cuda:
        torch.cuda.synchronize()
    assert B.device_status() == 0
    offsets = wk.routing.offsets.cpu().numpy().astype(np.int64)
    counts = np.diff(offsets)
    qh_sf = qh.sf.cpu().numpy()
    for g in _experts(counts, 8):
        _expert_check(run, orc, "down", h, qh, qh_sf, offsets, g, wk.w_down, wk.qwd, o, seed=20 + g)


SSM_ELEMENTS = 256 * 256 * 64 * 128     # SSM cache: sequences x heads x head dim x state


def test_expert_backward_full_size(run, orc):
    """Grouped backward of the up-projection at full size on a seeded dH:
    the grouped SR quantiser of dH, the grouped dgrad dA = dH . W_up against
    the per-expert W_up^T of the batched 2D quantiser, the expert-segmented
    RHT quantisers of dH (SR) and A (RNE), and the K-grouped FP32 wgrad
    dW_up = RHT(dH)^T . RHT(A) per expert."""
    from nvfp4_precision_02_b300 import workloads as wl
    wk, B = run.wk, run.B
    R, Hh, L, E = wk.R, wk.moe.expert_hidden, wk.moe.latent, wk.moe.experts
    dh = wl.normal_bf16((R, Hh), 1e-3, 2025, device=wk.a.device)
    qdh = B.quantize_1d_grouped(dh, wk.offsets, B.SR, wk.seed)
    _, qwt, _ = B.quantize_2d(wk.w_up, want_t=True)
    da = B.grouped_gemm(qdh, wk.offsets, qwt, L, B.OUT_BF16)
    kt = B.group_k_capacity(R, E)
    sdh = B.rht_quantize_grouped(dh, wk.offsets, wk.mask, B.SR, wk.wseed, kt=kt)
    sa = B.rht_quantize_grouped(wk.a, wk.offsets, wk.mask, B.RNE, 0, kt=kt)
    dw = B.grouped_gemm_k(sdh, sa, wk.offsets, B.OUT_FP32)
    if dw.is_cuda:
        torch.cuda.synchronize()
    assert B.device_status() == 0
    offsets = wk.routing.offsets.cpu().numpy().astype(np.int64)
    counts = np.diff(offsets)
    qdh_sf, sdh_sf, sa_sf = qdh.sf.cpu().numpy(), sdh.sf.cpu().numpy(), sa.sf.cpu().numpy()
    nsf = B.sf_bytes(L, Hh)
    for g in _experts(counts, 9):
        o0, o1 = int(offsets[g]), int(offsets[g + 1])
        dhb = fs.bits(dh[o0:o1])
        # dgrad operands and outputs
        am = orc.amax(dhb)
        assert float(qdh.amax[g]) == am, g
        loc = fs.sample_ids(o1 - o0, NS_E, 30 + g, must=edges(o1 - o0))
        rows = loc + o0
        dr = fs.rows_1d(orc, dhb[loc], rows, Hh, am, SR, wk.seed)
        _check_rows(f"dH (grouped SR), expert {g}", orc, dr, qdh, rows, Hh, sf=qdh_sf,
                    sf_rows=loc + orc.group_sf_row(offsets, g))
        wub = fs.bits(wk.w_up[g])
        aw = orc.amax(wub)
        assert float(qwt.amax[g]) == aw, g
        k_ids = fs.sample_ids(L, NS_E, 40 + g, must=edges(L))
        wtr = fs.rows_2d(orc, lambda k0: np.ascontiguousarray(wub[:, k0:k0 + 16].T), k_ids, Hh, aw)
        _check_rows(f"W_up^T, expert {g}", orc, wtr, qwt, k_ids, Hh, batch=g,
                    sf=qwt.sf[g * nsf:(g + 1) * nsf].cpu().numpy())
        _check_gemm(f"grouped dgrad, expert {g}", orc, da, rows, k_ids, dr, wtr, bf16=True)
        # wgrad operands (expert segments along K) and outputs
        ko = orc.group_k_offset(offsets, g)
        segh = fs.padded_segment(dhb, 0, o1 - o0)
        sega = fs.padded_segment(fs.bits(wk.a[o0:o1]), 0, o1 - o0)
        kp = segh.shape[0]
        arh, ara = orc.rht_amax(segh, wk.mask), orc.rht_amax(sega, wk.mask)
        assert float(sdh.amax[g]) == arh and float(sa.amax[g]) == ara, g
        n_ids = fs.sample_ids(Hh, NS_E, 50 + g, must=edges(Hh))
        c_ids = fs.sample_ids(L, NS_E, 60 + g, must=edges(L))
        hr = fs.rows_rht(orc, np.ascontiguousarray(segh[:, n_ids]), n_ids, kp, arh, wk.mask, SR, wk.wseed,
                         index_stride=kt, index_offset=ko)
        ar = fs.rows_rht(orc, np.ascontiguousarray(sega[:, c_ids]), c_ids, kp, ara, wk.mask, RNE, 0,
                         index_stride=kt, index_offset=ko)
        for name, q, sf, ids, orows in (("RHT(dH)^T", sdh, sdh_sf, n_ids, hr), ("RHT(A)^T", sa, sa_sf, c_ids, ar)):
            idx = torch.as_tensor(ids, device=q.codes.device)
            codes = q.codes[idx].cpu().numpy()[:, ko // 2:(ko + kp) // 2]
            scales = fs.scale_rows(orc, sf, ids, kt, b0=ko // 16, b1=(ko + kp) // 16)
            fs.assert_rows_equal(f"{name} segment, expert {g}", orows, codes, scales, ids)
        _check_gemm(f"K-grouped wgrad, expert {g}", orc, dw, g * Hh + n_ids, c_ids, hr, ar, bf16=False)


def test_ptq_mse_scales_full_size(run, orc):
    """Minimum-squared-error block scales of the in_proj weight at full size
    (with the weight's tensor amax), on sampled rows."""
    wk, B = run.wk, run.B
    N, K = wk.dense.out, wk.dense.hidden
    aw = orc.amax(_host(run, "w"))
    amax_in = torch.tensor([aw], dtype=torch.float32, device=wk.w.device)
    q = B.quantize_1d_mse(wk.w, amax_in=amax_in)
    ids = fs.sample_ids(N, NS, 70, must=edges(N))
    wb = _host(run, "w")
    orows = fs.OracleRows(len(ids), K, aw)
    for i, n in enumerate(ids):
        o = orc.quantize_1d_mse(np.ascontiguousarray(wb[n:n + 1]), amax_in=aw)
        orows.codes[i] = o["codes"][0]
        orows.scales[i] = fs.scale_rows(orc, o["sf"], [0], K)[0]
    _check_rows("W (MSE block scales)", orc, orows, q, ids, K)


def test_sr_fp16_full_size(run, orc):
    """FP16 stochastic rounding of an SSM-cache-sized FP32 tensor: sampled
    elements equal the oracle's rounding with the word of their index."""
    B = run.B
    dev = run.wk.a.device
    g = torch.Generator(device=dev)
    g.manual_seed(12)
    x = torch.randn(SSM_ELEMENTS, generator=g, device=dev)
    out = B.sr_fp16(x, 5)
    e = fs.sample_ids(SSM_ELEMENTS, 4096, 13)
    idx = torch.as_tensor(e, device=dev)
    xs = x[idx].cpu().numpy()
    got = out[idx].view(torch.int16).cpu().numpy().view(np.uint16)
    exp = np.array([orc.fp16_sr(float(v), orc.sr_word(5, int(i))) for v, i in zip(xs, e)], dtype=np.uint16)
    bad = np.flatnonzero(got != exp)
    assert bad.size == 0, f"{bad.size} of {len(e)} sampled elements differ, first {e[bad[:4]].tolist()}"


def test_zero_code_count_full_size(run, orc):
    """The zero-code counter over the SR-quantised dY equals a count of the
    zero-magnitude nibbles of the same codes."""
    wk, B = run.wk, run.B
    cnt = int(B.count_zero_codes(wk.qdy).item())
    assert int(wk.dy_zeros.item()) == cnt        # the count the step's dual SR quantiser returned
    c = wk.qdy.codes.cpu().numpy()
    assert cnt == int(((c & 7) == 0).sum()) + int((((c >> 4) & 7) == 0).sum())
    assert 0 < cnt < c.size * 2
