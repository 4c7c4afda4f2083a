"""GPU parity of the NVFP4 GEMMs (tcgen05 block-scaled MMA) against the FP64
GEMM of the oracle's own dequantised operands: every output element must
satisfy |gpu - ref| <= 1e-5 * sum_k |a_k b_k| (plus one bf16 rounding for a
bf16 output).  The oracle quantises the same bf16 inputs itself; nothing it
uses comes from the CUDA path."""
import numpy as np
import pytest
import torch

from parity import gemm_within_bound, np_u8

pytestmark = pytest.mark.gpu


@pytest.fixture(params=["pair", "single"], autouse=True)
def gemm_kernel(request, monkeypatch):
    """Every GEMM test runs on both kernels: CTA pairs (cta_group::2, the
    default) and single CTAs (NVFP4_GEMM_PAIR=0)."""
    if request.param == "single":
        monkeypatch.setenv("NVFP4_GEMM_PAIR", "0")
    else:
        monkeypatch.delenv("NVFP4_GEMM_PAIR", raising=False)
    return request.param


@pytest.fixture(scope="module")
def B():
    from nvfp4_precision_02_b300 import binding, build
    build.build()
    binding.lib()
    assert torch.cuda.is_available()
    return binding


def _rand(rows, cols, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(rows, cols, generator=g) * std).to(torch.bfloat16)


def _oracle_ref(orc, a, w, two_d=True):
    qa = orc.quantize_1d(a)
    M, K = a.shape
    N = w.shape[0]
    A = orc.dequantize(qa, M, K)
    if two_d:
        qw = orc.quantize_2d(w, want_t=False)
        W = orc.dequantize_rows(qw["codes"][0], qw["sf"], K, float(qw["amax"][0]), np.arange(N))
    else:
        W = orc.dequantize(orc.quantize_1d(w), N, K)
    return orc.gemm(A, W)


def _quant_b(B, w, two_d):
    """Weights take 16x16 blocks when N is a multiple of 16; any N takes 1x16."""
    if two_d:
        return B.quantize_2d(w, want_t=False)[0]
    return B.quantize_1d(w)


def _check(out, ref, absum, bf16):
    ok, worst = gemm_within_bound(out, ref, absum, bf16)
    bad = np.argwhere(~ok)
    assert ok.all(), f"{len(bad)} elements out of bound, worst ratio {worst:.3g}, first {bad[:5].tolist()}"
    return worst


SHAPES = [(256, 256, 256),    # the tiny fprop workload shape
          (1, 1, 32), (17, 33, 64), (128, 256, 256), (129, 257, 288), (300, 520, 1024),
          (256, 384, 96), (64, 1000, 512), (520, 130, 2048),
          (136, 264, 8192),   # K >= 8192
          # K % 32 == 16: code rows of K/2 bytes are not a 16-byte multiple (the
          # producer copies them; single-CTA kernel)
          (64, 96, 16), (130, 300, 48), (200, 256, 80), (129, 520, 272)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("fp32", [False, True])
def test_gemm_fprop_shapes(B, orc, M, N, K, fp32):
    a = _rand(M, K, seed=M * 31 + K)
    w = _rand(N, K, seed=N * 17 + K + 1, std=0.02)
    two_d = N % 16 == 0
    qa = B.quantize_1d(a.cuda())
    qw = _quant_b(B, w.cuda(), two_d)
    c_amax = torch.full((1,), -1.0, device="cuda")
    out = B.gemm(qa, qw, out_dtype=B.OUT_FP32 if fp32 else B.OUT_BF16, c_amax=c_amax)
    torch.cuda.synchronize()
    ref, absum = _oracle_ref(orc, a, w, two_d)
    o = out.float().cpu().numpy()
    _check(o, ref, absum, bf16=not fp32)
    # the epilogue's amax is the largest magnitude of the stored outputs, exactly
    assert float(c_amax[0]) == float(np.abs(o).max())


def test_tiny_fprop_workload(B, orc):
    """256x256 A and W ~ N(0,1), seed 0: 1x16 RNE A, 16x16 W, bf16 C = A.W^T."""
    from nvfp4_precision_02_b300 import workloads as wl
    a, w = wl.tiny_inputs()
    qa = B.quantize_1d(a.cuda())
    qw, _, _ = B.quantize_2d(w.cuda(), want_t=False)
    out = B.gemm(qa, qw)
    out32 = B.gemm(qa, qw, out_dtype=B.OUT_FP32)
    torch.cuda.synchronize()
    ref, absum = _oracle_ref(orc, a, w)
    _check(out.float().cpu().numpy(), ref, absum, bf16=True)
    _check(out32.cpu().numpy(), ref, absum, bf16=False)


def test_gemm_ldc_and_exact_products(B, orc):
    """Operands with one nonzero per row whose sixth is an E4M3 value
    dequantise exactly, so every output is one exact product: the GPU must
    reproduce it exactly (also through a padded ldc)."""
    K = 64
    A = torch.zeros(16, K)
    W = torch.zeros(16, K)
    for i in range(16):
        A[i, (5 * i) % K] = [6, 3, 1.5, 0.75, 9, 4.5, 7.5, -10.5][i % 8]
        W[i, (5 * i) % K] = [12, -6, 3, 1.5, 7.5, 0.375, 24, 9][i % 8]
    amax = torch.tensor([2688.0], device="cuda")
    qa = B.quantize_1d(A.to(torch.bfloat16).cuda(), amax_in=amax)
    qw = B.quantize_1d(W.to(torch.bfloat16).cuda(), amax_in=amax)
    out = torch.full((16, 24), 7.0, device="cuda")
    B.gemm(qa, qw, out_dtype=B.OUT_FP32, out=out[:, :16])
    torch.cuda.synchronize()
    o = out.cpu().numpy()
    assert (o[:, :16] == (A.double() @ W.double().T).numpy()).all()
    assert (o[:, 16:] == 7.0).all()                      # nothing written beyond N


def test_dgrad_and_wgrad_operands(B, orc):
    """dgrad: dY (SR) x W^T from the 2D quantiser's transposed copy; wgrad:
    RHT(dY)^T (SR) x RHT(X)^T (RNE) with one shared sign mask."""
    T, Kh, N = 256, 192, 320
    x = _rand(T, Kh, seed=1)
    w = _rand(N, Kh, seed=2, std=0.02)
    dy = _rand(T, N, seed=3, std=1e-3)
    seed, mask = 7, 0x6A35
    # dgrad: dX[T, Kh] = dY[T, N] . W[N, Kh] -> B operand is W^T [Kh, N]
    qdy = B.quantize_1d(dy.cuda(), mode=B.SR, seed=seed)
    _, qwt, _ = B.quantize_2d(w.cuda(), want_t=True)
    dx = B.gemm(qdy, qwt, out_dtype=B.OUT_FP32)
    # wgrad: dW[N, Kh] = dY^T . X over tokens, both through the RHT
    sdy = B.rht_quantize(dy.cuda(), mask, mode=B.SR, seed=seed ^ 0x9E3779B97F4A7C15)
    sx = B.rht_quantize(x.cuda(), mask, mode=B.RNE)
    dw = B.gemm(sdy, sx, out_dtype=B.OUT_FP32)
    torch.cuda.synchronize()
    # oracle
    r_dy = orc.quantize_1d(dy, mode=orc.SR, seed=seed)
    r_w = orc.quantize_2d(w)
    A = orc.dequantize(r_dy, T, N)
    Bt = orc.dequantize_rows(r_w["codes_t"][0], r_w["sf_t"], N, float(r_w["amax"][0]), np.arange(Kh))
    ref, absum = orc.gemm(A, Bt)
    _check(dx.cpu().numpy(), ref, absum, bf16=False)
    r_sdy = orc.rht_quantize(dy, mask, mode=orc.SR, seed=seed ^ 0x9E3779B97F4A7C15)
    r_sx = orc.rht_quantize(x, mask, mode=orc.RNE)
    A2 = orc.dequantize(r_sdy, N, T)
    B2 = orc.dequantize(r_sx, Kh, T)
    ref2, absum2 = orc.gemm(A2, B2)
    _check(dw.cpu().numpy(), ref2, absum2, bf16=False)
    # the RHT is orthogonal: the wgrad of the transformed operands estimates dY^T X
    exact = dy.double().T @ x.double()
    rel = np.linalg.norm(dw.cpu().double().numpy() - exact.numpy()) / np.linalg.norm(exact.numpy())
    assert rel < 0.25


@pytest.mark.parametrize("K", [256, 48])
@pytest.mark.parametrize("fp32", [False, True])
def test_grouped_gemm(B, orc, fp32, K):
    n = 304                  # last N tile ragged; its second 128-row scale block is absent
    offsets = np.array([0, 0, 1, 130, 130, 400, 656, 657, 800], dtype=np.int64)   # empty and 1-row groups
    E = len(offsets) - 1
    R = int(offsets[-1])
    a = _rand(R, K, seed=5)
    g = torch.Generator().manual_seed(6)
    w = (torch.randn(E, n, K, generator=g) * 0.02 * torch.linspace(0.5, 4, E)[:, None, None]).to(torch.bfloat16)
    off = torch.from_numpy(offsets).cuda()
    qa = B.quantize_1d_grouped(a.cuda(), off)
    qw, _, _ = B.quantize_2d(w.cuda(), want_t=False)
    out = torch.full((R, n), -3.0, device="cuda",
                     dtype=torch.float32 if fp32 else torch.bfloat16)
    c_amax = torch.full((E,), -1.0, device="cuda")
    B.grouped_gemm(qa, off, qw, n, out_dtype=B.OUT_FP32 if fp32 else B.OUT_BF16, out=out, c_amax=c_amax)
    torch.cuda.synchronize()
    o = out.float().cpu().numpy()
    # per group: the largest stored magnitude, exactly (0 for an empty group)
    got = c_amax.cpu().numpy()
    for e in range(E):
        want = float(np.abs(o[offsets[e]:offsets[e + 1]]).max()) if offsets[e + 1] > offsets[e] else 0.0
        assert got[e] == want, (e, got[e], want)
    ra = orc.quantize_1d_grouped(a, offsets)
    rw = orc.quantize_2d(w, want_t=False)
    nsf = orc.sf_bytes(n, K)
    for e in range(E):
        o0, o1 = offsets[e], offsets[e + 1]
        if o1 == o0:
            continue
        Ae = orc.dequantize_rows(ra["codes"], ra["sf"], K, float(ra["amax"][e]), np.arange(o0, o1),
                                 sf_row0=orc.group_sf_row(offsets, e) - int(o0))
        We = orc.dequantize_rows(rw["codes"][e], rw["sf"][e * nsf:(e + 1) * nsf], K, float(rw["amax"][e]),
                                 np.arange(n))
        ref, absum = orc.gemm(Ae, We)
        _check(o[o0:o1], ref, absum, bf16=not fp32)


def test_grouped_gemm_leaves_rows_outside_groups(B):
    K, n = 64, 256
    offsets = torch.tensor([0, 100, 100], dtype=torch.int64)
    a = _rand(160, K, seed=8).cuda()
    w = _rand(2 * n, K, seed=9).reshape(2, n, K).cuda()
    off = offsets.cuda()
    qa = B.quantize_1d_grouped(a, off)
    qw, _, _ = B.quantize_2d(w, want_t=False)
    out = torch.full((160, n), 5.0, device="cuda", dtype=torch.float32)
    B.grouped_gemm(qa, off, qw, n, out_dtype=B.OUT_FP32, out=out)
    torch.cuda.synchronize()
    assert (out[100:] == 5.0).all()
    assert B.device_status() == 0


def test_wait_timeout_is_reported_not_hung(B):
    """A bounded wait that nothing completes returns and records a timeout
    in the device status word; the context stays usable."""
    assert B.device_status() == 0
    B.debug_wait_timeout(50_000_000)          # 50 ms
    assert B.device_status() & B.DEV_TIMEOUT
    assert B.device_status() == 0             # read clears
    x = torch.ones(16, 16, dtype=torch.bfloat16, device="cuda")
    q = B.quantize_1d(x)
    torch.cuda.synchronize()
    assert np_u8(q.amax)[0] == 1.0


@pytest.mark.parametrize("fp32", [False, True])
def test_grouped_dgrad_with_transposed_expert_weights(B, orc, fp32):
    """Backward of the LatentMoE up-projection H = A . W_e^T: the input
    gradient dA_e = dH_e . W_e runs on the grouped GEMM with the SR-quantised
    expert-sorted dH as A and, as B, the per-expert W_e^T that the batched 2D
    quantiser emits (16x16 tiles quantise identically in both orientations)."""
    latent, hidden = 192, 320                 # dA is [R, latent]; the dgrad K is hidden
    offsets = np.array([0, 3, 3, 150, 300, 301, 520], dtype=np.int64)   # an empty and 1-row experts
    E = len(offsets) - 1
    R = int(offsets[-1])
    g = torch.Generator().manual_seed(21)
    dh = (torch.randn(R, hidden, generator=g) * 1e-3).to(torch.bfloat16)
    w = (torch.randn(E, hidden, latent, generator=g) * 0.02 * torch.linspace(0.5, 3, E)[:, None, None]).to(torch.bfloat16)
    off = torch.from_numpy(offsets).cuda()
    qdh = B.quantize_1d_grouped(dh.cuda(), off, mode=B.SR, seed=17)
    _, qwt, _ = B.quantize_2d(w.cuda(), want_t=True)             # W_e^T: [E, latent, hidden]
    out = torch.full((R, latent), -3.0, device="cuda", dtype=torch.float32 if fp32 else torch.bfloat16)
    B.grouped_gemm(qdh, off, qwt, latent, out_dtype=B.OUT_FP32 if fp32 else B.OUT_BF16, out=out)
    torch.cuda.synchronize()
    o = out.float().cpu().numpy()
    rdh = orc.quantize_1d_grouped(dh, offsets, mode=orc.SR, seed=17)
    rw = orc.quantize_2d(w)
    nsf = orc.sf_bytes(latent, hidden)
    for e in range(E):
        o0, o1 = offsets[e], offsets[e + 1]
        if o1 == o0:
            continue
        A = orc.dequantize_rows(rdh["codes"], rdh["sf"], hidden, float(rdh["amax"][e]), np.arange(o0, o1),
                                sf_row0=orc.group_sf_row(offsets, e) - int(o0))
        Wt = orc.dequantize_rows(rw["codes_t"][e], rw["sf_t"][e * nsf:(e + 1) * nsf], hidden, float(rw["amax"][e]),
                                 np.arange(latent))
        ref, absum = orc.gemm(A, Wt)
        _check(o[o0:o1], ref, absum, bf16=not fp32)
    assert B.device_status() == 0


@pytest.mark.parametrize("fp32", [False, True])
def test_grouped_wgrad_groups_along_k(B, orc, fp32):
    """wgrad of the LatentMoE up-projection: dW_g = RHT(dH_g)^T . RHT(A_g) over
    expert g's tokens, both operands from the expert-segmented RHT quantiser
    (SR for dH, RNE for A) and the GEMM splitting K by expert.  An expert
    without tokens gets dW_g = 0."""
    hidden, latent = 320, 192                 # dW_g is [hidden, latent]
    offsets = np.array([0, 0, 1, 90, 90, 300, 301, 430], dtype=np.int64)
    E = len(offsets) - 1
    R = int(offsets[-1])
    g = torch.Generator().manual_seed(33)
    dh = (torch.randn(R, hidden, generator=g) * 1e-3).to(torch.bfloat16)
    a = torch.randn(R, latent, generator=g).to(torch.bfloat16)
    off = torch.from_numpy(offsets).cuda()
    mask, seed = 0x6B1D, 29
    kt = B.group_k_capacity(R, E)
    sdh = B.rht_quantize_grouped(dh.cuda(), off, mask, mode=B.SR, seed=seed, kt=kt)
    sa = B.rht_quantize_grouped(a.cuda(), off, mask, mode=B.RNE, kt=kt)
    out = torch.full((E * hidden, latent), -3.0, device="cuda", dtype=torch.float32 if fp32 else torch.bfloat16)
    c_amax = torch.full((E,), -1.0, device="cuda")
    B.grouped_gemm_k(sdh, sa, off, out_dtype=B.OUT_FP32 if fp32 else B.OUT_BF16, out=out, c_amax=c_amax)
    torch.cuda.synchronize()
    o = out.float().cpu().numpy().reshape(E, hidden, latent)
    rdh = orc.rht_quantize_grouped(dh, offsets, kt, mask, mode=orc.SR, seed=seed)
    ra = orc.rht_quantize_grouped(a, offsets, kt, mask, mode=orc.RNE)
    got_amax = c_amax.cpu().numpy()
    for e in range(E):
        ko0, ko1 = orc.group_k_offset(offsets, e), orc.group_k_offset(offsets, e + 1)
        if ko1 == ko0:
            assert (o[e] == 0).all() and got_amax[e] == 0.0
            continue
        Ad = orc.dequantize_rows(rdh["codes"], rdh["sf"], kt, float(rdh["amax"][e]), np.arange(hidden))[:, ko0:ko1]
        Bd = orc.dequantize_rows(ra["codes"], ra["sf"], kt, float(ra["amax"][e]), np.arange(latent))[:, ko0:ko1]
        ref, absum = orc.gemm(np.ascontiguousarray(Ad), np.ascontiguousarray(Bd))
        _check(o[e], ref, absum, bf16=not fp32)
        assert got_amax[e] == float(np.abs(o[e]).max())
        # the transform is orthogonal: the result estimates dH_g^T A_g
        exact = dh[offsets[e]:offsets[e + 1]].double().T @ a[offsets[e]:offsets[e + 1]].double()
        if offsets[e + 1] - offsets[e] > 64:
            rel = np.linalg.norm(o[e] - exact.numpy()) / np.linalg.norm(exact.numpy())
            assert rel < 0.3
    assert B.device_status() == 0
