"""The checks of the full-size GPU parity tests, run on the CPU against a
small stand-in of the benchmark's Workload whose "GPU" results are the
oracle's own whole-tensor results.  The checks must accept them, and must
reject each planted mistake.  This keeps the full-size tests honest (they
compare what they claim to) and free of plain programming errors before
they reach a GPU."""
import types

import numpy as np
import pytest
import torch

import test_gpu_zfull as full
from nvfp4_precision_02_b300.binding import QTensor

T, K, N = 512, 320, 272                       # dense: tokens, hidden, out
E, L, HH = 6, 64, 96                          # experts, latent, expert hidden
OFFSETS = [0, 300, 300, 301, 620, 700, 900]   # one empty and one single-row expert
MASK, SEED = 0x5A3C, 7


def _bf16(shape, std, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * std).to(torch.bfloat16)


def _q(d, rows, cols, codes_key="codes", sf_key="sf", amax=None):
    am = np.asarray(d["amax"] if amax is None else amax, dtype=np.float32).reshape(-1)
    return QTensor(torch.from_numpy(np.ascontiguousarray(d[codes_key])), torch.from_numpy(d[sf_key].copy()),
                   torch.from_numpy(am.copy()), rows, cols)


def _deq(orc, q, rows, cols, amax, sf_row0=0, row_ids=None):
    ids = np.arange(rows) if row_ids is None else row_ids
    return orc.dequantize_rows(q.codes.numpy().reshape(-1, cols // 2), q.sf.numpy(), cols, amax, ids, sf_row0)


class FakeB:
    """The binding calls the full-size tests make, answered by the oracle.
    A call named in `corrupt` returns a slightly wrong result."""
    RNE, SR = 0, 1
    OUT_BF16, OUT_FP32 = 0, 1

    def __init__(self, orc):
        self.orc = orc
        self.corrupt = set()

    def _bad(self, name, q):
        return _flip_codes(q) if name in self.corrupt else q

    def sf_bytes(self, rows, cols):
        return self.orc.sf_bytes(rows, cols)

    def device_status(self):
        return 0

    def quantize_1d_grouped(self, x, offsets, mode=0, seed=0):
        d = self.orc.quantize_1d_grouped(x, offsets.numpy(), mode=mode, seed=seed)
        return self._bad("quantize_1d_grouped", _q(d, x.shape[0], x.shape[1]))

    def quantize_2d(self, w, want_t=True):
        d = self.orc.quantize_2d(w, want_t=want_t)
        E, n, k = w.shape
        qw = _q(d, n, k)
        qt = _q(d, k, n, codes_key="codes_t", sf_key="sf_t") if want_t else None
        return qw, self._bad("quantize_2d", qt) if want_t else None, None

    def grouped_gemm(self, qx, offsets, qw, n, out_dtype):
        out = _grouped(self.orc, qx, offsets.numpy(), qw, n)
        return out * 1.01 if "grouped_gemm" in self.corrupt else out

    def group_k_capacity(self, rows, groups):
        return (rows + 63 * groups + 63) // 64 * 64

    def rht_quantize_grouped(self, x, offsets, mask, mode, seed, kt):
        d = self.orc.rht_quantize_grouped(x, offsets.numpy(), kt, mask, mode=mode, seed=seed)
        q = _q(d, x.shape[1], kt)
        return _flip_scales(q) if ("rht_quantize_grouped", mode) in self.corrupt else q

    def grouped_gemm_k(self, qa, qb, offsets, out_dtype):
        orc, offs = self.orc, offsets.numpy()
        M, Nb, kt = qa.rows, qb.rows, qa.cols
        out = torch.zeros((len(offs) - 1) * M, Nb, dtype=torch.float32)
        for g in range(len(offs) - 1):
            cnt = int(offs[g + 1] - offs[g])
            if cnt == 0:
                continue
            ko, kp = orc.group_k_offset(offs, g), (cnt + 63) // 64 * 64
            a = orc.dequantize_rows(qa.codes.numpy(), qa.sf.numpy(), kt, float(qa.amax[g]), np.arange(M))
            b = orc.dequantize_rows(qb.codes.numpy(), qb.sf.numpy(), kt, float(qb.amax[g]), np.arange(Nb))
            ref, _ = orc.gemm(a[:, ko:ko + kp], b[:, ko:ko + kp])
            out[g * M:(g + 1) * M] = torch.from_numpy(ref)
        return -out if "grouped_gemm_k" in self.corrupt else out

    def quantize_1d_mse(self, w, amax_in):
        q = _q(self.orc.quantize_1d_mse(w, amax_in=float(amax_in[0])), w.shape[0], w.shape[1])
        return _flip_scales(q) if "quantize_1d_mse" in self.corrupt else q

    def sr_fp16(self, x, seed):
        b = self.orc.sr_fp16(x.numpy(), seed)
        if "sr_fp16" in self.corrupt:
            b = b ^ np.uint16(1)
        return torch.from_numpy(b.view(np.float16))

    def count_zero_codes(self, q):
        c = q.codes.numpy()
        n = int(((c & 7) == 0).sum()) + int((((c >> 4) & 7) == 0).sum())
        return torch.tensor([n + ("count_zero_codes" in self.corrupt)], dtype=torch.int64)


def _grouped(orc, qx, offs, qw, n):
    cols = qx.cols
    out = torch.zeros(qx.rows, n, dtype=torch.bfloat16)
    nsf = orc.sf_bytes(n, cols)
    for g in range(len(offs) - 1):
        o0, o1 = int(offs[g]), int(offs[g + 1])
        if o1 == o0:
            continue
        p = orc.group_sf_row(offs, g)
        a = orc.dequantize_rows(qx.codes.numpy(), qx.sf.numpy(), cols, float(qx.amax[g]),
                                np.arange(o0, o1), p - o0)
        w = orc.dequantize_rows(qw.codes.numpy()[g], qw.sf.numpy()[g * nsf:(g + 1) * nsf], cols,
                                float(qw.amax[g]), np.arange(n))
        ref, _ = orc.gemm(a, w)
        out[o0:o1] = torch.from_numpy(ref).to(torch.bfloat16)
    return out


def _fake_run(orc):
    wk = types.SimpleNamespace()
    wk.dense = types.SimpleNamespace(tokens=T, hidden=K, out=N)
    wk.moe = types.SimpleNamespace(experts=E, latent=L, expert_hidden=HH)
    wk.x, wk.w, wk.dy = _bf16((T, K), 1.0, 1), _bf16((N, K), 0.02, 2), _bf16((T, N), 1e-3, 3)
    offs = torch.tensor(OFFSETS, dtype=torch.int64)
    wk.routing = types.SimpleNamespace(offsets=offs)
    wk.offsets = offs
    wk.R = OFFSETS[-1]
    wk.a = _bf16((wk.R, L), 1.0, 4)
    wk.w_up, wk.w_down = _bf16((E, HH, L), 0.02, 5), _bf16((E, L, HH), 0.02, 6)
    wk.seed, wk.wseed, wk.mask = SEED, SEED ^ 0x9E3779B97F4A7C15, MASK
    wk.qx = _q(orc.quantize_1d(wk.x), T, K)
    q2 = orc.quantize_2d(wk.w, want_t=True)
    wk.qw = QTensor(torch.from_numpy(q2["codes"][0].copy()), torch.from_numpy(q2["sf"].copy()),
                    torch.from_numpy(q2["amax"].copy()), N, K)
    wk.qwt = QTensor(torch.from_numpy(q2["codes_t"][0].copy()), torch.from_numpy(q2["sf_t"].copy()),
                     torch.from_numpy(q2["amax"].copy()), K, N)
    wk.dy_amax = torch.tensor([orc.amax(wk.dy), orc.rht_amax(wk.dy, MASK)], dtype=torch.float32)
    wk.qdy = _q(orc.quantize_1d(wk.dy, mode=1, seed=SEED), T, N)
    c = wk.qdy.codes.numpy()
    wk.dy_zeros = torch.tensor([int(((c & 7) == 0).sum()) + int((((c >> 4) & 7) == 0).sum())], dtype=torch.int64)
    wk.sdy = _q(orc.rht_quantize(wk.dy, MASK, mode=1, seed=wk.wseed), N, T)
    wk.sx = _q(orc.rht_quantize(wk.x, MASK, mode=0), K, T)
    wk.qwu = _q(orc.quantize_2d(wk.w_up, want_t=False), HH, L)
    wk.qwd = _q(orc.quantize_2d(wk.w_down, want_t=False), L, HH)
    wk.qa = _q(orc.quantize_1d_grouped(wk.a, np.array(OFFSETS)), wk.R, L)
    ref, _ = orc.gemm(_deq(orc, wk.qx, T, K, wk.qx.amax.item()), _deq(orc, wk.qw, N, K, wk.qw.amax.item()))
    wk.y = torch.from_numpy(ref).to(torch.bfloat16)
    ref, _ = orc.gemm(_deq(orc, wk.qdy, T, N, wk.qdy.amax.item()), _deq(orc, wk.qwt, K, N, wk.qwt.amax.item()))
    wk.dx = torch.from_numpy(ref).to(torch.bfloat16)
    ref, _ = orc.gemm(_deq(orc, wk.sdy, N, T, wk.sdy.amax.item()), _deq(orc, wk.sx, K, T, wk.sx.amax.item()))
    wk.dw = torch.from_numpy(ref).to(torch.float32)
    wk.h = _grouped(orc, wk.qa, np.array(OFFSETS), wk.qwu, HH)
    hmax = [float(wk.h[OFFSETS[g]:OFFSETS[g + 1]].abs().max()) if OFFSETS[g + 1] > OFFSETS[g] else 0.0
            for g in range(E)]
    wk.qh = types.SimpleNamespace(amax=torch.tensor(hmax, dtype=torch.float32))
    return types.SimpleNamespace(wk=wk, B=FakeB(orc), host={})


TESTS = [full.test_fprop_full_size, full.test_dgrad_full_size, full.test_wgrad_full_size,
         full.test_moe_up_full_size, full.test_moe_down_full_size, full.test_expert_backward_full_size,
         full.test_ptq_mse_scales_full_size, full.test_sr_fp16_full_size, full.test_zero_code_count_full_size]


@pytest.fixture(scope="module")
def fake(orc):
    return _fake_run(orc)


@pytest.fixture(autouse=True)
def small_ssm_cache(monkeypatch):
    monkeypatch.setattr(full, "SSM_ELEMENTS", 6000)


@pytest.mark.parametrize("test", TESTS, ids=lambda t: t.__name__)
def test_checks_accept_the_oracles_results(fake, orc, test):
    fake.host.clear()
    test(fake, orc)


def _flip_codes(q):
    c = q.codes.clone()
    c.view(-1)[1::7] ^= 0x01
    return QTensor(c, q.sf, q.amax, q.rows, q.cols)


def _flip_scales(q):
    s = q.sf.clone()
    s[s != 0] ^= 0x01
    return QTensor(q.codes, s, q.amax, q.rows, q.cols)


PLANTS = [
    ("qx", _flip_codes, full.test_fprop_full_size),
    ("qw", _flip_scales, full.test_fprop_full_size),
    ("y", lambda y: y * 1.01, full.test_fprop_full_size),
    ("qdy", _flip_codes, full.test_dgrad_full_size),
    ("qwt", _flip_codes, full.test_dgrad_full_size),
    ("dx", lambda y: -y, full.test_dgrad_full_size),
    ("sdy", _flip_scales, full.test_wgrad_full_size),
    ("sx", _flip_codes, full.test_wgrad_full_size),
    ("dw", lambda y: y + 1e-3 * y.abs().max(), full.test_wgrad_full_size),
    ("dy_amax", lambda a: a * 2, full.test_wgrad_full_size),
    ("qa", _flip_codes, full.test_moe_up_full_size),
    ("qwu", _flip_scales, full.test_moe_up_full_size),
    ("h", lambda y: y * 1.01, full.test_moe_up_full_size),
    ("qwd", _flip_codes, full.test_moe_down_full_size),
]


CORRUPT = [
    ("quantize_1d_grouped", full.test_expert_backward_full_size),
    ("quantize_2d", full.test_expert_backward_full_size),
    ("grouped_gemm", full.test_expert_backward_full_size),
    (("rht_quantize_grouped", 0), full.test_expert_backward_full_size),
    (("rht_quantize_grouped", 1), full.test_expert_backward_full_size),
    ("grouped_gemm_k", full.test_expert_backward_full_size),
    ("quantize_1d_mse", full.test_ptq_mse_scales_full_size),
    ("sr_fp16", full.test_sr_fp16_full_size),
    ("count_zero_codes", full.test_zero_code_count_full_size),
]


@pytest.mark.parametrize("call,test", CORRUPT, ids=[str(c[0]) for c in CORRUPT])
def test_checks_reject_a_wrong_call_result(fake, orc, call, test):
    fake.B.corrupt = {call}
    fake.host.clear()
    try:
        with pytest.raises(AssertionError):
            test(fake, orc)
    finally:
        fake.B.corrupt = set()


@pytest.mark.parametrize("name,plant,test", PLANTS, ids=[p[0] for p in PLANTS])
def test_checks_reject_a_planted_mistake(fake, orc, name, plant, test):
    saved = getattr(fake.wk, name)
    setattr(fake.wk, name, plant(saved))
    fake.host.clear()
    try:
        with pytest.raises(AssertionError):
            test(fake, orc)
    finally:
        setattr(fake.wk, name, saved)
