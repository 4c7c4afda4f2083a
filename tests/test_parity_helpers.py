"""The GEMM acceptance rule used by every GPU GEMM test: the per-element
bound 1e-5 * sum_k |a_k b_k| against the FP64 reference, plus one bf16
rounding (half an ulp) for bf16 outputs."""
import numpy as np
import torch

from parity import bf16_ulp, gemm_within_bound


def test_bf16_ulp():
    assert bf16_ulp(np.array([1.0]))[0] == 2.0 ** -7
    assert bf16_ulp(np.array([1.99]))[0] == 2.0 ** -7
    assert bf16_ulp(np.array([2.0]))[0] == 2.0 ** -6
    assert bf16_ulp(np.array([-0.75]))[0] == 2.0 ** -8
    assert bf16_ulp(np.array([0.0]))[0] == 2.0 ** -133          # clamped at the smallest normal
    # agrees with the spacing of torch's bfloat16 numbers
    x = torch.tensor([1.0, 3.0, 1000.0, 1e-3], dtype=torch.bfloat16)
    nxt = torch.nextafter(x, torch.full_like(x, float("inf")))
    assert np.allclose((nxt - x).double().numpy(), bf16_ulp(x.double().numpy()), rtol=0, atol=0)


def test_bound_fp32_and_bf16():
    rng = np.random.default_rng(0)
    ref = rng.standard_normal(1000) * 10
    absum = np.abs(ref) * 3 + 1.0
    ok, worst = gemm_within_bound(ref.copy(), ref, absum, bf16=False)
    assert ok.all() and worst == 0.0
    # FP32: just inside and just outside 1e-5 * absum
    ok, _ = gemm_within_bound(ref + 0.99e-5 * absum, ref, absum, bf16=False)
    assert ok.all()
    ok, worst = gemm_within_bound(ref + 1.01e-5 * absum, ref, absum, bf16=False)
    assert not ok.any() and 1.0 < worst < 1.02
    # bf16: the correctly rounded reference passes even where the rounding exceeds the FP32 bound
    tiny = np.full_like(absum, 1e-12)
    rounded = torch.from_numpy(ref).to(torch.bfloat16).double().numpy()
    assert (np.abs(rounded - ref) > 1e-5 * tiny).any()
    ok, _ = gemm_within_bound(rounded, ref, tiny, bf16=True)
    assert ok.all()
    ok, _ = gemm_within_bound(rounded, ref, tiny, bf16=False)
    assert not ok.all()
    # one bf16 ulp off is rejected when the FP32 bound is negligible, except where the step
    # crosses into the next binade (the half ulp is taken of the larger magnitude)
    up = np.abs(rounded) + bf16_ulp(rounded)
    aref = np.abs(ref)
    ok, _ = gemm_within_bound(up, aref, tiny, bf16=True)
    crossed = bf16_ulp(up) > bf16_ulp(np.abs(rounded))
    assert not ok[~crossed].any()
    assert ok.mean() < 0.1


def test_zero_tolerance_elements():
    ref = np.array([0.0, 0.0])
    absum = np.array([0.0, 0.0])
    ok, worst = gemm_within_bound(np.array([0.0, 1e-30]), ref, absum, bf16=False)
    assert ok[0] and not ok[1] and worst == np.inf
