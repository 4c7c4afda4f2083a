"""Launch one op of the NVFP4 path on a named workload, for profiling.

Usage:
  python profile_cases.py <op> [--workload super|ultra] [--iters N]

The op's inputs are generated on the device, its operands (and, where the
step supplies it, the tensor amax) are prepared once, and then the op itself
is launched `iters` times back to back, so that a profiler can skip the
set-up launches and the first launch of the op and capture one launch alone
(for example `ncu -k regex:<kernel> -s 1 -c 1 python profile_cases.py <op>`).
It prints the mean CUDA-event time per launch.  The commands that produced
the summaries under profiles/ are written in each summary.

Quantiser ops take the amax as the step supplies it (one launch, one read of
the input):
  amax              k_amax over the in_proj weight W [N, K]
  quant1d_rne       k_quant1d<RNE>: X [T, K]
  quant1d_sr        k_quant1d<SR>: dY [T, N]
  quant2d           k_quant2d: W with W^T
  quant2d_moe       k_quant2d_w: the batched expert up-projection weights (W only)
  quant2d_moe_fused k_quant2d_resident: the same weights with their per-expert amax in one launch
  dual_amax         k_rht<3>: max |dY| and max |RHT(dY)| in one read
  rht_sr            k_rht<2>: RHT(dY)^T with SR
  dual_sr           k_rht<4>: 1x16 SR rows of dY and RHT(dY)^T with SR from one read
  rht_rne           k_rht<1>: RHT(X)^T with RNE
  amax_grouped      k_amax_grouped (then k_quant1d): per-expert amax of the routed activations A
  quant1d_grouped_a k_quant1d<RNE, grouped>: A
  quant1d_grouped_h k_quant1d<RNE, grouped>: the expert hidden activations H
  rht_grouped_sr    k_rht<2, grouped>: expert-segmented RHT of dH with SR
  quant1d_mse       k_quant1d_mse: W with minimum-error block scales
  sr_fp16           k_sr_fp16: an SSM-cache-sized FP32 tensor to FP16
  count_zero        k_count_zero_codes: the SR-quantised dY
GEMM ops (operands quantised once):
  gemm_fprop, gemm_dgrad, gemm_wgrad, grouped_up (with the per-expert amax
  of H, as the step runs it), grouped_down, grouped_dgrad, grouped_wgrad.
"""
from __future__ import annotations

import argparse
import os
import sys

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from nvfp4_precision_02_b300 import binding as B  # noqa: E402
from nvfp4_precision_02_b300 import workloads as wl  # noqa: E402

OPS = ["amax", "quant1d_rne", "quant1d_sr", "quant2d", "quant2d_moe", "quant2d_moe_fused", "dual_amax", "rht_sr",
       "dual_sr", "rht_rne",
       "amax_grouped", "quant1d_grouped_a", "quant1d_grouped_h", "rht_grouped_sr", "quant1d_mse", "sr_fp16",
       "count_zero", "gemm_fprop", "gemm_dgrad", "gemm_wgrad", "grouped_up", "grouped_down", "grouped_dgrad",
       "grouped_wgrad"]


def prepare(op: str, which: str, dev):
    """Returns a zero-argument callable that launches the op once."""
    d = wl.ULTRA_DENSE if which == "ultra" else wl.SUPER_DENSE
    m = wl.ULTRA_MOE if which == "ultra" else wl.SUPER_MOE
    seed, mask = wl.SEEDS["sr"], wl.sign_mask_from_seed(wl.SEEDS["rht_sign"])
    T, K, N = d.tokens, d.hidden, d.out
    if op in ("quant1d_sr", "dual_amax", "rht_sr", "count_zero", "dual_sr"):
        dy = wl.dense_inputs(d, which, device=dev, want=("dy",))["dy"]
        am = torch.empty(2, dtype=torch.float32, device=dev)
        B.dual_amax(dy, mask, out=am)
        if op == "dual_amax":
            return lambda: B.dual_amax(dy, mask, out=am)
        if op == "dual_sr":
            qr, qt = B.empty_qtensor(T, N, dev), B.empty_qtensor(N, T, dev)
            zc = torch.empty(1, dtype=torch.int64, device=dev)
            return lambda: B.dual_sr_quantize(dy, mask, seed, wl.wgrad_seed(seed), am, out_row=qr, out_t=qt,
                                              zero_count=zc)
        if op == "rht_sr":
            q = B.empty_qtensor(N, T, dev)
            return lambda: B.rht_quantize(dy, mask, B.SR, wl.wgrad_seed(seed), amax_in=am[1:2], out=q)
        q = B.empty_qtensor(T, N, dev)
        if op == "count_zero":
            B.quantize_1d(dy, B.SR, seed, amax_in=am[0:1], out=q)
            return lambda: B.count_zero_codes(q)
        return lambda: B.quantize_1d(dy, B.SR, seed, amax_in=am[0:1], out=q)
    if op in ("quant1d_rne", "rht_rne"):
        x = wl.dense_inputs(d, which, device=dev, want=("x",))["x"]
        if op == "rht_rne":
            q = B.empty_qtensor(K, T, dev)
            B.rht_quantize(x, mask, B.RNE, 0, out=q)
            return lambda: B.rht_quantize(x, mask, B.RNE, 0, amax_in=q.amax, out=q)
        q = B.empty_qtensor(T, K, dev)
        B.quantize_1d(x, B.RNE, 0, out=q)
        return lambda: B.quantize_1d(x, B.RNE, 0, amax_in=q.amax, out=q)
    if op in ("amax", "quant2d", "quant1d_mse"):
        w = wl.dense_inputs(d, which, device=dev, want=("w",))["w"]
        if op == "amax":
            out = torch.empty(1, dtype=torch.float32, device=dev)
            return lambda: B.amax(w, out=out)
        qw, qwt = B.empty_qtensor(N, K, dev), B.empty_qtensor(K, N, dev)
        B.quantize_2d(w, want_t=True, out=qw, out_t=qwt)
        if op == "quant1d_mse":
            q = B.empty_qtensor(N, K, dev)
            return lambda: B.quantize_1d_mse(w, amax_in=qw.amax, out=q)
        return lambda: B.quantize_2d(w, want_t=True, amax_in=qw.amax, out=qw, out_t=qwt)
    if op in ("quant2d_moe", "quant2d_moe_fused"):
        w = wl.batched_normal_bf16(m.experts, m.expert_hidden, m.latent, 0.02, wl.SEEDS[which + "_moe_w"], dev)
        qw = B.empty_qtensor(m.expert_hidden, m.latent, dev, batch=m.experts, n_amax=m.experts)
        if op == "quant2d_moe_fused":
            ws = torch.empty(B.quantize_2d_fused_workspace(m.experts), dtype=torch.uint8, device=dev)
            return lambda: B.quantize_2d_fused(w, workspace=ws, out=qw)
        B.quantize_2d(w, want_t=False, out=qw)
        return lambda: B.quantize_2d(w, want_t=False, amax_in=qw.amax, out=qw)
    if op == "sr_fp16":
        g = torch.Generator(device=dev)
        g.manual_seed(12)
        x = torch.randn(256 * 256 * 64 * 128 // (4 if which == "super" else 1), generator=g, device=dev)
        out = torch.empty(x.numel(), dtype=torch.float16, device=dev)
        return lambda: B.sr_fp16(x, 5, out=out)
    if op in ("amax_grouped", "quant1d_grouped_a", "quant1d_grouped_h", "rht_grouped_sr"):
        mi = wl.moe_inputs(m, which, device=dev, want=("a",))
        off = mi["routing"].offsets.to(dev)
        R = int(mi["routing"].offsets[-1])
        if op == "rht_grouped_sr":
            dh = wl.normal_bf16((R, m.expert_hidden), 1e-3, 98, dev)
            kt = B.group_k_capacity(R, m.experts)
            q = B.empty_qtensor(m.expert_hidden, kt, dev, n_amax=m.experts)
            B.rht_quantize_grouped(dh, off, mask, B.SR, wl.wgrad_seed(seed), kt=kt, out=q)
            return lambda: B.rht_quantize_grouped(dh, off, mask, B.SR, wl.wgrad_seed(seed), kt=kt, amax_in=q.amax,
                                                  out=q)
        if op == "quant1d_grouped_h":
            x = wl.normal_bf16((R, m.expert_hidden), 1.0, 99, dev)
        else:
            x = mi["a"]
        cols = x.shape[1]
        q = B.empty_qtensor(R, cols, dev, n_amax=m.experts, sf_size=B.sf_bytes_grouped(R, cols, m.experts))
        B.quantize_1d_grouped(x, off, B.RNE, 0, out=q)
        if op == "amax_grouped":        # the grouped quantiser without a supplied amax runs k_amax_grouped first
            return lambda: B.quantize_1d_grouped(x, off, B.RNE, 0, out=q)
        return lambda: B.quantize_1d_grouped(x, off, B.RNE, 0, amax_in=q.amax, out=q)
    if op.startswith("gemm_"):
        ins = wl.dense_inputs(d, which, device=dev)
        x, w, dy = ins["x"], ins["w"], ins["dy"]
        if op == "gemm_fprop":
            qa, qb = B.quantize_1d(x), B.quantize_2d(w, want_t=False)[0]
            out = torch.empty(T, N, dtype=torch.bfloat16, device=dev)
            return lambda: B.gemm(qa, qb, B.OUT_BF16, out=out)
        if op == "gemm_dgrad":
            qa, qb = B.quantize_1d(dy, B.SR, seed), B.quantize_2d(w, want_t=True)[1]
            out = torch.empty(T, K, dtype=torch.bfloat16, device=dev)
            return lambda: B.gemm(qa, qb, B.OUT_BF16, out=out)
        qa = B.rht_quantize(dy, mask, B.SR, wl.wgrad_seed(seed))
        qb = B.rht_quantize(x, mask, B.RNE)
        out = torch.empty(N, K, dtype=torch.float32, device=dev)
        return lambda: B.gemm(qa, qb, B.OUT_FP32, out=out)
    if op in ("grouped_dgrad", "grouped_wgrad"):
        mi = wl.moe_inputs(m, which, device=dev, want=("a", "w_up") if op == "grouped_dgrad" else ("a",))
        off = mi["routing"].offsets.to(dev)
        R = int(mi["routing"].offsets[-1])
        dh = wl.normal_bf16((R, m.expert_hidden), 1e-3, 98, dev)
        if op == "grouped_dgrad":
            qdh = B.quantize_1d_grouped(dh, off, B.SR, seed)
            qwt = B.quantize_2d(mi["w_up"], want_t=True)[1]          # [E, latent, hidden]
            out = torch.empty(R, m.latent, dtype=torch.bfloat16, device=dev)
            return lambda: B.grouped_gemm(qdh, off, qwt, m.latent, B.OUT_BF16, out=out)
        kt = B.group_k_capacity(R, m.experts)
        sdh = B.rht_quantize_grouped(dh, off, mask, B.SR, wl.wgrad_seed(seed), kt=kt)
        sa = B.rht_quantize_grouped(mi["a"], off, mask, B.RNE, kt=kt)
        out = torch.empty(m.experts * m.expert_hidden, m.latent, dtype=torch.float32, device=dev)
        return lambda: B.grouped_gemm_k(sdh, sa, off, B.OUT_FP32, out=out)
    if op in ("grouped_up", "grouped_down"):
        up = op == "grouped_up"
        mi = wl.moe_inputs(m, which, device=dev, want=("a", "w_up") if up else ("a", "w_down"))
        off = mi["routing"].offsets.to(dev)
        R = int(mi["routing"].offsets[-1])
        if up:
            qa = B.quantize_1d_grouped(mi["a"], off)
            qw = B.quantize_2d(mi["w_up"], want_t=False)[0]
            n = m.expert_hidden
        else:
            h = wl.normal_bf16((R, m.expert_hidden), 1.0, 99, dev)
            qa = B.quantize_1d_grouped(h, off)
            qw = B.quantize_2d(mi["w_down"], want_t=False)[0]
            n = m.latent
        out = torch.empty(R, n, dtype=torch.bfloat16, device=dev)
        if up:
            hamax = torch.empty(m.experts, dtype=torch.float32, device=dev)
            return lambda: B.grouped_gemm(qa, off, qw, n, B.OUT_BF16, out=out, c_amax=hamax)
        return lambda: B.grouped_gemm(qa, off, qw, n, B.OUT_BF16, out=out)
    raise ValueError(f"unknown op {op}")


def main(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("op", choices=OPS)
    p.add_argument("--workload", choices=["super", "ultra"], default="super")
    p.add_argument("--iters", type=int, default=3)
    a = p.parse_args(argv)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    B.lib()
    fn = prepare(a.op, a.workload, dev)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(a.iters):
        fn()
    e1.record()
    torch.cuda.synchronize()
    if B.device_status() != 0:
        raise RuntimeError("device status word set")
    print(f"{a.op} {a.workload}: {e0.elapsed_time(e1) / max(a.iters, 1):.4f} ms per launch")
    return 0


if __name__ == "__main__":
    sys.exit(main())
