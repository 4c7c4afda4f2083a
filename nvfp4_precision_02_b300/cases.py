"""Run one step of the NVFP4 path on a named workload, for profiling.

Usage:
  python -m nvfp4_precision_02_b300.cases <op> [--workload super|ultra] [--iters N]

<op> is one of: amax, quant1d_rne, quant1d_sr, quant2d, quant2d_moe, quant2d_moe_fused, rht_sr,
quant1d_grouped_a (per-expert amax + RNE of the routed activations), quant1d_grouped_h (RNE of
the expert hidden activations with their amax supplied), gemm_fprop, gemm_dgrad, gemm_wgrad,
grouped_up, grouped_down, grouped_dgrad (dA = dH . W_up per expert, W_up^T from the 2D quantiser),
grouped_wgrad (dW_up = RHT(dH)^T . RHT(A) per expert, groups along K, FP32 out).  The inputs of the op are generated on the device and
its operands quantised once; the op itself is then launched `iters` times back to back, so
a profiler can skip the set-up launches and capture the op alone (for example with
`ncu -k regex:<kernel> -s 1 -c 1`).  It prints the mean CUDA-event time per launch.
"""
from __future__ import annotations

import argparse
import sys

import torch

from . import binding as B
from . import workloads as wl

OPS = ["amax", "quant1d_rne", "quant1d_sr", "quant2d", "quant2d_moe", "quant2d_moe_fused", "rht_sr",
       "quant1d_grouped_a", "quant1d_grouped_h", "gemm_fprop", "gemm_dgrad", "gemm_wgrad", "grouped_up",
       "grouped_down", "grouped_dgrad", "grouped_wgrad"]


def prepare(op: str, which: str, dev):
    """Returns a zero-argument callable that launches the op once."""
    d = wl.ULTRA_DENSE if which == "ultra" else wl.SUPER_DENSE
    m = wl.ULTRA_MOE if which == "ultra" else wl.SUPER_MOE
    seed, mask = wl.SEEDS["sr"], wl.sign_mask_from_seed(wl.SEEDS["rht_sign"])
    T, K, N = d.tokens, d.hidden, d.out
    if op in ("amax", "quant1d_rne", "quant1d_sr", "rht_sr"):
        x = wl.normal_bf16((T, N), 1e-3, wl.SEEDS[which + "_dy"], dev)
        if op == "amax":
            out = torch.empty(1, dtype=torch.float32, device=dev)
            return lambda: B.amax(x, out=out)
        if op == "rht_sr":
            q = B.empty_qtensor(N, T, dev)
            return lambda: B.rht_quantize(x, mask, B.SR, wl.wgrad_seed(seed), out=q)
        q = B.empty_qtensor(T, N, dev)
        mode = B.SR if op == "quant1d_sr" else B.RNE
        return lambda: B.quantize_1d(x, mode, seed, out=q)
    if op == "quant2d":
        w = wl.normal_bf16((N, K), 0.02, wl.SEEDS[which + "_w"], dev)
        qw, qwt = B.empty_qtensor(N, K, dev), B.empty_qtensor(K, N, dev)
        return lambda: B.quantize_2d(w, want_t=True, out=qw, out_t=qwt)
    if op in ("quant2d_moe", "quant2d_moe_fused"):
        w = wl.batched_normal_bf16(m.experts, m.expert_hidden, m.latent, 0.02, wl.SEEDS[which + "_moe_w"], dev)
        qw = B.empty_qtensor(m.expert_hidden, m.latent, dev, batch=m.experts, n_amax=m.experts)
        if op == "quant2d_moe":
            return lambda: B.quantize_2d(w, want_t=False, out=qw)
        ws = torch.empty(B.quantize_2d_fused_workspace(m.experts), dtype=torch.uint8, device=dev)
        return lambda: B.quantize_2d_fused(w, workspace=ws, out=qw)
    if op.startswith("quant1d_grouped"):
        mi = wl.moe_inputs(m, which, device=dev, want=("a",))
        off = mi["routing"].offsets.to(dev)
        R = int(mi["routing"].offsets[-1])
        if op == "quant1d_grouped_a":
            qa = B.empty_qtensor(R, m.latent, dev, n_amax=m.experts, sf_size=B.sf_bytes_grouped(R, m.latent, m.experts))
            return lambda: B.quantize_1d_grouped(mi["a"], off, B.RNE, 0, out=qa)
        h = wl.normal_bf16((R, m.expert_hidden), 1.0, 99, dev)
        qh = B.empty_qtensor(R, m.expert_hidden, dev, n_amax=m.experts,
                             sf_size=B.sf_bytes_grouped(R, m.expert_hidden, m.experts))
        B.quantize_1d_grouped(h, off, B.RNE, 0, out=qh)          # per-expert amax, reused below
        return lambda: B.quantize_1d_grouped(h, off, B.RNE, 0, amax_in=qh.amax, out=qh)
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
    if op.startswith("grouped_"):
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
