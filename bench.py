#!/usr/bin/env python
"""Benchmark of the NVFP4 training linear-layer hot path on B300.

One step = one pass of every hot-path step over one batch of the Ultra-shaped
workload (default ``--workload ultra``):
  fprop   X[16384, 8192] 1x16 RNE, W[33024, 8192] 16x16 (+W^T), Y = X.W^T
  dgrad   dY[16384, 33024] 1x16 SR (seed 7), dX = dY.(W^T)^T
  wgrad   16-point RHT along tokens on dY (SR) and X (RNE), dW = dY^T.X (FP32 out)
  MoE     512 experts, top-22 Zipf(1.1) routing of 16384 tokens (360448 rows):
          W_up[512, 5120, 2048], W_down[512, 2048, 5120] 16x16; A 1x16 per expert;
          H = up(A), requantised per expert, O = down(H)
Inputs are generated on the device from seeded generators and are resident
in HBM before the timed region; every step streams tens of GB, far more than
the 126 MB L2, so no separate L2 flush is done.

Printed: one JSON line (rank 0).  ``value`` = GEMM FLOPs of the step / step
time (quantisers included).  ``--impl reference`` times the CPU oracle on a
bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "NVFP4 GEMM TFLOPS (% dense FP4 peak); quantize GB/s (% HBM) on 1 B300"
FP4_OVER_BF16 = 13.5 / 2.25      # nominal dense FP4 : BF16 tensor throughput on B300
FP4_DATASHEET_TFLOPS = 13500.0   # nominal dense NVFP4 figure of a B300 (HGX class), unverified
# FP4 FLOP per SM per clock.  ncu's peak for
# sm__ops_path_tensor_op_utcomma_src_fp4_dst_fp32_sparsity_off is 7,274,496
# FLOP per cycle over 148 SMs (49152 per SM); back-to-back issue of the
# block-scaled MMA this library uses (kind::mxf4nvf4, scale_vec::4X, E4M3
# scales), with no data movement, completes one 128x256x64 MMA per 128 SM
# cycles on B300 (32768 FLOP per SM per cycle) for single CTAs and CTA pairs,
# N = 128 and 256 alike, at any number of active SMs.
FP4_FLOP_PER_CLK_SM_COUNTER = 49152
FP4_FLOP_PER_CLK_SM = 32768
HBM_NOMINAL_GBS = 8000.0         # the ~8 TB/s nominal HBM3e figure the quantiser target is stated against


def parse(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", choices=["ultra", "super"], default="ultra")
    p.add_argument("--e2e-steps", type=int, default=2)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-configs", action="store_true", help="skip the per-config measurements (c1-c4)")
    p.add_argument("--launch-check", action="store_true",
                   help="start the ranks, time an empty region and print the line (no GPU work; CPU ranks use gloo)")
    return p.parse_args(argv)


# Source of the GEMM kernel; the ncu traffic figure committed under
# profiles/ is only reported while it is unchanged since the capture.
GEMM_SOURCES = ("nvfp4_precision_02_b300/csrc/gemm.cuh",)


def code_text(src: str) -> str:
    """The code of a C/CUDA source without its comments and with whitespace
    runs folded, so that editing a comment does not detach a profile from the
    code it measured.  (String literals of the kernel sources hold no comment
    markers.)"""
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return " ".join(src.split())


def source_hash(paths=GEMM_SOURCES) -> str:
    h = hashlib.sha256()
    for f in paths:
        with open(os.path.join(ROOT, f)) as fh:
            h.update(code_text(fh.read()).encode())
    return h.hexdigest()


def profiled_traffic(summary: str):
    """DRAM bytes per launch from a committed ncu summary (lines
    `dram_bytes_per_launch: N` and `kernel_code_sha256: H`, the hash of the
    kernel source's code without comments), or None when the summary is
    missing or the kernel code changed after the capture."""
    path = os.path.join(ROOT, "profiles", summary)
    if not os.path.exists(path):
        return None
    text = open(path).read()
    b = re.search(r"dram_bytes_per_launch:\s*(\d+)", text)
    h = re.search(r"kernel_code_sha256:\s*([0-9a-f]{64})", text)
    if not b or not h or h.group(1) != source_hash():
        return None
    return int(b.group(1))


# Sources of the quantiser kernels (a quantiser profile is tied to these).
QUANT_SOURCES = ("nvfp4_precision_02_b300/csrc/quant.cuh", "nvfp4_precision_02_b300/csrc/common.cuh")


def profiled_quant_field(summary: str, field: str):
    """A number recorded as `<field>: X` in a committed quantiser ncu summary
    (whose `kernel_code_sha256: H` is the hash of the quantiser sources'
    code), or None when the summary or the field is missing or the code
    changed after the capture."""
    path = os.path.join(ROOT, "profiles", summary)
    if not os.path.exists(path):
        return None
    text = open(path).read()
    b = re.search(re.escape(field) + r":\s*([0-9.]+)", text)
    h = re.search(r"kernel_code_sha256:\s*([0-9a-f]{64})", text)
    if not b or not h or h.group(1) != source_hash(QUANT_SOURCES):
        return None
    return float(b.group(1))


def profiled_quant_traffic(summary: str, kernel: str):
    """DRAM bytes per launch of a quantiser from a committed ncu summary
    (`dram_bytes_per_launch: N`), or None when missing or stale."""
    v = profiled_quant_field(summary, "dram_bytes_per_launch")
    return None if v is None else int(v)


def max_over_ranks(value: float, world: int, device) -> float:
    """The largest of every rank's value (the job's time is its slowest rank's)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            mp = json.load(f)
        return {"hbm_gbs": mp["hbm_gbs"], "bf16_burst": mp["bf16_tflops"],
                "bf16_sustained": mp["bf16_tflops_sustained"], "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_burst": 1800.0, "bf16_sustained": 1400.0, "source": "fallback"}


# ---------------------------------------------------------------- workload
class Workload:
    def __init__(self, which: str, device):
        import torch
        from nvfp4_precision_02_b300 import workloads as wl
        from nvfp4_precision_02_b300 import binding as B
        self.B = B
        self.which = which
        self.dense = wl.ULTRA_DENSE if which == "ultra" else wl.SUPER_DENSE
        self.moe = wl.ULTRA_MOE if which == "ultra" else wl.SUPER_MOE
        d, m = self.dense, self.moe
        dev = device
        ins = wl.dense_inputs(d, which, device=dev)
        self.x, self.w, self.dy = ins["x"], ins["w"], ins["dy"]
        mi = wl.moe_inputs(m, which, device=dev)
        self.routing = mi["routing"]
        self.a, self.w_up, self.w_down = mi["a"], mi["w_up"], mi["w_down"]
        del mi["x_lat"]
        self.offsets = self.routing.offsets.to(dev)
        self.seed = wl.SEEDS["sr"]
        self.wseed = wl.wgrad_seed(self.seed)
        self.mask = wl.sign_mask_from_seed(wl.SEEDS["rht_sign"])
        T, K, N = d.tokens, d.hidden, d.out
        R, L, Hh, E = int(self.routing.offsets[-1]), m.latent, m.expert_hidden, m.experts
        self.R = R
        q = B.empty_qtensor
        self.qx = q(T, K, dev)
        self.qw = q(N, K, dev)
        self.qwt = q(K, N, dev)
        self.qdy = q(T, N, dev)
        self.sdy = q(N, T, dev)
        self.sx = q(K, T, dev)
        self.qwu = q(Hh, L, dev, batch=E, n_amax=E)
        self.qwd = q(L, Hh, dev, batch=E, n_amax=E)
        self.qa = q(R, L, dev, n_amax=E, sf_size=B.sf_bytes_grouped(R, L, E))
        self.qh = q(R, Hh, dev, n_amax=E, sf_size=B.sf_bytes_grouped(R, Hh, E))
        self.dy_amax = torch.empty(2, dtype=torch.float32, device=dev)
        self.dy_zeros = torch.empty(1, dtype=torch.int64, device=dev)
        self.y = torch.empty(T, N, dtype=torch.bfloat16, device=dev)
        self.dx = torch.empty(T, K, dtype=torch.bfloat16, device=dev)
        self.dw = torch.empty(N, K, dtype=torch.float32, device=dev)
        self.h = torch.empty(R, Hh, dtype=torch.bfloat16, device=dev)
        self.o = torch.empty(R, L, dtype=torch.bfloat16, device=dev)
        # per-op accounting: (name, kind, algorithmic work per step)
        gem = lambda M_, N_, K_: 2.0 * M_ * N_ * K_
        self.ops = [
            ("quantize_1d X (amax+RNE)", "hbm", 4.5625 * T * K),
            ("quantize_2d W (amax+W,W^T)", "hbm", 5.125 * N * K),
            ("gemm fprop", "tensor", gem(T, N, K)),
            ("dual amax dY (max |dY| and max |RHT(dY)|, one read)", "hbm", 2.0 * T * N),
            ("dual_sr_quantize dY (1x16 SR rows + RHT SR columns, one read)", "hbm", 3.125 * T * N),
            ("gemm dgrad", "tensor", gem(T, K, N)),
            ("rht_quantize X (amax+RNE)", "hbm", 4.5625 * T * K),
            ("gemm wgrad", "tensor", gem(N, K, T)),
            ("quantize_2d W_up, W_down (amax+W)", "hbm", 4.5625 * 2 * E * Hh * L),
            ("quantize_1d_grouped A", "hbm", 4.5625 * R * L),
            ("grouped_gemm up (+ per-expert amax of H)", "tensor", gem(R, Hh, L)),
            ("quantize_1d_grouped H (amax from the GEMM)", "hbm", 2.5625 * R * Hh),
            ("grouped_gemm down", "tensor", gem(R, L, Hh)),
        ]
        self.gemm_flops = sum(w_ for _, k, w_ in self.ops if k == "tensor")
        self.gemm_bytes = gemm_bytes_table(d, m, R)
        self.input_tensors = [self.x, self.w, self.dy, self.a, self.w_up, self.w_down]
        self.output_tensors = [self.y, self.dx, self.dw, self.o]

    def step(self, marks=None):
        """Enqueue one step; `marks(i)` is called after op i (event hooks)."""
        B = self.B
        mk = marks or (lambda i: None)
        B.quantize_1d(self.x, B.RNE, 0, out=self.qx); mk(0)
        B.quantize_2d(self.w, want_t=True, out=self.qw, out_t=self.qwt); mk(1)
        B.gemm(self.qx, self.qw, B.OUT_BF16, out=self.y); mk(2)
        # both tensor amaxes of dY (row SR quantiser, RHT quantiser) from one read,
        # then both SR operands (and the zero-code count) from one more
        B.dual_amax(self.dy, self.mask, out=self.dy_amax); mk(3)
        B.dual_sr_quantize(self.dy, self.mask, self.seed, self.wseed, self.dy_amax, out_row=self.qdy, out_t=self.sdy,
                           zero_count=self.dy_zeros); mk(4)
        self.qwt.amax = self.qw.amax
        B.gemm(self.qdy, self.qwt, B.OUT_BF16, out=self.dx); mk(5)
        B.rht_quantize(self.x, self.mask, B.RNE, 0, out=self.sx); mk(6)
        B.gemm(self.sdy, self.sx, B.OUT_FP32, out=self.dw); mk(7)
        B.quantize_2d(self.w_up, want_t=False, out=self.qwu)
        B.quantize_2d(self.w_down, want_t=False, out=self.qwd); mk(8)
        B.quantize_1d_grouped(self.a, self.offsets, B.RNE, 0, out=self.qa); mk(9)
        B.grouped_gemm(self.qa, self.offsets, self.qwu, self.moe.expert_hidden, B.OUT_BF16, out=self.h,
                       c_amax=self.qh.amax); mk(10)
        B.quantize_1d_grouped(self.h, self.offsets, B.RNE, 0, amax_in=self.qh.amax, out=self.qh); mk(11)
        B.grouped_gemm(self.qh, self.offsets, self.qwd, self.moe.latent, B.OUT_BF16, out=self.o); mk(12)


def gemm_bytes_table(d, m, R: int) -> dict:
    """Algorithmic bytes of each GEMM of the step: FP4 operands read once
    (0.5625 B per element: half a byte of code plus 1/16 B of block scale),
    every expert's weight read once, the output written once (bf16, or FP32
    for wgrad)."""
    T, K, N = d.tokens, d.hidden, d.out
    E, L, Hh = m.experts, m.latent, m.expert_hidden
    fp4 = 0.5625
    return {
        "gemm fprop": fp4 * (T + N) * K + 2.0 * T * N,
        "gemm dgrad": fp4 * (T + K) * N + 2.0 * T * K,
        "gemm wgrad": fp4 * (N + K) * T + 4.0 * N * K,
        "grouped_gemm up (+ per-expert amax of H)": fp4 * (R + E * Hh) * L + 2.0 * R * Hh,
        "grouped_gemm down": fp4 * (R + E * L) * Hh + 2.0 * R * L,
    }


def gemm_roofline(flops: float, nbytes, ms: float, hbm_gbs: float, fp4_tflops: float) -> dict:
    """The GEMM's roofline time max(bytes / HBM bandwidth, FLOPs / FP4 peak),
    which of the two bounds it, and the measured time's fraction of it."""
    if not nbytes or ms <= 0:
        return {}
    t_hbm = nbytes / (hbm_gbs * 1e9) * 1e3
    t_tc = flops / (fp4_tflops * 1e12) * 1e3
    t = max(t_hbm, t_tc)
    return {"bytes": int(nbytes), "bound": "hbm" if t_hbm > t_tc else "tensor", "roofline_ms": round(t, 4),
            "frac_roofline": round(t / ms, 4)}


# integer-ALU operations per element of one SR encoding, estimated from the
# source: about 10 for the rounding decision with its sign and packing, 2.5
# for Philox's three-input XORs (its multiplies run on the FMA pipe) and 3.5
# to unpack, find the block maximum and count zeros.  The ncu summaries of the
# SR kernels carry the counted figure (alu_ops_per_element), which the bench
# line reports beside this estimate while the kernel code is unchanged.
SR_ALU_OPS_PER_ELEMENT = 16
ALU_LANES_PER_SM = 64          # integer/logic lanes per SM per clock (4 partitions x 16)


def alu_roofline(elements: int, ms: float, sm_mhz, sms: int, ops_per_element: float = SR_ALU_OPS_PER_ELEMENT,
                 note: str = "operation count estimated from the source"):
    """ALU roof of an integer-bound kernel from an operation count per element:
    elements x ops / (lanes per SM x SMs x SM clock), against the measured time."""
    if not sm_mhz or ms <= 0 or sms <= 0:
        return None
    peak = ALU_LANES_PER_SM * sms * sm_mhz * 1e6            # lane-operations per second
    achieved = elements * ops_per_element / (ms * 1e-3)
    return {"bound": "alu", "unit": "Gop/s", "achieved": round(achieved / 1e9, 1), "peak": round(peak / 1e9, 1),
            "frac": round(achieved / peak, 4), "ops_per_element": ops_per_element,
            "floor_ms": round(elements * ops_per_element / peak * 1e3, 4),
            "note": note + ", clock = median SM clock of the timed region"}


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str):
        self.uuid = uuid
        self.proc = None
        self.f = None

    def start(self):
        try:
            self.f = tempfile.NamedTemporaryFile("w+", delete=False, suffix=".csv")
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
            if self.uuid:
                cmd += ["-i", self.uuid]
            self.proc = subprocess.Popen(cmd, stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.flush()
        self.f.seek(0)
        text = self.f.read()
        os.unlink(self.f.name)
        return summarise_clocks(text)


THROTTLE_NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")


def summarise_clocks(text: str):
    """Median SM clock, maximum SM clock, the throttle reasons seen Active and
    the peak power from `nvidia-smi --query-gpu=<ClockSampler.FIELDS>
    --format=csv,noheader,nounits` output; rows that do not parse are
    skipped.  None when no row parses."""
    sm, power = [], []
    reasons = set()
    smax = None
    for line in text.splitlines():
        r = [v.strip() for v in line.split(",")]
        if len(r) < 8:
            continue
        try:
            mhz, mx = float(r[0]), float(r[1])
        except ValueError:
            continue
        sm.append(mhz)
        smax = mx
        try:
            power.append(float(r[2]))
        except ValueError:
            pass
        for n, v in zip(THROTTLE_NAMES, r[4:8]):
            if v.lower() == "active":
                reasons.add(n)
    if not sm:
        return None
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
            "samples": len(sm), "power_w_max": max(power) if power else None}


# ---------------------------------------------------------------- CPU oracle timing
def oracle_sample(which: str, budget_s: float):
    """Time the oracle on bounded slices of every op of the step and
    extrapolate by element / multiply-add counts.  Each op is timed once on a
    small slice, then once on a slice sized to take about budget_s / 5
    seconds, which gives the reported rate.  Returns (seconds per full step,
    description, threads)."""
    import torch
    import oracle as orc
    from nvfp4_precision_02_b300 import workloads as wl
    d = wl.ULTRA_DENSE if which == "ultra" else wl.SUPER_DENSE
    m = wl.ULTRA_MOE if which == "ultra" else wl.SUPER_MOE
    orc.build()
    T, K, N = d.tokens, d.hidden, d.out
    R = m.tokens * m.topk
    E, L, Hh = m.experts, m.latent, m.expert_hidden
    g = torch.Generator().manual_seed(0)
    target = budget_s / 5.0

    def timed(fn, units):
        t0 = time.perf_counter()
        fn()
        return (time.perf_counter() - t0), units

    def grow(make, n0, nmax, power=1):
        dt, _ = make(n0)
        n = int(n0 * (target / max(dt, 1e-4)) ** (1.0 / power))
        n = max(n0, min(nmax, n // 16 * 16))
        dt, units = make(n)
        return dt / units, n

    def q_op(kind):
        def make(rows):
            if kind == "q1d_rne":
                x = torch.randn(rows, K, generator=g).to(torch.bfloat16)
                return timed(lambda: orc.quantize_1d(x), x.numel())
            if kind == "q2d":
                x = torch.randn(rows, K, generator=g).to(torch.bfloat16)
                return timed(lambda: orc.quantize_2d(x), x.numel())
            x = (torch.randn(rows, N, generator=g) * 1e-3).to(torch.bfloat16)
            if kind == "q1d_sr":
                return timed(lambda: orc.quantize_1d(x, orc.SR, 7), x.numel())
            return timed(lambda: orc.rht_quantize(x, 0x1234, orc.SR, 9), x.numel())
        return make

    per, sizes = {}, {}
    for kind in ("q1d_rne", "q1d_sr", "q2d", "rht"):
        per[kind], sizes[kind] = grow(q_op(kind), 64, T)

    def gemm_make(mm):
        A = torch.randn(mm, K, generator=g, dtype=torch.float64).numpy()
        Bm = torch.randn(mm, K, generator=g, dtype=torch.float64).numpy()
        return timed(lambda: orc.gemm(A, Bm), mm * mm * K)

    per["gemm_mac"], mm = grow(gemm_make, 32, 4096, power=2)
    elems = {"q1d_rne": T * K + R * L + R * Hh, "q1d_sr": T * N, "q2d": N * K + 2 * E * Hh * L,
             "rht": T * N + T * K}
    macs = T * N * K * 3 + 2 * R * Hh * L
    sec = sum(per[k] * v for k, v in elems.items()) + per["gemm_mac"] * macs
    desc = (f"oracle on {sizes['q1d_rne']}/{sizes['q1d_sr']}/{sizes['q2d']}/{sizes['rht']} rows of the step's "
            f"X [.,{K}] / dY [.,{N}] for 1D RNE / 1D SR / 2D / RHT+SR and a {mm}x{mm}x{K} FP64 GEMM, each slice "
            f"sized to take about {target:.1f} s; per-element and per-multiply-add times extrapolated to the "
            f"full step")
    return sec, desc, orc.num_threads()


# ---------------------------------------------------------------- main
def relaunch_ranks(n: int, argv) -> int:
    """Start n ranks of this script on this node with torch.distributed.run
    (rendezvous on 127.0.0.1) and return their exit status; used when
    --gpus N > 1 is given without a launcher (no WORLD_SIZE in the
    environment)."""
    import socket
    with socket.socket() as s_:
        s_.bind(("127.0.0.1", 0))
        port = s_.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr=127.0.0.1", f"--master-port={port}", os.path.abspath(__file__)] + list(argv)
    return subprocess.call(cmd)


def fp4_peaks(pk: dict, sms: int, sm_mhz) -> dict:
    """Dense FP4 denominators of the GEMM fractions: the measured bf16 burst
    and sustained rates x 6 (the nominal FP4:BF16 ratio), the 13.5 PFLOP/s
    datasheet figure, and, at the median SM clock of the timed region, the
    measured issue rate of the block-scaled MMA and ncu's counter peak."""
    out = {"burst_x6": pk["bf16_burst"] * FP4_OVER_BF16, "sustained_x6": pk["bf16_sustained"] * FP4_OVER_BF16,
           "datasheet": FP4_DATASHEET_TFLOPS}
    if sm_mhz and sms:
        out["mma_issue_at_clock"] = FP4_FLOP_PER_CLK_SM * sms * sm_mhz * 1e6 / 1e12
        out["counter_at_clock"] = FP4_FLOP_PER_CLK_SM_COUNTER * sms * sm_mhz * 1e6 / 1e12
    return out


def gemm_fracs(tflops: float, fp4: dict) -> dict:
    return {f"frac_fp4_{k}": round(tflops / v, 4) for k, v in fp4.items()}


def hbm_fracs(gbs: float, pk: dict) -> dict:
    return {"frac_hbm": round(gbs / pk["hbm_gbs"], 4), "frac_hbm_nominal_8tbs": round(gbs / HBM_NOMINAL_GBS, 4)}


def op_entry(kind: str, work: float, ms: float, pk: dict, fp4: dict, nbytes=None) -> dict:
    """One op's time and rate with its fractions: TFLOP/s against every FP4
    denominator (and its roofline when its bytes are known) for a GEMM, GB/s
    against the measured and the nominal HBM bandwidth for a quantiser."""
    if kind == "tensor":
        tf = work / (ms * 1e-3) / 1e12
        e = {"ms": round(ms, 4), "tflops": round(tf, 1), **gemm_fracs(tf, fp4)}
        if nbytes:
            e.update(gemm_roofline(work, nbytes, ms, pk["hbm_gbs"], fp4["burst_x6"]))
        return e
    gbs = work / (ms * 1e-3) / 1e9
    return {"ms": round(ms, 4), "gbs": round(gbs, 1), **hbm_fracs(gbs, pk)}


def time_ops(wk, steps: int = 5):
    """Median CUDA-event time of each op of wk's step over `steps` steps."""
    import torch
    nops = len(wk.ops)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nops + 1)] for _ in range(steps)]
    torch.cuda.synchronize()
    for s_ in range(steps):
        ev[s_][0].record()
        wk.step(marks=lambda i, s_=s_: ev[s_][i + 1].record())
    torch.cuda.synchronize()
    return [statistics.median(ev[s_][i].elapsed_time(ev[s_][i + 1]) for s_ in range(steps)) for i in range(nops)]


# the ops of the Workload step that make up each stated configuration
CONFIG_OPS = {"c2": (0, 3), "c3": (3, 8), "c4": (8, 13)}


def measure_configs(dev, pk: dict, fp4: dict, super_wk=None, steps: int = 5) -> dict:
    """Configurations 1-4 timed on their own shapes after the timed region:
    c1 the 256 x 256 tiny fprop (1D RNE A, 16x16 W, GEMM); c2-c4 the ops of a
    Super-shaped step -- c2 the in_proj fprop (X 8192 x 6144 with outliers,
    W 18560 x 6144), c3 its backward (SR dY, dgrad, RHT wgrad), c4 the
    LatentMoE (1024 -> 2688 -> 1024, 180224 routed rows).  Each op's median
    CUDA-event time with its rate and fractions; each config's total."""
    import torch
    from nvfp4_precision_02_b300 import binding as B, workloads as wl
    out = {}
    a, w = (t.to(dev) for t in wl.tiny_inputs())
    qa = B.quantize_1d(a)
    qw = B.quantize_2d(w)[0]
    y = torch.empty(256, 256, dtype=torch.bfloat16, device=dev)
    tiny = [("quantize_1d A (amax+RNE)", "hbm", 4.5625 * 256 * 256, lambda: B.quantize_1d(a, out=qa)),
            ("quantize_2d W (amax+W)", "hbm", 4.5625 * 256 * 256, lambda: B.quantize_2d(w, want_t=False, out=qw)),
            ("gemm fprop", "tensor", 2.0 * 256 ** 3, lambda: B.gemm(qa, qw, B.OUT_BF16, out=y))]
    c1 = {}
    for name, kind, work, fn in tiny:
        fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(50):
            fn()
        e1.record()
        torch.cuda.synchronize()
        c1[name] = op_entry(kind, work, e0.elapsed_time(e1) / 50, pk, fp4,
                            0.5625 * 512 * 256 + 2 * 256 * 256 if kind == "tensor" else None)
    out["c1_tiny_fprop_256"] = {"ops": c1, "ms": round(sum(v["ms"] for v in c1.values()), 4),
                                "note": "launch-bound: 50 back-to-back calls per op"}
    own = super_wk is None
    wk = Workload("super", dev) if own else super_wk
    steady_ms(wk.step, warm_ms=30.0, timed_ms=0.0, min_iters=1)     # out of the idle state first
    ms = time_ops(wk, steps)
    names = {"c2": "c2_super_in_proj_fprop", "c3": "c3_super_backward", "c4": "c4_super_latent_moe"}
    for key, (i0, i1) in CONFIG_OPS.items():
        ops = {}
        for i in range(i0, i1):
            n, kind, work = wk.ops[i]
            ops[n] = op_entry(kind, work, ms[i], pk, fp4, wk.gemm_bytes.get(n))
        flops = sum(wk.ops[i][2] for i in range(i0, i1) if wk.ops[i][1] == "tensor")
        t = sum(ms[i0:i1])
        out[names[key]] = {"ops": ops, "ms": round(t, 4), "gemm_tflops_incl_quantisers": round(flops / (t * 1e-3) / 1e12, 1)}
    out["c5_ultra_full_step"] = "the step of this line (ops, roofline)"
    if own:
        del wk
        torch.cuda.empty_cache()
    return out


def launch_check(args, world: int, rank: int) -> int:
    """The multi-rank launch path without GPU work: every rank joins the
    process group (gloo without CUDA), meets the others at a barrier, times
    an empty region, and rank 0 prints n_gpus = the ranks that ran."""
    import torch
    import torch.distributed as dist
    if world > 1:
        dist.init_process_group("gloo")
        dist.barrier()
    t0 = time.perf_counter()
    if world > 1:
        dist.barrier()
    ms = max_over_ranks((time.perf_counter() - t0) * 1e3 + rank, world, "cpu")
    n = world
    if world > 1:
        t = torch.tensor([1.0])
        dist.all_reduce(t)
        n = int(t.item())
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps({"launch_check": True, "n_gpus": n, "world_size": world, "max_ms": round(ms, 3)}), flush=True)
    return 0


def main(argv=None):
    argv = sys.argv[1:] if argv is None else argv
    args = parse(argv)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        return relaunch_ranks(args.gpus, argv)
    if args.launch_check:
        return launch_check(args, world, rank)

    if args.impl == "reference":
        if rank != 0:
            return 0
        return reference_arm(args)

    import torch
    from nvfp4_precision_02_b300 import binding as B, build as nb
    nb.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    B.lib()

    wk = Workload(args.workload, dev)
    torch.cuda.synchronize()
    for _ in range(max(args.warmup, 0)):
        wk.step()
    torch.cuda.synchronize()
    if B.device_status() != 0:
        raise RuntimeError("device status word set during warm-up")

    nops = len(wk.ops)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nops + 1)] for _ in range(args.steps)]
    props = torch.cuda.get_device_properties(dev)
    sms = getattr(props, "multi_processor_count", 0)
    uuid = str(getattr(props, "uuid", ""))
    if uuid and not uuid.startswith("GPU-"):
        uuid = "GPU-" + uuid
    clocks = ClockSampler(uuid)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    launches0 = B.launch_count()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record()
    for s in range(args.steps):
        ev[s][0].record()
        wk.step(marks=lambda i, s=s: ev[s][i + 1].record())
    end.record()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    launches = B.launch_count() - launches0
    clk = clocks.stop()
    total_ms = max_over_ranks(start.elapsed_time(end), world, dev)
    ms_step = total_ms / args.steps
    op_ms = [statistics.median(ev[s][i].elapsed_time(ev[s][i + 1]) for s in range(args.steps))
             for i in range(nops)]
    status = B.device_status()

    pk = peaks()
    sm_mhz = (clk or {}).get("sm_mhz")
    fp4 = fp4_peaks(pk, sms, sm_mhz)
    value = wk.gemm_flops * world / (ms_step * 1e-3) / 1e12
    gemm_ms = sum(t for (n, k, _), t in zip(wk.ops, op_ms) if k == "tensor")
    quant_ms = sum(t for (n, k, _), t in zip(wk.ops, op_ms) if k == "hbm")
    quant_bytes = sum(w for _, k, w in wk.ops if k == "hbm")
    ops = {n: op_entry(k, w, t, pk, fp4, wk.gemm_bytes.get(n)) for (n, k, w), t in zip(wk.ops, op_ms)}
    # dominant kernel: k_gemm_nvfp4; its roofline is given for the fprop launch
    fprop_i = [n for n, _, _ in wk.ops].index("gemm fprop")
    fprop_flops = wk.ops[fprop_i][2]
    achieved = fprop_flops / (op_ms[fprop_i] * 1e-3) / 1e12
    traffic = profiled_traffic(f"k_gemm_nvfp4_fprop_{args.workload}.md")
    roofline = {"kernel": "k_gemm_nvfp4 (fprop launch)", "bound": "tensor",
                "achieved": round(achieved, 1), "peak": round(fp4["burst_x6"], 1), "unit": "TFLOP/s",
                "frac": round(achieved / fp4["burst_x6"], 4),
                "peak_note": f"{pk['source']} burst bf16 x {FP4_OVER_BF16:g} (nominal dense FP4:BF16); "
                             "frac_fp4_* give the same launch against the other denominators",
                **gemm_fracs(achieved, fp4),
                "clock_mhz_median": sm_mhz,
                "traffic": traffic, "traffic_unit": "bytes per launch (ncu dram read + write)",
                "algorithmic_bytes": int(0.5625 * (wk.dense.tokens + wk.dense.out) * wk.dense.hidden
                                         + 2 * wk.dense.tokens * wk.dense.out)}
    qi = [n for n, _, _ in wk.ops].index("dual_sr_quantize dY (1x16 SR rows + RHT SR columns, one read)")
    q_dy = op_ms[qi]
    q_gbs = wk.ops[qi][2] / (q_dy * 1e-3) / 1e9
    roofline_q = {"kernel": "k_rht<4> (dY: 1x16 SR rows and RHT SR columns from one read, amaxes supplied)",
                  "bound": "hbm",
                  "achieved": round(q_gbs, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                  "frac": round(q_gbs / pk["hbm_gbs"], 4), "frac_hbm_nominal_8tbs": round(q_gbs / HBM_NOMINAL_GBS, 4),
                  "peak_note": "HBM copy bandwidth (measured)",
                  "traffic": profiled_quant_traffic(f"k_rht_dual_sr_{args.workload}.md", "k_rht"),
                  "alu_estimate": alu_roofline(wk.dense.tokens * wk.dense.out, q_dy, sm_mhz, sms,
                                               2 * SR_ALU_OPS_PER_ELEMENT)}
    alu_counted = profiled_quant_field(f"k_rht_dual_sr_{args.workload}.md", "alu_ops_per_element")
    if alu_counted is not None:
        roofline_q["alu_counted"] = alu_roofline(
            wk.dense.tokens * wk.dense.out, q_dy, sm_mhz, sms, alu_counted,
            note="ALU-pipe operations per element counted by ncu (smsp__inst_executed_pipe_alu.sum x 32 / elements)")

    supplied = measure_supplied_amax(wk, pk)
    zeros = int(wk.dy_zeros.item())
    zero_frac = zeros / float(wk.dense.tokens * wk.dense.out)
    next_rows = measure_next_rows(wk, pk, fp4)
    configs = None
    if not args.no_configs:
        configs = measure_configs(dev, pk, fp4, super_wk=wk if args.workload == "super" else None)

    e2e = None
    if not args.no_e2e and args.e2e_steps > 0:
        e2e = measure_e2e(wk, args.e2e_steps, dev)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        sec, desc, th = oracle_sample(args.workload, budget_s=15.0)
        cpu = {"value": round(wk.gemm_flops / sec / 1e12, 9), "unit": "TFLOP/s", "cores": th,
               "kind": "oracle", "sample": desc, "seconds_per_step_extrapolated": round(sec, 1)}

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "nvfp4",
        "data": "synthetic (seeded device generators; no dataset)",
        "config": workload_config(args.workload, wk.dense, wk.moe, wk.R, world),
        "gemm_tflops": round(wk.gemm_flops / (gemm_ms * 1e-3) / 1e12, 1),
        "quantize_gbs": round(quant_bytes / (quant_ms * 1e-3) / 1e9, 1),
        "quantize_frac_hbm": round(quant_bytes / (quant_ms * 1e-3) / 1e9 / pk["hbm_gbs"], 4),
        "quantize_frac_hbm_nominal_8tbs": round(quant_bytes / (quant_ms * 1e-3) / 1e9 / HBM_NOMINAL_GBS, 4),
        "fp4_peaks_tflops": {k: round(v, 1) for k, v in fp4.items()},
        "ops": ops, "roofline": roofline, "roofline_quantize": roofline_q,
        "quantize_supplied_amax": supplied,
        "configs": configs,
        "dy_zero_code_fraction": round(zero_frac, 6),
        "next_rows": next_rows,
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": int(launches), "clocks": clk,
        "device_status": status, "routing": {"max_vio": round(wk.routing.max_vio, 3),
                                             "empty_experts": int((wk.routing.counts == 0).sum())},
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def host_mem_available() -> int:
    """MemAvailable of /proc/meminfo in bytes (0 if unreadable)."""
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 0


def steady_ms(fn, warm_ms: float = 30.0, timed_ms: float = 10.0, min_iters: int = 5) -> float:
    """CUDA-event time per call of fn in steady state.  The calls run back to
    back for at least warm_ms first, then enough calls to cover timed_ms are
    timed.  After a pause, the first milliseconds of work run slower even with
    the SM clock at its maximum: on a B300, the Ultra X quantiser took
    0.073 ms per call after its inputs were generated and 0.123 ms after 5 s
    idle, each timed over 5 calls."""
    import torch
    fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    fn()
    e1.record()
    torch.cuda.synchronize()
    est = max(e0.elapsed_time(e1), 1e-3)
    for _ in range(max(1, math.ceil(warm_ms / est))):
        fn()
    n = max(min_iters, math.ceil(timed_ms / est))
    e0.record()
    for _ in range(n):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / n


def measure_supplied_amax(wk: Workload, pk: dict, iters: int = 5):
    """Each quantiser of the step with its amax supplied (the step's own
    amaxes, already in the output tensors), timed alone after the timed
    region: one HBM read of the input, so the algorithmic bytes are 2.5625 per
    element (3.125 with the transposed 2D copy).  Not part of the step."""
    import torch
    B = wk.B
    d, m = wk.dense, wk.moe
    T, K, N = d.tokens, d.hidden, d.out
    E, L, Hh, R = m.experts, m.latent, m.expert_hidden, wk.R
    cases = [
        ("quantize_1d X (RNE)", 2.5625 * T * K, lambda: B.quantize_1d(wk.x, B.RNE, 0, amax_in=wk.qx.amax, out=wk.qx)),
        ("quantize_1d dY (SR)", 2.5625 * T * N,
         lambda: B.quantize_1d(wk.dy, B.SR, wk.seed, amax_in=wk.qdy.amax, out=wk.qdy)),
        ("quantize_2d W (W, W^T)", 3.125 * N * K,
         lambda: B.quantize_2d(wk.w, want_t=True, amax_in=wk.qw.amax, out=wk.qw, out_t=wk.qwt)),
        ("quantize_2d W_up (batched, W)", 2.5625 * E * Hh * L,
         lambda: B.quantize_2d(wk.w_up, want_t=False, amax_in=wk.qwu.amax, out=wk.qwu)),
        ("rht_quantize dY (SR)", 2.5625 * T * N,
         lambda: B.rht_quantize(wk.dy, wk.mask, B.SR, wk.wseed, amax_in=wk.sdy.amax, out=wk.sdy)),
        ("dual_sr_quantize dY (rows and RHT columns, SR)", 3.125 * T * N,
         lambda: B.dual_sr_quantize(wk.dy, wk.mask, wk.seed, wk.wseed, wk.dy_amax, out_row=wk.qdy, out_t=wk.sdy,
                                    zero_count=wk.dy_zeros)),
        ("rht_quantize X (RNE)", 2.5625 * T * K,
         lambda: B.rht_quantize(wk.x, wk.mask, B.RNE, 0, amax_in=wk.sx.amax, out=wk.sx)),
        ("quantize_1d_grouped A (RNE)", 2.5625 * R * L,
         lambda: B.quantize_1d_grouped(wk.a, wk.offsets, B.RNE, 0, amax_in=wk.qa.amax, out=wk.qa)),
        ("quantize_1d_grouped H (RNE)", 2.5625 * R * Hh,
         lambda: B.quantize_1d_grouped(wk.h, wk.offsets, B.RNE, 0, amax_in=wk.qh.amax, out=wk.qh)),
    ]
    out = {}
    for name, nbytes, fn in cases:
        out[name] = op_entry("hbm", nbytes, steady_ms(fn, min_iters=iters), pk, {})
    return out


def measure_next_rows(wk: Workload, pk: dict, fp4: dict, iters: int = 3):
    """The grouped backward of the LatentMoE up-projection, timed alone after
    the timed region (not part of the step): dgrad dA = dH . W_up per expert
    (W_up^T from the batched 2D quantiser, dH in 1x16 SR) and wgrad
    dW_up = RHT(dH)^T . RHT(A) per expert (expert-segmented RHT quantisers,
    groups along K, FP32 dW).  The step's H stands in for dH.  Also the FP16
    stochastic rounding of an SSM cache (FP32 in, FP16 out)."""
    import torch
    B = wk.B
    m = wk.moe
    E, L, Hh, R = m.experts, m.latent, m.expert_hidden, wk.R
    dev = wk.h.device
    dh = wk.h
    qdh = B.quantize_1d_grouped(dh, wk.offsets, B.SR, wk.seed)
    qwt = B.quantize_2d(wk.w_up, want_t=True)[1]
    da = torch.empty(R, L, dtype=torch.bfloat16, device=dev)
    kt = B.group_k_capacity(R, E)
    sdh = B.empty_qtensor(Hh, kt, dev, n_amax=E)
    sa = B.empty_qtensor(L, kt, dev, n_amax=E)
    dw = torch.empty(E * Hh, L, dtype=torch.float32, device=dev)
    gem = 2.0 * R * Hh * L
    cases = [
        ("grouped_gemm dgrad (dA = dH . W_up)", "tensor", gem,
         lambda: B.grouped_gemm(qdh, wk.offsets, qwt, L, B.OUT_BF16, out=da)),
        ("rht_quantize_grouped dH (amax + SR)", "hbm", 4.5625 * R * Hh,
         lambda: B.rht_quantize_grouped(dh, wk.offsets, wk.mask, B.SR, wk.wseed, kt=kt, out=sdh)),
        ("rht_quantize_grouped A (amax + RNE)", "hbm", 4.5625 * R * L,
         lambda: B.rht_quantize_grouped(wk.a, wk.offsets, wk.mask, B.RNE, 0, kt=kt, out=sa)),
        ("grouped_gemm_k wgrad (dW_up, FP32)", "tensor", gem,
         lambda: B.grouped_gemm_k(sdh, sa, wk.offsets, B.OUT_FP32, out=dw)),
    ]
    out = {}
    for name, kind, work, fn in cases:
        out[name] = op_entry(kind, work, steady_ms(fn, min_iters=iters), pk, fp4)
    # PTQ block scales by minimum squared error (next row f3) on the in_proj weight
    qptq = B.empty_qtensor(wk.dense.out, wk.dense.hidden, dev)
    B.quantize_1d_mse(wk.w, amax_in=wk.qw.amax, out=qptq)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    B.quantize_1d_mse(wk.w, amax_in=wk.qw.amax, out=qptq)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    nel = wk.dense.out * wk.dense.hidden
    out["quantize_1d_mse W (PTQ scales, 126 trial scales per block)"] = {
        "ms": round(ms, 4), "gbs": round(2.5625 * nel / (ms * 1e-3) / 1e9, 1),
        "g_elements_per_s": round(nel / (ms * 1e-3) / 1e9, 2)}
    del qptq
    # FP16 SR of an SSM cache (next row f4): 256 sequences x 256 heads x 64 x state 128, FP32 in
    ssm = torch.randn(256 * 256 * 64 * 128, device=dev)
    ssm16 = torch.empty(ssm.numel(), dtype=torch.float16, device=dev)
    ms = steady_ms(lambda: B.sr_fp16(ssm, 5, out=ssm16), min_iters=iters)
    out["sr_fp16 SSM cache (FP32 -> FP16, 6 B / element)"] = op_entry("hbm", 6.0 * ssm.numel(), ms, pk, fp4)
    del ssm, ssm16
    # the wgrad writes E * Hh * L FP32 outputs: its HBM roof
    w = out["grouped_gemm_k wgrad (dW_up, FP32)"]
    wbytes = 4.0 * E * Hh * L + 0.5625 * (Hh + L) * kt
    w["hbm_gbs"] = round(wbytes / (w["ms"] * 1e-3) / 1e9, 1)
    w["frac_hbm"] = round(w["hbm_gbs"] / pk["hbm_gbs"], 4)
    del qdh, qwt, da, sdh, sa, dw
    torch.cuda.empty_cache()
    return out


def measure_e2e(wk: Workload, steps: int, dev):
    """Same metric through the public API with host buffers: every step copies
    all inputs from pinned host memory, runs the step and reads every output
    back.  Skipped (None) when pinned host memory for it is not available."""
    import torch
    in_bytes = sum(t.numel() * t.element_size() for t in wk.input_tensors)
    out_bytes = sum(t.numel() * t.element_size() for t in wk.output_tensors)
    avail = host_mem_available()
    if avail < 2 * (in_bytes + out_bytes):
        return {"value": None, "unit": "TFLOP/s", "h2d_bytes_per_step": in_bytes, "d2h_bytes_per_step": out_bytes,
                "skipped": f"needs {2 * (in_bytes + out_bytes) / 1e9:.0f} GB free host memory, {avail / 1e9:.0f} GB available"}
    host_in = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in wk.input_tensors]
    host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in wk.output_tensors]
    for h, t in zip(host_in, wk.input_tensors):
        h.copy_(t)
    torch.cuda.synchronize()
    s0 = torch.cuda.Event(enable_timing=True)
    s1 = torch.cuda.Event(enable_timing=True)
    s0.record()
    for _ in range(steps):
        for h, t in zip(host_in, wk.input_tensors):
            t.copy_(h, non_blocking=True)
        wk.step()
        for h, t in zip(host_out, wk.output_tensors):
            h.copy_(t, non_blocking=True)
    s1.record()
    torch.cuda.synchronize()
    ms = s0.elapsed_time(s1) / steps
    del host_in, host_out
    return {"value": round(wk.gemm_flops / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s", "ms_per_step": round(ms, 2),
            "h2d_bytes_per_step": in_bytes, "d2h_bytes_per_step": out_bytes, "steps": steps}


def reference_arm(args):
    """The CPU oracle as the reference arm: each step runs a bounded sample of
    the workload on the host cores (sized so the whole run stays within a few
    minutes); value is the full step's GEMM FLOPs over the extrapolated time
    of a full step, averaged over the timed steps."""
    budget = max(0.5, min(4.0, 120.0 / max(1, args.steps + args.warmup)))
    secs, walls = [], []
    desc, th = "", 1
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        sec, desc, th = oracle_sample(args.workload, budget_s=budget)
        if i >= args.warmup:
            secs.append(sec)
            walls.append(time.perf_counter() - t0)
    from nvfp4_precision_02_b300 import workloads as wl
    d = wl.ULTRA_DENSE if args.workload == "ultra" else wl.SUPER_DENSE
    m = wl.ULTRA_MOE if args.workload == "ultra" else wl.SUPER_MOE
    R = m.tokens * m.topk
    flops = 3 * 2.0 * d.tokens * d.out * d.hidden + 2 * 2.0 * R * m.expert_hidden * m.latent
    sec = statistics.mean(secs)
    value = flops / sec / 1e12
    config = workload_config(args.workload, d, m, R, 1)
    line = {"metric": METRIC, "value": round(value, 9), "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec * 1e3, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference", "config": config,
            "cpu_baseline": {"value": round(value, 9), "unit": "TFLOP/s", "cores": th, "kind": "oracle",
                             "sample": desc, "sample_wall_s_per_step": round(statistics.mean(walls), 2)},
            "e2e": {"value": round(value, 9), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def workload_config(which, d, m, rows, world):
    return {"workload": f"{which}_full_step", "dense_tokens": d.tokens, "hidden": d.hidden,
            "in_proj_out": d.out, "moe_tokens": m.tokens, "moe_latent": m.latent,
            "moe_expert_hidden": m.expert_hidden, "experts": m.experts, "topk": m.topk,
            "moe_rows": rows, "parallelism": f"replicas x{world}",
            "l2": "inputs larger than L2 (tens of GB streamed per step); no flush"}


if __name__ == "__main__":
    sys.exit(main())
