"""Seeded synthetic inputs for the NVFP4 linear-layer workloads.

This module only draws inputs; it holds none of the quantisation or GEMM
arithmetic, so both the CUDA path and the CPU oracle may use it.

Shapes follow the pages: Mamba-2 in_proj of Nemotron 3 Super (hidden 6144,
128 heads x 64, 8 groups x state 128 -- "Nemotron 3 Super -- technical report
summary", section 1 table) and of Ultra (hidden 8192, 256 heads x 64 --
"Nemotron 3 Ultra -- technical report summary", section 1 table); LatentMoE
with 512 experts, top-22 routing, latent 1024 / expert hidden 2688 (Super)
and latent 2048 / hidden 5120 (Ultra).  in_proj output width is
2*d_inner + 2*groups*state + heads (z, x, B, C, dt).

Recipe (all draws from ``torch.Generator`` seeded as stated; tensors are
drawn in FP32 and rounded once to bf16):
  * activations ~ N(0, 1); 0.1% of channels (round(0.001*K)) multiplied by 50,
    the channels taken from ``randperm(K)`` of the same generator after the
    values;
  * weights ~ N(0, 0.02); gradients dY ~ N(0, 1e-3);
  * routing: expert popularity w_r = r^-1.1 (r = 1..E) assigned to expert ids
    by a seeded permutation; every token takes k distinct experts by
    Gumbel-top-k on log w + Gumbel noise; assignments are sorted expert-major
    (stable in token id), giving per-expert offsets (empty experts allowed).
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal_bf16(shape, std: float, seed: int, device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def activations_with_outliers(rows: int, cols: int, seed: int, device="cpu",
                              frac: float = 0.001, factor: float = 50.0) -> torch.Tensor:
    """N(0,1) activations with round(frac*cols) channels scaled by ``factor``."""
    g = _gen(seed, device)
    x = torch.randn(rows, cols, generator=g, device=device, dtype=torch.float32)
    n_out = int(round(frac * cols))
    if n_out > 0:
        ch = torch.randperm(cols, generator=g, device=device)[:n_out]
        x[:, ch] *= factor
    return x.to(torch.bfloat16)


def batched_normal_bf16(batch: int, rows: int, cols: int, std: float, seed: int,
                        device="cpu") -> torch.Tensor:
    """[batch, rows, cols]; one generator, one draw per batch entry in order
    (keeps the FP32 temporary at one entry)."""
    g = _gen(seed, device)
    out = torch.empty(batch, rows, cols, device=device, dtype=torch.bfloat16)
    for b in range(batch):
        out[b] = (torch.randn(rows, cols, generator=g, device=device, dtype=torch.float32)
                  .mul_(std).to(torch.bfloat16))
    return out


@dataclass
class Routing:
    token_ids: torch.Tensor     # [R] int64, expert-major, stable in token id
    expert_ids: torch.Tensor    # [R] int64
    offsets: torch.Tensor       # [E+1] int64
    counts: torch.Tensor        # [E] int64
    topk: int

    @property
    def max_vio(self) -> float:
        """MaxVio = max_i T_i / mean_i T_i (Ultra report, section 2.7)."""
        c = self.counts.to(torch.float64)
        return float(c.max() / c.mean())


def zipf_routing(tokens: int, experts: int, topk: int, seed: int, s: float = 1.1) -> Routing:
    """Top-k of E experts per token under a Zipf(s) popularity (CPU)."""
    g = _gen(seed, "cpu")
    perm = torch.randperm(experts, generator=g)
    w = torch.empty(experts, dtype=torch.float64)
    w[perm] = torch.arange(1, experts + 1, dtype=torch.float64).pow(-s)
    logw = w.log()
    u = torch.rand(tokens, experts, generator=g, dtype=torch.float64).clamp_(1e-300, 1.0)
    gumbel = -torch.log(-torch.log(u))
    choice = torch.topk(logw[None, :] + gumbel, topk, dim=1).indices      # [T, k]
    tok = torch.arange(tokens, dtype=torch.int64)[:, None].expand(tokens, topk).reshape(-1)
    exp = choice.reshape(-1).to(torch.int64)
    order = torch.argsort(exp * tokens + tok)                              # expert-major, stable
    exp_sorted = exp[order]
    tok_sorted = tok[order]
    counts = torch.bincount(exp_sorted, minlength=experts).to(torch.int64)
    offsets = torch.zeros(experts + 1, dtype=torch.int64)
    offsets[1:] = torch.cumsum(counts, 0)
    return Routing(tok_sorted, exp_sorted, offsets, counts, topk)


def sign_mask_from_seed(seed: int) -> int:
    """A 16-bit random sign pattern for the Hadamard transform, drawn from a
    seeded torch generator (shared by both wgrad operands)."""
    g = _gen(seed, "cpu")
    return int(torch.randint(0, 1 << 16, (1,), generator=g).item())


# ---------------------------------------------------------------- configs
@dataclass(frozen=True)
class DenseShape:
    tokens: int       # M of fprop/dgrad, K of wgrad
    hidden: int       # K of fprop
    out: int          # N of fprop


@dataclass(frozen=True)
class MoEShape:
    tokens: int
    latent: int
    expert_hidden: int
    experts: int = 512
    topk: int = 22


def in_proj_width(d_model: int, heads: int, head_dim: int = 64, groups: int = 8,
                  state: int = 128) -> int:
    """Mamba-2 in_proj output width: z and x (heads*head_dim each), B and C
    (groups*state each), dt (heads)."""
    d_inner = heads * head_dim
    return 2 * d_inner + 2 * groups * state + heads


SUPER_DENSE = DenseShape(tokens=8192, hidden=6144, out=in_proj_width(6144, 128))      # N = 18560
# Ultra: the workload definition states N = 33024 for "2*16384 + 2*8*128 + 256",
# whose terms sum to 35072 (= in_proj_width(8192, 256)); the stated 33024 is
# used, as every FLOP count of that workload assumes it.
ULTRA_DENSE = DenseShape(tokens=16384, hidden=8192, out=33024)
SUPER_MOE = MoEShape(tokens=8192, latent=1024, expert_hidden=2688)
ULTRA_MOE = MoEShape(tokens=16384, latent=2048, expert_hidden=5120)

SEEDS = {
    "tiny": 0,
    "super_x": 1, "super_w": 2, "super_dy": 3, "super_moe_x": 4, "super_moe_w": 5,
    "ultra_x": 6, "ultra_w": 61, "ultra_dy": 62, "ultra_moe": 8, "ultra_moe_w": 81,
    "sr": 7, "rht_sign": 11,
}
# The wgrad copy of dY uses a second SR stream: the seed XOR a fixed odd
# 64-bit constant (the golden-ratio constant 0x9E3779B97F4A7C15).
WGRAD_SEED_XOR = 0x9E3779B97F4A7C15


def wgrad_seed(seed: int) -> int:
    return seed ^ WGRAD_SEED_XOR


def tiny_inputs(device="cpu"):
    """256x256 A and W ~ N(0,1): one generator seeded 0, A drawn first."""
    g = _gen(SEEDS["tiny"], device)
    a = torch.randn(256, 256, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    w = torch.randn(256, 256, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    return a, w


def dense_inputs(shape: DenseShape, which: str, device="cpu", want=("x", "w", "dy")):
    """X [tokens, hidden] with outliers, W [out, hidden], dY [tokens, out]."""
    pre = which  # "super" or "ultra"
    out = {}
    if "x" in want:
        out["x"] = activations_with_outliers(shape.tokens, shape.hidden, SEEDS[pre + "_x"], device)
    if "w" in want:
        out["w"] = normal_bf16((shape.out, shape.hidden), 0.02, SEEDS[pre + "_w"], device)
    if "dy" in want:
        out["dy"] = normal_bf16((shape.tokens, shape.out), 1e-3, SEEDS[pre + "_dy"], device)
    return out


def moe_inputs(shape: MoEShape, which: str, device="cpu", want=("a", "w_up", "w_down")):
    """Expert-sorted activations A [R, latent], offsets [E+1], and per-expert
    weights W_up [E, hidden, latent], W_down [E, latent, hidden]."""
    seed = SEEDS[which + "_moe_x"] if which == "super" else SEEDS["ultra_moe"]
    wseed = SEEDS[which + "_moe_w"]
    routing = zipf_routing(shape.tokens, shape.experts, shape.topk, seed)
    out = {"routing": routing}
    if "a" in want:
        x = normal_bf16((shape.tokens, shape.latent), 1.0, seed + 1000, device)
        out["x_lat"] = x
        out["a"] = x[routing.token_ids.to(x.device)].contiguous()
    if "w_up" in want:
        out["w_up"] = batched_normal_bf16(shape.experts, shape.expert_hidden, shape.latent,
                                          0.02, wseed, device)
    if "w_down" in want:
        out["w_down"] = batched_normal_bf16(shape.experts, shape.latent, shape.expert_hidden,
                                            0.02, wseed + 1, device)
    return out


def max_vio_bound(experts: int, topk: int) -> float:
    """Largest reachable MaxVio, N/k (Ultra report, section 2.7)."""
    return experts / topk


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def describe_routing(r: Routing) -> dict:
    return {
        "assignments": int(r.offsets[-1]),
        "empty_experts": int((r.counts == 0).sum()),
        "max_count": int(r.counts.max()),
        "min_count": int(r.counts.min()),
        "max_vio": round(r.max_vio, 3),
        "max_vio_bound": round(max_vio_bound(r.counts.numel(), r.topk), 3),
    }

