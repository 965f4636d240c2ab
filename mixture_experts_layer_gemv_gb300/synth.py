"""Seeded synthetic inputs for the MoE layer: layer shapes, tokens and weights.

This module is the one piece that both the CUDA path (tests, benchmark) and the
CPU oracle consume. It draws random numbers and packs them into the layouts the
library takes; it holds none of the layer's arithmetic (no routing, no FFN, no
activation quantisation).

Shapes follow the DeepSeek-V2 MoE layer of "DSV2-236B-MegaKernel" (README,
"Model geometry" and the MoE subgraph of the stage flowchart: hidden 5120,
moe_intermediate_size 1536, 160 routed experts in 8 groups, top-3 groups, top-6
experts, routed_scaling_factor 16.0, 2 shared experts) plus a tiny layer, a
prefill-sized layer (hidden 7168, 64 experts) and a load-imbalanced variant.
The checkpoint those pages load is not used: weights are drawn N(0, 0.02) and
quantised to FP8 E4M3 with one fp32 scale per 128x128 block (the "per-128
block-scaled FP8" of the README's "Results"), the router is fp32 N(0, 0.02) and
activations are bf16 N(0, 1).

The weight quantiser here is data preparation: scale = amax / 448 per block, the
codes come from torch's float8_e4m3fn conversion (round to nearest even) of the
clamped quotient. Both sides receive the same codes and scales.

Random streams: one torch.Generator per (seed, tensor name), on the device the
tensor is made on. A CPU-made and a GPU-made tensor of the same name therefore
differ; every parity check hands the very same tensors to both sides.
"""
from __future__ import annotations

import hashlib

from dataclasses import dataclass
from typing import Dict, Optional

import torch

__all__ = [
    "MoEConfig",
    "Workload",
    "WORKLOADS",
    "make_weights",
    "make_weights_mx",
    "make_router",
    "make_tokens",
    "replicate_weights",
    "ZIPF_S",
    "ZIPF_BETA",
]


@dataclass(frozen=True)
class MoEConfig:
    """The layer's arguments, named as on the pages (DeepSeek-V2 config names)."""

    hidden: int
    moe_inter: int
    n_routed: int
    n_group: int
    topk_group: int
    top_k: int
    routed_scaling_factor: float
    n_shared: int

    @property
    def shared_inter(self) -> int:
        """Width of the fused shared MLP: n_shared experts of moe_inter each."""
        return self.n_shared * self.moe_inter


@dataclass(frozen=True)
class Workload:
    name: str
    cfg: MoEConfig
    T: int
    seed: int
    zipf_bias: bool = False
    description: str = ""


DSV2 = MoEConfig(hidden=5120, moe_inter=1536, n_routed=160, n_group=8, topk_group=3, top_k=6,
                 routed_scaling_factor=16.0, n_shared=2)

WORKLOADS: Dict[str, Workload] = {
    w.name: w
    for w in [
        Workload("tiny_t8", MoEConfig(512, 256, 16, 4, 2, 4, 1.0, 1), T=8, seed=0,
                 description="tiny MoE layer, T=8"),
        Workload("dsv2_decode_t1", DSV2, T=1, seed=1,
                 description="DeepSeek-V2 MoE layer, decode T=1"),
        Workload("dsv2_decode_t64", DSV2, T=64, seed=2,
                 description="DeepSeek-V2 MoE layer, T=64 decode tokens"),
        Workload("prefill_t4096", MoEConfig(7168, 2048, 64, 8, 4, 8, 2.5, 1), T=4096, seed=3,
                 description="prefill / training-forward MoE layer, T=4096"),
        Workload("dsv2_zipf_t2048", DSV2, T=2048, seed=4, zipf_bias=True,
                 description="DeepSeek-V2 MoE layer, T=2048, Zipf(1.1) expert popularity"),
    ]
}

# Load-imbalance workload: expert e gets logit bias -ZIPF_BETA * ZIPF_S * ln(rank_e),
# rank_e a seeded permutation of 1..E. ZIPF_BETA was fitted (oracle/fit_zipf_beta.py,
# with the oracle's routing) so that the 16 most popular experts take ~60% of the
# assignments on the DeepSeek-V2 shape.
ZIPF_S = 1.1
ZIPF_BETA = 0.8233


def _generator(seed: int, name: str, device) -> torch.Generator:
    h = hashlib.sha256(f"{seed}:{name}".encode()).digest()
    g = torch.Generator(device=device)
    g.manual_seed(int.from_bytes(h[:8], "little") & ((1 << 63) - 1))
    return g


def _randn(shape, seed, name, device, std=1.0, dtype=torch.float32):
    g = _generator(seed, name, device)
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def _quantise_blocks(w: torch.Tensor):
    """w fp32 [..., R, C] -> (E4M3 codes uint8 [..., R, C], fp32 scales [..., R/128, C/128])."""
    *lead, R, C = w.shape
    blk = w.reshape(*lead, R // 128, 128, C // 128, 128)
    amax = blk.abs().amax(dim=(-3, -1))
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    q = (blk / scale[..., :, None, :, None]).clamp_(-448.0, 448.0)
    codes = q.reshape(*lead, R, C).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes.contiguous(), scale.to(torch.float32).contiguous()


def _quantise_mx(w: torch.Tensor):
    """w fp32 [..., R, C] -> (E4M3 codes uint8 [..., R, C], E8M0 scale bytes uint8 [..., R, C/32]).

    MXFP8 data preparation: per row and 32 consecutive columns, the scale is the smallest
    power of two 2^k with amax <= 448 * 2^k (k >= -126; amax = 0 gives 2^0), stored as the
    byte k + 127; codes are torch's float8_e4m3fn conversion (round to nearest even) of
    the clamped quotient. Both sides receive the same codes and scale bytes."""
    *lead, R, C = w.shape
    blk = w.reshape(*lead, R, C // 32, 32)
    amax = blk.abs().amax(dim=-1)
    m, e = torch.frexp(amax)  # amax = m * 2^e, m in [0.5, 1); 448 = 0.875 * 2^9
    k = torch.where(m <= 0.875, e - 9, e - 8)
    k = torch.where(amax > 0, k, torch.zeros_like(k)).clamp(min=-126)
    scale = torch.ldexp(torch.ones_like(amax), k)
    q = (blk / scale[..., None]).clamp_(-448.0, 448.0)
    codes = q.reshape(*lead, R, C).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes.contiguous(), (k + 127).to(torch.uint8).contiguous()


def _expert_stack(E, R, C, seed, name, device, std=0.02, mx=False):
    codes = torch.empty((E, R, C), dtype=torch.uint8, device=device)
    if mx:
        scales = torch.empty((E, R, C // 32), dtype=torch.uint8, device=device)
    else:
        scales = torch.empty((E, R // 128, C // 128), dtype=torch.float32, device=device)
    quant = _quantise_mx if mx else _quantise_blocks
    for e in range(E):  # one expert at a time keeps the fp32 temporaries small
        c, s = quant(_randn((R, C), seed, f"{name}[{e}]", device, std))
        codes[e].copy_(c)
        scales[e].copy_(s)
    return codes, scales


def zipf_bias(cfg: MoEConfig, seed: int, device="cpu", beta: float = None) -> torch.Tensor:
    """Per-expert router bias -beta * s * ln(rank_e), ranks a seeded permutation of 1..E."""
    beta = ZIPF_BETA if beta is None else beta
    g = _generator(seed, "zipf_rank", "cpu")
    rank = torch.randperm(cfg.n_routed, generator=g).to(torch.float64) + 1.0
    return (-beta * ZIPF_S * torch.log(rank)).to(torch.float32).to(device)


def make_router(cfg: MoEConfig, seed: int, device="cpu", zipf: bool = False,
                zipf_beta: Optional[float] = None):
    """(w_router fp32 [E, H], router_bias fp32 [E] or None) of one layer."""
    wr = _randn((cfg.n_routed, cfg.hidden), seed, "w_router", device, 0.02)
    return wr, (zipf_bias(cfg, seed, device, zipf_beta) if zipf else None)


def make_weights(cfg: MoEConfig, seed: int, device="cpu", zipf: bool = False,
                 zipf_beta: Optional[float] = None) -> Dict[str, Optional[torch.Tensor]]:
    """All weights of one layer, in the library's layouts.

    w_gate, w_up  uint8 (E4M3 codes) [E, I, H]   s_gate, s_up  fp32 [E, I/128, H/128]
    w_down        uint8 [E, H, I]                s_down        fp32 [E, H/128, I/128]
    ws_gate/ws_up uint8 [Is, H], ws_down [H, Is] with fp32 block scales (None if n_shared=0)
    w_router      fp32 [E, H]                    router_bias   fp32 [E] or None
    """
    H, I, E, Is = cfg.hidden, cfg.moe_inter, cfg.n_routed, cfg.shared_inter
    out: Dict[str, Optional[torch.Tensor]] = {}
    out["w_router"], out["router_bias"] = make_router(cfg, seed, device, zipf, zipf_beta)
    out["w_gate"], out["s_gate"] = _expert_stack(E, I, H, seed, "w_gate", device)
    out["w_up"], out["s_up"] = _expert_stack(E, I, H, seed, "w_up", device)
    out["w_down"], out["s_down"] = _expert_stack(E, H, I, seed, "w_down", device)
    if cfg.n_shared > 0:
        for nm, (R, C) in (("gate", (Is, H)), ("up", (Is, H)), ("down", (H, Is))):
            c, s = _quantise_blocks(_randn((R, C), seed, f"ws_{nm}", device, 0.02))
            out[f"ws_{nm}"], out[f"ss_{nm}"] = c, s
    else:
        for nm in ("gate", "up", "down"):
            out[f"ws_{nm}"] = out[f"ss_{nm}"] = None
    return out


def make_weights_mx(cfg: MoEConfig, seed: int, device="cpu", zipf: bool = False,
                    zipf_beta: Optional[float] = None) -> Dict[str, Optional[torch.Tensor]]:
    """The layer of make_weights (the same fp32 draws) quantised to MXFP8 instead.

    w_gate, w_up  uint8 (E4M3 codes) [E, I, H]   s_gate, s_up  uint8 (E8M0) [E, I, H/32]
    w_down        uint8 [E, H, I]                s_down        uint8 (E8M0) [E, H, I/32]
    ws_gate/ws_up uint8 [Is, H], ws_down [H, Is] with E8M0 scales [Is, H/32], [H, Is/32]
    w_router      fp32 [E, H]                    router_bias   fp32 [E] or None
    """
    H, I, E, Is = cfg.hidden, cfg.moe_inter, cfg.n_routed, cfg.shared_inter
    out: Dict[str, Optional[torch.Tensor]] = {}
    out["w_router"], out["router_bias"] = make_router(cfg, seed, device, zipf, zipf_beta)
    out["w_gate"], out["s_gate"] = _expert_stack(E, I, H, seed, "w_gate", device, mx=True)
    out["w_up"], out["s_up"] = _expert_stack(E, I, H, seed, "w_up", device, mx=True)
    out["w_down"], out["s_down"] = _expert_stack(E, H, I, seed, "w_down", device, mx=True)
    if cfg.n_shared > 0:
        for nm, (R, C) in (("gate", (Is, H)), ("up", (Is, H)), ("down", (H, Is))):
            c, s = _quantise_mx(_randn((R, C), seed, f"ws_{nm}", device, 0.02))
            out[f"ws_{nm}"], out[f"ss_{nm}"] = c, s
    else:
        for nm in ("gate", "up", "down"):
            out[f"ws_{nm}"] = out[f"ss_{nm}"] = None
    return out


def replicate_weights(weights: Dict[str, Optional[torch.Tensor]]):
    """A copy at fresh addresses (same values): stacked layer replicas for timing."""
    return {k: (None if v is None else v.clone()) for k, v in weights.items()}


def make_tokens(cfg: MoEConfig, T: int, seed: int, device="cpu", name: str = "x") -> torch.Tensor:
    """bf16 [T, H] activations, N(0, 1) rounded to bf16."""
    return _randn((T, cfg.hidden), seed, name, device, 1.0, torch.bfloat16)


def make_workload(name: str, device="cpu", T: Optional[int] = None):
    """(cfg, x, weights) of a named workload."""
    w = WORKLOADS[name]
    T = w.T if T is None else T
    weights = make_weights(w.cfg, w.seed, device, zipf=w.zipf_bias)
    x = make_tokens(w.cfg, T, w.seed, device)
    return w.cfg, x, weights
