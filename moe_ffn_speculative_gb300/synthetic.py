"""Seeded synthetic inputs for the MoE-FFN layer.

This module only draws random tensors of the right shapes, value distributions
and dtypes; it contains none of the layer's arithmetic.  It is the one module
that both the CUDA library's callers (tests, bench) and the CPU oracle's
callers share.

Workloads (all synthetic; the pages' serving runs use real prompts and trained
drafters, which these shapes and distributions stand in for):

* ``tiny``: T=16, H=64, E=8, I=32, top-2, softmax, renormalised.
* ``qwen3_8b_dspark``: Qwen3-8B DSpark draft layer, T=72 (8 requests x verify
  block 9), H=4096, E=8, I=1536, top-1, softmax, renormalised.
* ``qwen38_27b_dspark``: Qwen3.8-27B-style drafter layer, T=72, H=5120, E=512,
  I=512, top-10, softmax with a folded router bias, one sigmoid-gated shared
  expert of I=2048.
* ``dsv3_style``: T=72, H=7168, E=256, I=2048, top-8, sigmoid, selection-only
  expert bias, group-limited 8/4, routed scale 2.5, one ungated shared expert
  of I=2048.
* ``dsv4_style``: H=4096, E=256, I=1024, top-6, sqrt(softplus), selection-only
  expert bias, route scale 1.5, SwiGLU clamp 7, one ungated shared expert of
  I=1024, T in {9, 72, 576, 4096}.

x ~ N(0, 1); every weight ~ N(0, 0.02); all bf16.  Router bias ~ N(0, 0.1) and
expert bias ~ N(0, 0.05) in fp32.  Tensors are drawn in the fixed order x,
gate, router_bias, expert_bias, w_gate_up, w_down, sh_gate_up, sh_down,
sh_gate from one torch.Generator seeded with the workload's seed.  Layers
with FP4 routed experts draw uniform code bytes and e8m0 scale bytes uniform
on three values around the one that gives the weights an RMS near w_std,
in place of the bf16 expert weights.  FP8 weights (routed experts, or the
shared expert) are N(0, 1) draws cast to e4m3 codes, with one e8m0 scale per
32 x 32 block uniform on three values around 2^round(log2(w_std)).
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass
from typing import Dict, Optional

import torch

# score-function codes of the C header
SOFTMAX, SIGMOID, SQRTSOFTPLUS = 0, 1, 2


@dataclass(frozen=True)
class LayerConfig:
    name: str
    T: int
    H: int
    E: int
    I: int
    K: int
    score_fn: int = SOFTMAX
    n_group: int = 1
    topk_group: int = 1
    group_topn: int = 2
    norm_topk_prob: bool = True
    norm_eps: float = 1e-20
    route_scale: float = 1.0
    swiglu_limit: float = 0.0
    router_bias_std: float = 0.0
    expert_bias_std: float = 0.0
    shared_I: int = 0
    shared_gated: bool = False
    seed: int = 0
    x_std: float = 1.0
    w_std: float = 0.02
    # routed experts: "bf16", "fp4" (e2m1 codes + e8m0 scale per 32 inputs) or
    # "fp8" (e4m3 codes + e8m0 scale per 32 x 32 block)
    expert_format: str = "bf16"
    # shared expert: "bf16" or "fp8"
    shared_format: str = "bf16"

    def with_(self, **kw) -> "LayerConfig":
        return dataclasses.replace(self, **kw)

    @property
    def weight_bytes(self) -> int:
        """Bytes of all routed experts' weights (codes and scales)."""
        n = 3 * self.E * self.H * self.I
        if self.expert_format == "fp4":
            return n // 2 + n // 32
        if self.expert_format == "fp8":
            return n + n // 1024
        return n * 2


CONFIGS: Dict[str, LayerConfig] = {
    "tiny": LayerConfig("tiny", T=16, H=64, E=8, I=32, K=2, seed=0),
    "qwen3_8b_dspark": LayerConfig("qwen3_8b_dspark", T=72, H=4096, E=8, I=1536, K=1, seed=1),
    "qwen38_27b_dspark": LayerConfig("qwen38_27b_dspark", T=72, H=5120, E=512, I=512, K=10,
                                     router_bias_std=0.1, shared_I=2048, shared_gated=True,
                                     seed=2),
    "dsv3_style": LayerConfig("dsv3_style", T=72, H=7168, E=256, I=2048, K=8, score_fn=SIGMOID,
                              expert_bias_std=0.05, n_group=8, topk_group=4, route_scale=2.5,
                              shared_I=2048, seed=3),
    "dsv4_style": LayerConfig("dsv4_style", T=72, H=4096, E=256, I=1024, K=6,
                              score_fn=SQRTSOFTPLUS, expert_bias_std=0.05, route_scale=1.5,
                              swiglu_limit=7.0, shared_I=1024, seed=4),
}

# Further MoE-FFN shapes the pages name, for parity and measurement (the
# pages give the expert shape and recipe; hidden sizes and shared-expert
# widths they leave open are the plainest readings, see the design notes):
# * DeepSeek-V4-Flash drafter: 64 experts x 2048, top-6, ungated shared expert,
#   sqrt(softplus), selection bias, scale 1.5, SwiGLU clamp 10;
# * DeepSeek-V4.1's own DSpark draft: 128 experts x 2304, top-3, one shared
#   expert, sqrt(softplus) x 1.5, clamped SwiGLU, expert bias;
# * a dense draft layer (no expert fields: E = 1, top-1) of Qwen3-8B's MLP
#   width, through the same engine.
VARIANTS: Dict[str, LayerConfig] = {
    "dsv4_flash_drafter": LayerConfig("dsv4_flash_drafter", T=72, H=4096, E=64, I=2048, K=6,
                                      score_fn=SQRTSOFTPLUS, expert_bias_std=0.05, route_scale=1.5,
                                      swiglu_limit=10.0, shared_I=2048, seed=21),
    "dsv41_dspark_draft": LayerConfig("dsv41_dspark_draft", T=72, H=4096, E=128, I=2304, K=3,
                                      score_fn=SQRTSOFTPLUS, expert_bias_std=0.05, route_scale=1.5,
                                      swiglu_limit=10.0, shared_I=2304, seed=22),
    "dense_draft": LayerConfig("dense_draft", T=72, H=4096, E=1, I=12288, K=1, seed=23),
}
CONFIGS.update(VARIANTS)
DSV4_TOKEN_SWEEP = (9, 72, 576, 4096)


def _normal(gen: torch.Generator, shape, std: float, dtype, device) -> torch.Tensor:
    return (torch.randn(shape, generator=gen, device=device, dtype=torch.float32) * std).to(dtype)


def _normal_rows(gen, n_outer: int, inner_shape, std: float, device) -> torch.Tensor:
    """A [n_outer, *inner] bf16 tensor drawn one outer slice at a time, so the
    fp32 staging never exceeds one slice."""
    out = torch.empty((n_outer, *inner_shape), dtype=torch.bfloat16, device=device)
    for i in range(n_outer):
        out[i] = _normal(gen, inner_shape, std, torch.bfloat16, device)
    return out


def _bytes(gen, shape, lo: int, hi: int, device) -> torch.Tensor:
    """uint8 tensor uniform on [lo, hi)."""
    return torch.randint(lo, hi, shape, generator=gen, device=device, dtype=torch.uint8)


def _fp4_scale_center(w_std: float) -> int:
    """e8m0 byte around which FP4 block scales are drawn so that weights of
    uniformly drawn codes have about the RMS w_std (the sixteen e2m1 values
    have an RMS of about 2.93)."""
    return 127 + int(round(math.log2(w_std / 2.93)))


def _fp8_codes(gen, shape, device) -> torch.Tensor:
    """uint8 e4m3 codes of N(0, 1) draws (rounded by torch's e4m3 cast)."""
    v = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    return v.to(torch.float8_e4m3fn).view(torch.uint8)


def _fp8_weight(gen, n: int, k: int, w_std: float, device, outer: int = 0):
    """(codes [outer,] n x k, e8m0 scales [outer,] ceil(n/32) x ceil(k/32)):
    block scales uniform on three values around 2^round(log2(w_std))."""
    c = 127 + int(round(math.log2(w_std)))
    lead = (outer,) if outer else ()
    if outer:
        codes = torch.empty((outer, n, k), dtype=torch.uint8, device=device)
        for i in range(outer):
            codes[i] = _fp8_codes(gen, (n, k), device)
    else:
        codes = _fp8_codes(gen, (n, k), device)
    scales = _bytes(gen, lead + (-(-n // 32), -(-k // 32)), c - 1, c + 2, device)
    return codes, scales


def make_inputs(cfg: LayerConfig, device="cpu", seed: Optional[int] = None) -> Dict[str, torch.Tensor]:
    """Draw one layer's inputs and weights.  Keys: x, gate, router_bias,
    expert_bias, w_gate_up [E,2I,H], w_down [E,H,I], sh_gate_up [2Is,H],
    sh_down [H,Is], sh_gate [H] (absent entries are None).  With FP4 routed
    experts, w_gate_up / w_down are None and w_gate_up_q [E,2I,H/2],
    w_gate_up_s [E,2I,H/32], w_down_q [E,H,I/2], w_down_s [E,H,I/32] (uint8
    codes and e8m0 scales) take their place in the draw order."""
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(cfg.seed if seed is None else seed)
    bf = torch.bfloat16
    d: Dict[str, Optional[torch.Tensor]] = {}
    d["x"] = _normal(gen, (cfg.T, cfg.H), cfg.x_std, bf, device)
    d["gate"] = _normal(gen, (cfg.E, cfg.H), cfg.w_std, bf, device)
    d["router_bias"] = (_normal(gen, (cfg.E,), cfg.router_bias_std, torch.float32, device)
                        if cfg.router_bias_std > 0 else None)
    d["expert_bias"] = (_normal(gen, (cfg.E,), cfg.expert_bias_std, torch.float32, device)
                        if cfg.expert_bias_std > 0 else None)
    if cfg.expert_format == "fp4":
        c = _fp4_scale_center(cfg.w_std)
        d["w_gate_up_q"] = _bytes(gen, (cfg.E, 2 * cfg.I, cfg.H // 2), 0, 256, device)
        d["w_gate_up_s"] = _bytes(gen, (cfg.E, 2 * cfg.I, cfg.H // 32), c - 1, c + 2, device)
        d["w_down_q"] = _bytes(gen, (cfg.E, cfg.H, cfg.I // 2), 0, 256, device)
        d["w_down_s"] = _bytes(gen, (cfg.E, cfg.H, cfg.I // 32), c - 1, c + 2, device)
        d["w_gate_up"] = d["w_down"] = None
    elif cfg.expert_format == "fp8":
        d["w_gate_up_q"], d["w_gate_up_s"] = _fp8_weight(gen, 2 * cfg.I, cfg.H, cfg.w_std, device, cfg.E)
        d["w_down_q"], d["w_down_s"] = _fp8_weight(gen, cfg.H, cfg.I, cfg.w_std, device, cfg.E)
        d["w_gate_up"] = d["w_down"] = None
    else:
        d["w_gate_up"] = _normal_rows(gen, cfg.E, (2 * cfg.I, cfg.H), cfg.w_std, device)
        d["w_down"] = _normal_rows(gen, cfg.E, (cfg.H, cfg.I), cfg.w_std, device)
    if cfg.shared_I > 0:
        if cfg.shared_format == "fp8":
            d["sh_gate_up_q"], d["sh_gate_up_s"] = _fp8_weight(gen, 2 * cfg.shared_I, cfg.H, cfg.w_std, device)
            d["sh_down_q"], d["sh_down_s"] = _fp8_weight(gen, cfg.H, cfg.shared_I, cfg.w_std, device)
            d["sh_gate_up"] = d["sh_down"] = None
        else:
            d["sh_gate_up"] = _normal(gen, (2 * cfg.shared_I, cfg.H), cfg.w_std, bf, device)
            d["sh_down"] = _normal(gen, (cfg.H, cfg.shared_I), cfg.w_std, bf, device)
        d["sh_gate"] = (_normal(gen, (cfg.H,), cfg.w_std, bf, device)
                        if cfg.shared_gated else None)
    else:
        d["sh_gate_up"] = d["sh_down"] = d["sh_gate"] = None
    return d


def make_router_inputs(cfg: LayerConfig, device="cpu", seed: Optional[int] = None) -> Dict[str, torch.Tensor]:
    """Only x, gate, router_bias and expert_bias, drawn as make_inputs draws
    them first (the same values), without the experts' weights."""
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(cfg.seed if seed is None else seed)
    d: Dict[str, Optional[torch.Tensor]] = {}
    d["x"] = _normal(gen, (cfg.T, cfg.H), cfg.x_std, torch.bfloat16, device)
    d["gate"] = _normal(gen, (cfg.E, cfg.H), cfg.w_std, torch.bfloat16, device)
    d["router_bias"] = (_normal(gen, (cfg.E,), cfg.router_bias_std, torch.float32, device)
                        if cfg.router_bias_std > 0 else None)
    d["expert_bias"] = (_normal(gen, (cfg.E,), cfg.expert_bias_std, torch.float32, device)
                        if cfg.expert_bias_std > 0 else None)
    return d


def make_x(cfg: LayerConfig, T: int, device="cpu", seed: int = 0) -> torch.Tensor:
    """Only the activations, for sweeps over the token count."""
    gen = torch.Generator(device=torch.device(device))
    gen.manual_seed(seed)
    return _normal(gen, (T, cfg.H), cfg.x_std, torch.bfloat16, torch.device(device))


def make_logits(T: int, E: int, std: float = 1.0, device="cpu", seed: int = 0,
                tie_every: int = 0) -> torch.Tensor:
    """fp32 router logits fed identically to both sides of a routing test.
    With ``tie_every`` > 0, every such column copies its left neighbour so
    exact ties occur."""
    gen = torch.Generator(device=torch.device(device))
    gen.manual_seed(seed)
    l = torch.randn((T, E), generator=gen, device=device, dtype=torch.float32) * std
    if tie_every > 0:
        for j in range(tie_every, E, tie_every):
            l[:, j] = l[:, j - 1]
    return l
