"""Seeded synthetic inputs for the DeepSeekMoE layer forward.

This module is shared by the CPU oracle's tests, the CUDA library's tests, the smoke check and
the benchmark. It holds workload shapes and random-number recipes only: none of the layer's
arithmetic (routing, expert FFNs, combine, balance statistics) lives here.

Shapes follow the model sizes the DeepSeekMoE pages describe (2B: hidden 1280, 1 shared + 63
routed experts, top-7; 16B: hidden 2048, 2 shared + 64 routed, top-6; 145B: hidden 4096), see
"DeepSeekMoE 论文解读" (xxmr.cn), sections 两大核心策略 and 三阶段实验规模. The pages train on
public text corpora that are not available here; seeded Gaussian tensors of the same shapes stand
in for trained weights and activations.

Every tensor is drawn on the CPU from its own ``torch.Generator`` (seed = config seed * 100 +
tensor id), in fp32, divided by the stated standard deviation and then rounded once to the
config's storage dtype. The same bytes therefore reach the GPU and the oracle, and changing the
token count T changes only ``u``.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class MoEShape:
    """One layer configuration.

    Expert numbering: experts ``0..n_shared-1`` are the always-active shared experts; routed
    expert ``j`` (local id ``0..n_routed-1``) has global id ``n_shared + j``.
    """

    name: str
    T: int              # tokens in one call
    d: int              # model width
    n_shared: int       # K_s
    n_routed: int       # N' (routed experts)
    inter: int          # expert intermediate width I (already divided by m)
    top_k: int          # K' (routed experts per token)
    n_groups: int       # D, contiguous routed-expert groups for the device-level statistic
    dtype: str          # "f32" or "bf16": storage and compute-input type
    seed: int
    alpha1: float = 0.01
    alpha2: float = 0.05
    renormalize: int = 0
    zipf_s: Optional[float] = None   # logit bias -zipf_s*ln(rank) per routed expert
    skip_top: int = 0                # ablation: disable each token's skip_top best routed experts
    drop_shared: int = 0             # ablation: disable the shared experts
    description: str = ""

    @property
    def n_experts(self) -> int:
        return self.n_shared + self.n_routed

    def with_(self, **kw) -> "MoEShape":
        return dataclasses.replace(self, **kw)

    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


CONFIGS = {
    "tiny_f32": MoEShape(
        "tiny_f32", T=256, d=128, n_shared=1, n_routed=15, inter=64, top_k=3, n_groups=4,
        dtype="f32", seed=0,
        description="tiny fp32 layer: 4 base experts split m=4 into 16, 1 shared + 15 routed, "
                    "I=64, top-3"),
    "2b_bf16": MoEShape(
        "2b_bf16", T=8192, d=1280, n_shared=1, n_routed=63, inter=320, top_k=7, n_groups=8,
        dtype="bf16", seed=1, description="2B-like layer, 2x4096 tokens"),
    "16b_bf16": MoEShape(
        "16b_bf16", T=16384, d=2048, n_shared=2, n_routed=64, inter=1408, top_k=6, n_groups=8,
        dtype="bf16", seed=2, description="16B-like layer, 4x4096 tokens"),
    "16b_decode_bf16": MoEShape(
        "16b_decode_bf16", T=64, d=2048, n_shared=2, n_routed=64, inter=1408, top_k=6,
        n_groups=8, dtype="bf16", seed=3,
        description="16B-like decode step: batch 64 x 1 token (weight-bandwidth bound)"),
    # the pages' analysis variants (section 专家特化深度分析 and the coarse baseline of Fig. 2(a))
    "2b_half_activated_bf16": MoEShape(
        "2b_half_activated_bf16", T=8192, d=1280, n_shared=1, n_routed=63, inter=320, top_k=3,
        n_groups=8, dtype="bf16", seed=5,
        description="2B-like layer with half the activated experts: 1 shared + top-3 routed"),
    "2b_gshard_top2_bf16": MoEShape(
        "2b_gshard_top2_bf16", T=8192, d=1280, n_shared=0, n_routed=16, inter=1280, top_k=2,
        n_groups=8, dtype="bf16", seed=6,
        description="coarse top-2 baseline (m = 1, no shared expert): 16 experts of width 4*320"),
    "145b_zipf_bf16": MoEShape(
        "145b_zipf_bf16", T=8192, d=4096, n_shared=4, n_routed=128, inter=1536, top_k=12,
        n_groups=8, dtype="bf16", seed=4, zipf_s=1.1,
        description="145B-like layer with Zipf(1.1)-skewed routing bias"),
}

# tensor ids used to derive per-tensor generator seeds
_TID = {"u": 1, "centroids": 2, "w_gate": 3, "w_up": 4, "w_down": 5, "zipf_perm": 6}


def _gen(shape: MoEShape, tensor: str, seed: Optional[int] = None) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed((shape.seed if seed is None else seed) * 100 + _TID[tensor])
    return g


def _gaussian(rows: int, cols: int, std: float, gen: torch.Generator, dtype: torch.dtype,
              out: Optional[torch.Tensor] = None, chunk_rows: int = 4096) -> torch.Tensor:
    """N(0, std^2) in fp32, rounded once to ``dtype``; drawn in row chunks to bound memory."""
    if out is None:
        out = torch.empty(rows, cols, dtype=dtype)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        x = torch.randn(r1 - r0, cols, generator=gen, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        out[r0:r1].copy_(x.to(dtype))
    return out


def make_tokens(shape: MoEShape, T: Optional[int] = None, seed: Optional[int] = None) -> torch.Tensor:
    """u [T, d]: token activations, u ~ N(0, 1)."""
    T = shape.T if T is None else T
    return _gaussian(T, shape.d, 1.0, _gen(shape, "u", seed), shape.torch_dtype())


def make_centroids(shape: MoEShape) -> torch.Tensor:
    """e [N', d]: routed-expert centroids, e ~ N(0, 1/d)."""
    return _gaussian(shape.n_routed, shape.d, 1.0 / math.sqrt(shape.d),
                     _gen(shape, "centroids"), shape.torch_dtype())


def make_logit_bias(shape: MoEShape) -> Optional[torch.Tensor]:
    """b [N'] fp32, or None. For a Zipf-skewed workload: a seeded random ranking of the routed
    experts, b_j = -s * ln(rank_j), so the prior routing weight of rank r is r^-s."""
    if shape.zipf_s is None:
        return None
    perm = torch.randperm(shape.n_routed, generator=_gen(shape, "zipf_perm"))
    rank = (perm + 1).to(torch.float64)
    return (-shape.zipf_s * torch.log(rank)).to(torch.float32)


def make_expert_weights(shape: MoEShape):
    """(w_gate [E, I, d], w_up [E, I, d], w_down [E, d, I]); shared experts first.

    W_gate, W_up ~ N(0, 1/d); W_down ~ N(0, 1/I).
    """
    E, I, d, dt = shape.n_experts, shape.inter, shape.d, shape.torch_dtype()
    w_gate = torch.empty(E, I, d, dtype=dt)
    w_up = torch.empty(E, I, d, dtype=dt)
    w_down = torch.empty(E, d, I, dtype=dt)
    for w, name, std, rows, cols in ((w_gate, "w_gate", 1 / math.sqrt(d), E * I, d),
                                     (w_up, "w_up", 1 / math.sqrt(d), E * I, d),
                                     (w_down, "w_down", 1 / math.sqrt(I), E * d, I)):
        _gaussian(rows, cols, std, _gen(shape, name), dt, out=w.view(rows, cols))
    return w_gate, w_up, w_down


def make_inputs(shape: MoEShape, T: Optional[int] = None, seed: Optional[int] = None) -> dict:
    """All layer inputs on the CPU, in the config's storage dtype (bias in fp32)."""
    w_gate, w_up, w_down = make_expert_weights(shape)
    return {
        "u": make_tokens(shape, T, seed),
        "centroids": make_centroids(shape),
        "bias": make_logit_bias(shape),
        "w_gate": w_gate,
        "w_up": w_up,
        "w_down": w_down,
    }
