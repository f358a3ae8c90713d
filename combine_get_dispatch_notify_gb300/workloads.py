"""Seeded synthetic workloads for the MoE dispatch/combine path.

This module only *generates inputs*: router top-k maps, router weights and
token activations.  It holds none of the dispatch/combine arithmetic, so the
CUDA path and the CPU oracle can both consume exactly the same tensors.

Workloads (the sizes the dispatch/combine pages discuss, made synthetic):

=============  ==  =====  ====  ===  =  ==  ===============================
name           R   T      H     E    K  C   routing
=============  ==  =====  ====  ===  =  ==  ===============================
tiny           2   128    256   16   2  2   uniform, distinct experts
low_latency    16  128    7168  256  8  8   uniform, distinct experts
prefill        8   4096   7168  256  8  24  uniform, distinct experts
skewed         16  8192   7168  256  8  24  Zipf(1.2) popularity, distinct
large          32  16384  7168  256  8  32  uniform, 10% of slots set to -1
=============  ==  =====  ====  ===  =  ==  ===============================

Recipe (seed 0 everywhere unless stated):

* routing of source rank s uses ``torch.Generator().manual_seed(seed*1000+s)``
  on the CPU, drawn in a fixed order: expert keys, weight logits, mask draws;
* uniform routing takes the K largest of E uniform keys per token (a uniformly
  random K-subset of distinct experts, in random order);
* Zipf routing adds Gumbel noise to ``-s_zipf * log(e+1)`` and takes the K
  largest (sampling K distinct experts without replacement with probability
  proportional to ``(e+1)^-s_zipf``);
* with-replacement routing (``routing="replace"``, edge-case tests only) draws K
  independent uniform expert ids per token, so a token may repeat an expert;
* masking sets each slot to -1 independently with probability ``mask``, after
  the ids and weights are drawn (the weight of a masked slot is left as is);
* weights are ``softmax`` of K standard normals, in fp32;
* activations x are N(0,1) in fp32, rounded to bf16; generated per source rank
  with generator seed ``seed*1000 + 500 + s`` on the requested device.
"""
from __future__ import annotations

import dataclasses

import torch

NODE_SIZE = 8


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    R: int
    T: int
    H: int
    E: int
    K: int
    C: int
    routing: str = "uniform"  # "uniform" | "zipf" | "replace"
    zipf_s: float = 1.2
    mask: float = 0.0
    seed: int = 0
    expert_alignment: int = 1

    @property
    def N(self) -> int:
        return 1 if self.R <= NODE_SIZE else self.R // NODE_SIZE

    @property
    def E_loc(self) -> int:
        return self.E // self.R

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


CONFIGS = {
    "tiny": Workload("tiny", R=2, T=128, H=256, E=16, K=2, C=2),
    "low_latency": Workload("low_latency", R=16, T=128, H=7168, E=256, K=8, C=8),
    "prefill": Workload("prefill", R=8, T=4096, H=7168, E=256, K=8, C=24),
    "skewed": Workload("skewed", R=16, T=8192, H=7168, E=256, K=8, C=24, routing="zipf"),
    "large": Workload("large", R=32, T=16384, H=7168, E=256, K=8, C=32, mask=0.1),
}

DESCRIPTIONS = {
    "tiny": "Tiny: R=2, T=128, H=256, E=16, top-2 uniform distinct, C=2, seed 0",
    "low_latency": "Low-latency shape: R=16 (2 nodes), T=128, H=7168, E=256, top-8 uniform, C=8",
    "prefill": "Prefill uniform: R=8 (1 node), T=4096, H=7168, E=256, top-8 uniform, C=24",
    "skewed": "Skewed routing: R=16 (2 nodes), T=8192, H=7168, E=256, top-8 Zipf(1.2), C=24",
    "large": "Large + masked: R=32 (4 nodes), T=16384, H=7168, E=256, top-8, 10% slots -1, C=32",
}


def _rank_routing(w: Workload, s: int):
    g = torch.Generator().manual_seed(w.seed * 1000 + s)
    T, E, K = w.T, w.E, w.K
    if w.routing == "uniform":
        keys = torch.rand(T, E, generator=g)
        idx = keys.topk(K, dim=1).indices
    elif w.routing == "zipf":
        u = torch.rand(T, E, generator=g).clamp_(min=1e-12, max=1.0 - 1e-7)
        gumbel = -torch.log(-torch.log(u))
        logp = -w.zipf_s * torch.log(torch.arange(1, E + 1, dtype=torch.float32))
        idx = (logp[None, :] + gumbel).topk(K, dim=1).indices
    elif w.routing == "replace":
        idx = torch.randint(0, E, (T, K), generator=g)
    else:
        raise ValueError(f"unknown routing {w.routing!r}")
    logits = torch.randn(T, K, generator=g, dtype=torch.float32)
    weights = torch.softmax(logits, dim=1)
    idx = idx.to(torch.int64)
    if w.mask > 0:
        drop = torch.rand(T, K, generator=g) < w.mask
        idx = torch.where(drop, torch.full_like(idx, -1), idx)
    return idx, weights.to(torch.float32)


def gen_routing(w: Workload):
    """Router output of every source rank: (topk_idx int64 [R,T,K], topk_w fp32 [R,T,K])."""
    if w.T == 0:
        return (torch.zeros(w.R, 0, w.K, dtype=torch.int64),
                torch.zeros(w.R, 0, w.K, dtype=torch.float32))
    parts = [_rank_routing(w, s) for s in range(w.R)]
    topk_idx = torch.stack([p[0] for p in parts]).contiguous()
    topk_w = torch.stack([p[1] for p in parts]).contiguous()
    return topk_idx, topk_w


def gen_x(w: Workload, device="cpu") -> torch.Tensor:
    """Token activations x, bf16 [R,T,H], N(0,1) rounded from fp32."""
    device = torch.device(device)
    x = torch.empty(w.R, w.T, w.H, dtype=torch.bfloat16, device=device)
    for s in range(w.R):
        g = torch.Generator(device=device).manual_seed(w.seed * 1000 + 500 + s)
        x[s].copy_(torch.randn(w.T, w.H, generator=g, device=device, dtype=torch.float32))
    return x


def worst_case_rows(w: Workload) -> int:
    """Upper bound on the receive pool: every token reaches min(K, R) ranks."""
    return w.R * w.T * min(w.K, w.R)


def describe(w: Workload) -> str:
    return DESCRIPTIONS.get(w.name, f"{w.name}: R={w.R}, T={w.T}, H={w.H}, E={w.E}, K={w.K}, C={w.C}")


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def nodes(R: int) -> int:
    return 1 if R <= NODE_SIZE else R // NODE_SIZE


__all__ = ["Workload", "CONFIGS", "gen_routing", "gen_x", "worst_case_rows", "describe",
           "ceil_div", "nodes"]
