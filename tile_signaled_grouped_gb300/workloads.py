"""Seeded synthetic workloads for the MoE expert-combine path.

This module holds the five workload shapes and the seeded generators that
draw their inputs. It contains none of the method's arithmetic (no softmax,
no top-k, no layout, no FFN): it only draws random numbers and, for the two
workloads whose routing is prescribed rather than gated (balanced and
Zipf-skewed), writes the prescribed expert ids. Both the CUDA path and the
CPU oracle consume what it returns; neither is imported here.

Shapes follow the MoE layer of the TileMoE notes (zhongzhuzhou.org,
"Fine-grained Computation-Communication Overlap via Tile-level Signaling and
Scheduling for Mixture-of-Experts", section 2.1-2.2): W expert-parallel
ranks, L experts per rank (E = W*L), top-k routing, T tokens per rank,
d_model = D, expert d_ff = F, band height tb_M.
"""
from __future__ import annotations

import dataclasses

import torch

__all__ = ["Workload", "WORKLOADS", "get_workload", "Inputs", "make_inputs", "router_weights"]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    W: int            # logical expert-parallel ranks
    L: int            # experts per rank
    topk: int
    T: int            # tokens per rank
    d_model: int
    d_ff: int
    tb_M: int         # row-band height (the tile M of the layout)
    routing: str      # "gate" (softmax top-k of N(0,1) logits), "balanced", "zipf"
    x_std: float = 1.0
    w_std: float = 0.02
    zipf_s: float = 1.2
    mgb: int = 1      # bands merged per middle segment
    seed: int = 0

    @property
    def E(self) -> int:
        return self.W * self.L


# The five shapes.  x ~ N(0, x_std), weights ~ N(0, w_std), gate logits ~ N(0, 1).
WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny", W=4, L=2, topk=2, T=64, d_model=128, d_ff=256, tb_M=64,
                 routing="gate"),
        Workload("a100_like", W=4, L=2, topk=2, T=4096, d_model=2048, d_ff=8192, tb_M=128,
                 routing="balanced"),
        Workload("qwen3_235b_like", W=8, L=16, topk=8, T=512, d_model=4096, d_ff=1536,
                 tb_M=128, routing="gate"),
        Workload("deepseek_v3_like", W=8, L=32, topk=8, T=256, d_model=7168, d_ff=2048,
                 tb_M=64, routing="gate"),
        Workload("stress_skew", W=4, L=4, topk=1, T=2048, d_model=5120, d_ff=8192, tb_M=256,
                 routing="zipf"),
    ]
}


def get_workload(name: str, **overrides) -> Workload:
    return dataclasses.replace(WORKLOADS[name], **overrides)


@dataclasses.dataclass
class Inputs:
    """Per-rank tensors; every list has W entries (one allocation per logical rank)."""
    wl: Workload
    x: list          # [T, D] bf16
    w_gate: list     # [L, F, D] bf16 (nn.Linear layout: out x in)
    w_up: list       # [L, F, D] bf16
    w_down: list     # [L, D, F] bf16
    logits: torch.Tensor            # [W, T, E] fp32 gate logits
    forced_ids: torch.Tensor | None  # [W, T, k] int32 prescribed routing, or None (gate decides)


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal_bf16(shape, std, device, seed):
    t = torch.empty(shape, dtype=torch.float32, device=device)
    t.normal_(0.0, std, generator=_gen(device, seed))
    return t.to(torch.bfloat16)


def balanced_ids(W: int, T: int, k: int, E: int, device="cpu") -> torch.Tensor:
    """Round-robin routing: slot j of token t on rank s goes to ((s*T + t)*k + j) mod E.

    With k <= E the k ids of one token are distinct, and every expert receives
    the same number of slots from every rank when T*k is a multiple of E.
    """
    s = torch.arange(W, device=device).view(W, 1, 1)
    t = torch.arange(T, device=device).view(1, T, 1)
    j = torch.arange(k, device=device).view(1, 1, k)
    return (((s * T + t) * k + j) % E).to(torch.int32)


def zipf_ids(W: int, T: int, k: int, E: int, s_exp: float, device, seed: int) -> torch.Tensor:
    """Expert popularity P(e) proportional to (e+1)^-s; k distinct draws per token."""
    p = torch.arange(1, E + 1, dtype=torch.float64).pow(-s_exp)
    p = (p / p.sum()).to(torch.float32).to(device)
    probs = p.expand(W * T, E).contiguous()
    ids = torch.multinomial(probs, k, replacement=False, generator=_gen(device, seed))
    return ids.view(W, T, k).to(torch.int32)


def make_inputs(wl: Workload, device="cpu", with_weights: bool = True) -> Inputs:
    """Draw one workload's inputs with fixed seeds (seed + a per-tensor offset)."""
    W, L, T, D, F, E, k = wl.W, wl.L, wl.T, wl.d_model, wl.d_ff, wl.E, wl.topk
    base = wl.seed * 1000
    x = [_normal_bf16((T, D), wl.x_std, device, base + 10 + s) for s in range(W)]
    if with_weights:
        w_gate = [_normal_bf16((L, F, D), wl.w_std, device, base + 100 + s) for s in range(W)]
        w_up = [_normal_bf16((L, F, D), wl.w_std, device, base + 200 + s) for s in range(W)]
        w_down = [_normal_bf16((L, D, F), wl.w_std, device, base + 300 + s) for s in range(W)]
    else:
        w_gate = w_up = w_down = []
    logits = torch.empty((W, T, E), dtype=torch.float32, device=device)
    logits.normal_(0.0, 1.0, generator=_gen(device, base + 1))
    if wl.routing == "gate":
        forced = None
    elif wl.routing == "balanced":
        forced = balanced_ids(W, T, k, E, device)
    elif wl.routing == "zipf":
        forced = zipf_ids(W, T, k, E, wl.zipf_s, device, base + 2)
    else:
        raise ValueError(f"unknown routing {wl.routing!r}")
    return Inputs(wl, x, w_gate, w_up, w_down, logits, forced)


def router_weights(wl: Workload, device="cpu") -> torch.Tensor:
    """Router weights [E, D] bf16 ~ N(0, 1/(D * x_std^2)): the scores of N(0, x_std)
    token rows then have unit variance, like the drawn gate logits."""
    std = 1.0 / (wl.d_model ** 0.5 * wl.x_std)
    return _normal_bf16((wl.E, wl.d_model), std, device, wl.seed * 1000 + 3)
