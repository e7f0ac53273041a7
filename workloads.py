"""Seeded synthetic workloads for the MoE layer hot path.

This module is the only code shared by the CUDA path's tests/benchmark and the
CPU oracle's tests.  It holds shapes and random-number recipes and nothing of
the method's arithmetic: no routing, no capacity rounding, no permutation, no
expert math.  Every tensor is drawn from ``torch.Generator`` seeded with the
workload's seed, on whatever device the caller names; the oracle always runs on
a host copy of exactly the tensors the GPU path received.

Workload recipes (shapes follow the pages' model families):

* ``tiny``   T=256, d=64, E=8, top-2, I=128, capacity factor 1.25, softmax
             gates over the selected logits.  Seed 0.
* ``decode`` Qwen3-30B-A3B-shaped: d=2048, E=128, top-8, I=768, dropless,
             T in {1, 8, 32, 128}; logits N(0,1) plus a per-expert N(0, 0.5)
             bias (std 0.5) to skew load.  Seed 1.
* ``prefill`` Mixtral-shaped: T=4096, d=4096, E=8, top-2, I=14336, dropless.
             Seed 2.
* ``v3``     DeepSeek-V3-shaped: T=8192, d=7168, 256 experts in 8 groups,
             top-4 groups then top-8 experts, I=2048, one always-on shared
             expert of I=2048, capacity factor 1.0 with drops counted, sigmoid
             gates with route scale 2.5; selection-only bias 0.2 * r^-1.1
             (Zipf s=1.1 over a seeded expert ranking).  Seed 3.
* ``pooled`` 8-of-384 pooled-wave layout: T=65,536, d=3072 latent, E=384 =
             64 destinations x 6 local experts, 3 waves, sender capacity
             factor 1.10, receiver capacity factor 1.15, I=1536; logits N(0,1)
             plus 1.0 * r^-1.0 (Zipf s=1.0).  Seed 4.

Activations are bf16 N(0,1); expert weights are bf16 N(0, std=1/sqrt(fan_in))
with fan_in = d for the gate/up matrices [E,d,I] and fan_in = I for the down
matrix [E,I,d].  Router logits are fp32 and are given as inputs.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    E: int
    k: int
    I: int
    seed: int
    capacity_factor: Optional[float] = None  # None = dropless
    score_fn: str = "softmax"  # "softmax" (selected-logit softmax) or "sigmoid_group"
    n_group: int = 1
    topk_group: int = 1
    route_scale: float = 1.0
    shared_I: int = 0  # intermediate width of the always-on shared expert (0 = none)
    logit_bias: str = "none"  # "none" | "normal0.5" | "zipf1.0" | "hot<n>" (edge-case tests)
    selection_bias: str = "none"  # "none" | "zipf1.1x0.2" (sigmoid_group only)
    # pooled-wave layout (0 = not pooled)
    n_dest: int = 0
    local_per_dest: int = 0
    n_waves: int = 0
    sender_cf: float = 0.0
    receiver_cf: float = 0.0

    @property
    def R(self) -> int:
        return self.T * self.k

    @property
    def pooled(self) -> bool:
        return self.n_dest > 0


def tiny() -> Workload:
    return Workload("tiny", T=256, d=64, E=8, k=2, I=128, seed=0, capacity_factor=1.25)


def decode(T: int = 128) -> Workload:
    assert T in (1, 8, 32, 128) or T > 0
    return Workload(f"decode_T{T}", T=T, d=2048, E=128, k=8, I=768, seed=1,
                    logit_bias="normal0.5")


def prefill() -> Workload:
    return Workload("prefill", T=4096, d=4096, E=8, k=2, I=14336, seed=2)


def v3(T: int = 8192) -> Workload:
    return Workload(f"v3_T{T}" if T != 8192 else "v3", T=T, d=7168, E=256, k=8, I=2048,
                    seed=3, capacity_factor=1.0, score_fn="sigmoid_group", n_group=8,
                    topk_group=4, route_scale=2.5, shared_I=2048,
                    selection_bias="zipf1.1x0.2")


def pooled(T: int = 65536) -> Workload:
    return Workload(f"pooled_T{T}" if T != 65536 else "pooled", T=T, d=3072, E=384, k=8,
                    I=1536, seed=4, logit_bias="zipf1.0", n_dest=64, local_per_dest=6,
                    n_waves=3, sender_cf=1.10, receiver_cf=1.15)


def scaled(w: Workload, **kw) -> Workload:
    """A smaller copy of a workload (same recipe, different sizes) for fast tests."""
    return dataclasses.replace(w, **kw)


# ----------------------------------------------------------------------------
# Generators
# ----------------------------------------------------------------------------

def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _zipf_ranked(E: int, s: float, scale: float, g: torch.Generator, device) -> torch.Tensor:
    """scale * r_e^-s with r_e = 1 + position of expert e in a seeded permutation."""
    perm = torch.randperm(E, generator=g, device=device)
    rank = torch.empty(E, dtype=torch.float64, device=device)
    rank[perm] = torch.arange(1, E + 1, dtype=torch.float64, device=device)
    return (scale * rank.pow(-s)).to(torch.float32)


def _randn_bf16(shape, std: float, g: torch.Generator, device, chunk_rows: int = 1 << 14):
    """bf16 N(0, std) drawn in fp32 chunks along dim 0 (bounds the fp32 temporary)."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(shape[0], -1)
    for r0 in range(0, shape[0], chunk_rows):
        r1 = min(shape[0], r0 + chunk_rows)
        tmp = torch.randn((r1 - r0, flat.shape[1]), generator=g, device=device,
                          dtype=torch.float32)
        flat[r0:r1] = (tmp * std).to(torch.bfloat16)
    return out


def make_router_inputs(w: Workload, device="cpu"):
    """Router logits fp32 [T,E] and the selection-only bias fp32 [E] (or None)."""
    g = _gen(w.seed, device)
    logits = torch.randn((w.T, w.E), generator=g, device=device, dtype=torch.float32)
    gb = _gen(w.seed + 1000, device)
    if w.logit_bias == "normal0.5":
        b = torch.randn((w.E,), generator=gb, device=device, dtype=torch.float32) * 0.5
        logits = logits + b
    elif w.logit_bias == "zipf1.0":
        logits = logits + _zipf_ranked(w.E, 1.0, 1.0, gb, device)
    elif w.logit_bias.startswith("hot"):
        # degenerate skew for edge-case tests: every token prefers the first n experts
        n = int(w.logit_bias[3:])
        logits[:, :n] += 20.0
    sel_bias = None
    if w.selection_bias == "zipf1.1x0.2":
        sel_bias = _zipf_ranked(w.E, 1.1, 0.2, gb, device)
    return logits.contiguous(), sel_bias


def make_activations(w: Workload, device="cpu") -> torch.Tensor:
    """Token activations bf16 [T,d] ~ N(0,1)."""
    g = _gen(w.seed + 2000, device)
    return _randn_bf16((w.T, w.d), 1.0, g, device)


def n_weight_sets(w: Workload) -> int:
    """Routed expert weight sets held: E, or the local experts per destination when pooled."""
    return w.local_per_dest if w.pooled else w.E


def make_expert_weights(w: Workload, device="cpu", n_experts: Optional[int] = None, I=None,
                        seed_offset: int = 0):
    """(W_gate [n,d,I], W_up [n,d,I], W_down [n,I,d]) bf16, std 1/sqrt(fan_in)."""
    n = n_weight_sets(w) if n_experts is None else n_experts
    I = w.I if I is None else I
    g = _gen(w.seed + 3000 + seed_offset, device)
    wg = _randn_bf16((n, w.d, I), 1.0 / math.sqrt(w.d), g, device, chunk_rows=1)
    wu = _randn_bf16((n, w.d, I), 1.0 / math.sqrt(w.d), g, device, chunk_rows=1)
    wd = _randn_bf16((n, I, w.d), 1.0 / math.sqrt(I), g, device, chunk_rows=1)
    return wg, wu, wd


def make_shared_weights(w: Workload, device="cpu"):
    """The always-on shared expert's (W_gate, W_up, W_down) with one leading expert axis."""
    if w.shared_I == 0:
        return None
    return make_expert_weights(w, device, n_experts=1, I=w.shared_I, seed_offset=500)


def bf16_bits(t: torch.Tensor):
    """Raw uint16 bits of a bf16 tensor as a host numpy array (for the oracle)."""
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view("uint16")
