"""Seeded synthetic inputs for the routed top-k expert layer.

This module only draws caller-side inputs: tokens ``x[T,D]``, top-k expert ids ``[T,K]``,
top-k scores ``[T,K]`` and expert weights ``w13[E,2,F,D]`` / ``w2[E,D,F]``. It holds none of the
layer's arithmetic, so the CUDA path and the CPU oracle can both be fed from it without sharing
any computation.

Workloads (shapes and distributions):

* ``tiny`` -- the Dist-MoE 0.1.0 "BF16 Quickstart" shapes (T=16, D=256, F=256, K=2, two ranks of
  four local experts, so E=8) with its round-robin routing ``(t*K + k) % E`` and scores ``1/K``.
  The Primus MegaMoE guide, "Router force load balancing" table, row ``even``, names the same
  round-robin rule and notes that it gives exactly equal per-expert counts.
* ``medium``, ``decode``, ``large`` -- per token K distinct experts drawn uniformly without
  replacement (the ``uniform`` row of that table: random logits, balanced only statistically),
  scores = softmax of K standard-normal logits, renormalised to sum 1, fp32.
* ``skewed`` -- experts drawn without replacement (successive sampling, i.e. Gumbel-top-K on
  ``log p_e``) from ``p_e ~ (e+1)^-s`` over the first ``E - round(0.05 E)`` experts, zero for the
  rest. ``s`` is chosen so that the hottest expert's expected load is 3.0x the mean load
  ``T*K/E``; 3.0 is the peak-to-mean ratio of the TeraMoE README's imbalance result.

Weights are bf16 draws from N(0, 1/sqrt(fan_in)) (fan_in = D for w13, F for w2), so the gate/up
pre-activations and the outputs stay near unit scale; x ~ N(0, 1) in bf16.

Every tensor has its own generator, seeded from (seed, tensor name, index), so no tensor depends
on the order in which the others were drawn. Expert weights are drawn one expert at a time with
one generator per expert, which keeps the peak temporary memory at one expert.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import torch

__all__ = [
    "Workload",
    "WORKLOADS",
    "SKEW_ZIPF_S",
    "skew_zipf_probs",
    "make_x",
    "make_topk_ids",
    "make_scores",
    "make_weights",
    "make_inputs",
    "generator",
]


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    D: int
    F: int
    E: int
    K: int
    routing: str  # "round_robin" | "uniform" | "zipf"
    scores: str  # "one_over_k" | "softmax"

    @property
    def R(self) -> int:
        return self.T * self.K

    def dims(self) -> tuple[int, int, int, int, int]:
        return self.T, self.D, self.F, self.E, self.K


WORKLOADS: dict[str, Workload] = {
    "tiny": Workload("tiny", 16, 256, 256, 8, 2, "round_robin", "one_over_k"),
    "medium": Workload("medium", 4096, 2048, 1408, 64, 6, "uniform", "softmax"),
    "decode": Workload("decode", 64, 7168, 2048, 256, 8, "uniform", "softmax"),
    "large": Workload("large", 16384, 7168, 2048, 256, 8, "uniform", "softmax"),
    "skewed": Workload("skewed", 16384, 4096, 1536, 128, 8, "zipf", "softmax"),
}

# Zipf exponent for the skewed workload (E=128, K=8, 122 non-empty experts). It solves
#   P(expert 0 is among the K draws) = 3.0 * K / E
# for successive sampling without replacement, with the inclusion probability evaluated as the
# exponential-race integral  int_0^inf p_0 exp(-p_0 t) P(fewer than K other clocks fired by t) dt
# (Poisson-binomial tail by dynamic programming). tests/test_workloads.py re-derives it.
SKEW_ZIPF_S = 0.30112681887945536
SKEW_ZERO_FRACTION = 0.05
SKEW_PEAK_TO_MEAN = 3.0

_STREAMS = {"x": 1, "ids": 2, "scores": 3, "w13": 4, "w2": 5}


def generator(seed: int, name: str, index: int = 0, device: str | torch.device = "cpu") -> torch.Generator:
    """A torch generator seeded from (seed, tensor name, index) only."""
    mixed = (int(seed) * 1_000_003 + _STREAMS[name] * 7_919 + int(index) * 104_729 + 12_345) % (2**63 - 1)
    g = torch.Generator(device=device)
    g.manual_seed(mixed)
    return g


def make_x(T: int, D: int, seed: int = 0, device="cpu") -> torch.Tensor:
    g = generator(seed, "x", 0, device)
    return torch.randn((T, D), generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def skew_zipf_probs(E: int, s: float = SKEW_ZIPF_S, zero_fraction: float = SKEW_ZERO_FRACTION) -> torch.Tensor:
    """p_e ~ (e+1)^-s on the first E - round(zero_fraction*E) experts, 0 on the rest (float64)."""
    n_zero = int(round(zero_fraction * E))
    p = torch.zeros(E, dtype=torch.float64)
    live = E - n_zero
    p[:live] = (torch.arange(live, dtype=torch.float64) + 1.0) ** (-s)
    return p / p.sum()


def make_topk_ids(T: int, E: int, K: int, routing: str, seed: int = 0, device="cpu") -> torch.Tensor:
    """Top-k expert ids [T,K] int32, contiguous."""
    if routing == "round_robin":
        t = torch.arange(T, device=device, dtype=torch.int64)[:, None]
        k = torch.arange(K, device=device, dtype=torch.int64)[None, :]
        return ((t * K + k) % E).to(torch.int32).contiguous()
    g = generator(seed, "ids", 0, device)
    if routing == "uniform":
        if K > E:
            raise ValueError("uniform distinct routing needs K <= E")
        keys = torch.rand((T, E), generator=g, device=device, dtype=torch.float32)
        return keys.topk(K, dim=1).indices.to(torch.int32).contiguous()
    if routing == "zipf":
        p = skew_zipf_probs(E).to(device)
        logp = torch.where(p > 0, p.log(), torch.full_like(p, -math.inf)).to(torch.float32)
        u = torch.rand((T, E), generator=g, device=device, dtype=torch.float32)
        u = u.clamp_(min=1e-12, max=1.0 - 1e-7)
        gumbel = -torch.log(-torch.log(u))
        return (logp[None, :] + gumbel).topk(K, dim=1).indices.to(torch.int32).contiguous()
    raise ValueError(f"unknown routing {routing!r}")


def make_scores(T: int, K: int, kind: str, seed: int = 0, device="cpu") -> torch.Tensor:
    """Top-k scores [T,K] fp32."""
    if kind == "one_over_k":
        return torch.full((T, K), 1.0 / K, device=device, dtype=torch.float32)
    if kind == "softmax":
        g = generator(seed, "scores", 0, device)
        logits = torch.randn((T, K), generator=g, device=device, dtype=torch.float32)
        s = torch.softmax(logits, dim=1)
        return (s / s.sum(dim=1, keepdim=True)).contiguous()
    raise ValueError(f"unknown score kind {kind!r}")


def make_weights(E: int, D: int, F: int, seed: int = 0, device="cpu", experts=None):
    """w13 [E,2,F,D] and w2 [E,D,F] bf16, drawn one expert at a time.

    ``experts`` (an iterable of expert indices) restricts the draw to those experts; the others are
    left zero. Expert e's values do not depend on which other experts are drawn.
    """
    w13 = torch.zeros((E, 2, F, D), dtype=torch.bfloat16, device=device)
    w2 = torch.zeros((E, D, F), dtype=torch.bfloat16, device=device)
    s13 = 1.0 / math.sqrt(D)
    s2 = 1.0 / math.sqrt(F)
    for e in range(E) if experts is None else experts:
        g = generator(seed, "w13", e, device)
        w13[e] = torch.randn((2, F, D), generator=g, device=device, dtype=torch.float32).mul_(s13).to(torch.bfloat16)
        g = generator(seed, "w2", e, device)
        w2[e] = torch.randn((D, F), generator=g, device=device, dtype=torch.float32).mul_(s2).to(torch.bfloat16)
    return w13, w2


def make_inputs(workload, seed: int = 0, device="cpu", weights: bool = True) -> dict:
    """All inputs of one workload (a name in WORKLOADS or a Workload)."""
    wl = WORKLOADS[workload] if isinstance(workload, str) else workload
    out = {
        "workload": wl,
        "x": make_x(wl.T, wl.D, seed, device),
        "topk_ids": make_topk_ids(wl.T, wl.E, wl.K, wl.routing, seed, device),
        "topk_scores": make_scores(wl.T, wl.K, wl.scores, seed, device),
    }
    if weights:
        out["w13"], out["w2"] = make_weights(wl.E, wl.D, wl.F, seed, device)
    return out
