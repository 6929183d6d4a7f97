"""Seeded synthetic inputs for the MoE layer (no arithmetic of the method here).

Recipe (the same for the tests, the smoke check and the benchmark):
  * activations x: bf16 ~ N(0, 1), seed 0;
  * router logits: fp32 ~ N(0, 1), seed 1 (uniform expert load), or the Zipf
    recipe below;
  * expert weights: fp32 ~ N(0, 0.02); gate_up expert e uses seed 2 + e and
    down expert e uses seed 2 + E + e, so any one expert can be regenerated
    alone.  Small cases draw on the CPU generator, full-size cases on the CUDA
    generator of the device (the same seeds; a CPU copy of an expert is
    produced by drawing on that device again and copying back).
  * Zipf(s) expert popularity: logits[t, e] = log p_e + Gumbel(0, 1) with
    p_e proportional to rank(e)^-s over a seed-fixed random ranking of the
    experts.  With Gumbel perturbations, the top-k experts of a token are a
    draw of k experts without replacement weighted by p (the Gumbel-top-k
    construction), so expert load follows the Zipf popularity.
"""
from __future__ import annotations

import math

import torch


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def activations(T: int, H: int, seed: int = 0, device="cpu") -> torch.Tensor:
    return torch.randn((T, H), generator=_gen(seed, device), device=device, dtype=torch.float32).to(torch.bfloat16)


def router_logits(T: int, E: int, seed: int = 1, zipf_s: float | None = None, device="cpu") -> torch.Tensor:
    if zipf_s is None:
        return torch.randn((T, E), generator=_gen(seed, device), device=device, dtype=torch.float32)
    g = _gen(seed, "cpu")
    ranking = torch.randperm(E, generator=g)
    rank_of = torch.empty(E, dtype=torch.float64)
    rank_of[ranking] = torch.arange(1, E + 1, dtype=torch.float64)
    logp = -zipf_s * torch.log(rank_of)
    logp = logp - torch.logsumexp(logp, 0)
    u = torch.rand((T, E), generator=g, dtype=torch.float64).clamp_(1e-300, 1.0)
    gumbel = -torch.log(-torch.log(u))
    return (logp[None, :] + gumbel).to(torch.float32).to(device)


def router_gate(E: int, H: int, seed: int = 100000, device="cpu", std: float = 0.02) -> torch.Tensor:
    """Gate matrix w_gate [E][H] in bf16, ~N(0, std)."""
    return (torch.randn((E, H), generator=_gen(seed, device), device=device, dtype=torch.float32) * std).to(
        torch.bfloat16)


def expert_weight(e: int, N: int, K: int, seed_base: int, device="cpu", std: float = 0.02) -> torch.Tensor:
    return torch.randn((N, K), generator=_gen(seed_base + e, device), device=device, dtype=torch.float32) * std


def gate_up_seed_base() -> int:
    return 2


def down_seed_base(E: int) -> int:
    return 2 + E


def expert_weights(E: int, N: int, K: int, seed_base: int, device="cpu", std: float = 0.02) -> torch.Tensor:
    out = torch.empty((E, N, K), dtype=torch.float32, device=device)
    for e in range(E):
        out[e] = expert_weight(e, N, K, seed_base, device, std)
    return out


def zipf_expected_max_load(E: int, k: int, T: int, s: float) -> float:
    """Rough upper estimate of the busiest expert's rows under Zipf(s) (sizing hint only)."""
    h = sum(r ** -s for r in range(1, E + 1))
    return min(T, T * k / h * 1.0 + 4 * math.sqrt(T))
