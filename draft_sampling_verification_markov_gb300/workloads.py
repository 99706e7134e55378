"""Seeded synthetic inputs for the speculative-decoding hot path.

This module only draws random tensors with the shapes, dtypes and value distributions of the
five workloads; it computes nothing that the method computes. Both the CUDA path and the CPU
oracle consume exactly these bytes (the bytes, not the generator, are what parity compares).

Generators are ``torch.Generator`` streams seeded per tensor, on the requested device: the CUDA
Philox stream for the large workloads, the CPU stream for host-only tests. A workload drawn on
one device type is therefore not byte-identical to the same workload drawn on another; every
parity comparison hands the same drawn bytes to both sides.

Workloads (names describe what they are; sizes are the defaults):
  greedy_toy             R=4, gamma=4, V=32000, rank 256, fp32 everything, greedy (T=0)
  mtp_greedy             R=64, gamma=3, V=129280, bf16, no Markov head, planted acceptance 0.88
  markov_rejection       R=256, gamma=7, V=129280, rank 256, bf16, T=1
  confidence_scheduling  R=512, gamma=16, V=129280, rank 256, bf16, T=1, SPS table to B=8704
  full_loop              R=1024, gamma=16, V=129280, rank 256, bf16, Zipf(1.1) prior, T=0.7,
                         20 chained iterations, SPS table to B=17408
  sparse_targets         markov_rejection's shapes on a vocab-shuffled Zipf(1.1) prior, with
                         top-k or top-p truncated target rows (-inf outside the nucleus)
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import torch


@dataclass
class Workload:
    name: str
    R: int
    gamma: int
    V: int
    rank: int
    temperature: float
    U: torch.Tensor                       # draft base logits [R, gamma, V]
    target: torch.Tensor                  # target logits [R, gamma + 1, V]
    W1: Optional[torch.Tensor] = None     # Markov embedding [V, rank]
    W2: Optional[torch.Tensor] = None     # Markov projection [V, rank] (row v -> token v)
    anchors: Optional[torch.Tensor] = None  # int32 [R]
    u_draft: Optional[torch.Tensor] = None  # fp32 [iters, R, gamma] or [R, gamma]
    u_accept: Optional[torch.Tensor] = None
    u_resid: Optional[torch.Tensor] = None  # fp32 [iters, R] or [R]
    sps: Optional[torch.Tensor] = None     # fp64 [Bmax + 1], index = B
    iterations: int = 1
    extra: dict = field(default_factory=dict)

    @property
    def logit_rows(self) -> int:
        """Draft rows R*gamma plus target rows R*(gamma+1)."""
        return self.R * self.gamma + self.R * (self.gamma + 1)

    def tensors(self):
        return {k: getattr(self, k) for k in ("U", "target", "W1", "W2", "anchors", "u_draft",
                                               "u_accept", "u_resid", "sps")
                if getattr(self, k) is not None}


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _normal(shape, std, seed, device):
    return torch.randn(shape, generator=_gen(device, seed), device=device,
                       dtype=torch.float32) * std


def _uniform(shape, seed, device):
    return torch.rand(shape, generator=_gen(device, seed), device=device, dtype=torch.float32)


def _anchors(R, V, seed, device):
    return torch.randint(0, V, (R,), generator=_gen(device, seed), device=device,
                         dtype=torch.int64).to(torch.int32)


def sps_table(Bmax: int, base_ms: float = 20.0, step_ms: float = 0.6, step: int = 128):
    """Synthetic steps-per-second table SPS[B] for B = 0..Bmax: a step time of
    base_ms + step_ms * ceil(B / step) milliseconds, i.e. a decreasing, staircase-shaped
    envelope whose throughput B * SPS(B) is a sawtooth with a tooth every `step` tokens.
    SPS[0] is the value of the first stair."""
    B = torch.arange(Bmax + 1, dtype=torch.float64)
    stairs = torch.clamp(torch.ceil(B / step), min=1.0)
    return 1000.0 / (base_ms + step_ms * stairs)


def _markov_weights(V, rank, std, seed, device, dtype):
    W1 = _normal((V, rank), std, seed * 10 + 1, device).to(dtype)
    W2 = _normal((V, rank), std, seed * 10 + 2, device).to(dtype)
    return W1, W2


def greedy_toy(device="cpu", R=4, gamma=4, V=32000, rank=256, seed=1001) -> Workload:
    """fp32 greedy toy: U ~ N(0, 2^2); W1, W2 ~ N(0, 0.02^2); target rows 0..gamma-1 are the
    U rows plus N(0, 0.5^2) noise, row gamma is a fresh N(0, 2^2) row plus the same noise;
    anchors uniform in [0, V); greedy (T = 0)."""
    U = _normal((R, gamma, V), 2.0, seed * 10 + 3, device)
    noise = _normal((R, gamma + 1, V), 0.5, seed * 10 + 4, device)
    fresh = _normal((R, 1, V), 2.0, seed * 10 + 5, device)
    target = torch.cat([U, fresh], dim=1) + noise
    W1, W2 = _markov_weights(V, rank, 0.02, seed, device, torch.float32)
    return Workload("greedy_toy", R, gamma, V, rank, 0.0, U.contiguous(), target.contiguous(),
                    W1, W2, _anchors(R, V, seed * 10 + 6, device))


def mtp_greedy(device="cpu", R=64, gamma=3, V=129280, seed=1002, p_plant=0.88,
               sigma=3.0) -> Workload:
    """MTP-1-style greedy verify, bf16: draft logits and target logits ~ N(0, 3^2). The draft
    tokens x are drawn uniformly and planted in the draft logits at 12 sigma (far above the
    row maximum of V normal draws, so x is the draft argmax); each target row i < gamma gets
    x_{i+1} planted at the same height with probability p_plant (seeded Bernoulli), which makes
    the expected accepted length p + p^2 + p^3 for gamma = 3."""
    plant = 12.0 * sigma
    D = _normal((R, gamma, V), sigma, seed * 10 + 3, device)
    T = _normal((R, gamma + 1, V), sigma, seed * 10 + 4, device)
    x = torch.randint(0, V, (R, gamma), generator=_gen(device, seed * 10 + 5), device=device)
    D.scatter_(2, x.unsqueeze(-1), plant)
    keep = _uniform((R, gamma), seed * 10 + 6, device) < p_plant
    rows = T[:, :gamma, :]                      # a view: the scatter below writes into T
    idx = x.unsqueeze(-1)
    cur = rows.gather(2, idx)
    rows.scatter_(2, idx, torch.where(keep.unsqueeze(-1), torch.full_like(cur, plant), cur))
    wl = Workload("mtp_greedy", R, gamma, V, 0, 0.0, D.to(torch.bfloat16).contiguous(),
                  T.to(torch.bfloat16).contiguous(), anchors=_anchors(R, V, seed * 10 + 7,
                                                                       device))
    wl.extra["planted_tokens"] = x.to(torch.int32)
    wl.extra["planted_mask"] = keep
    return wl


def _bf16_pair(R, gamma, V, seed, device, prior=None):
    """U ~ N(0, 2^2) and target rows = U rows + N(0, 1) (row gamma fresh N(0, 2^2) + N(0, 1)),
    optionally plus a per-token prior, all in fp32 before the bf16 cast."""
    U = _normal((R, gamma, V), 2.0, seed * 10 + 3, device)
    fresh = _normal((R, 1, V), 2.0, seed * 10 + 5, device)
    T = torch.cat([U, fresh], dim=1)
    T += _normal((R, gamma + 1, V), 1.0, seed * 10 + 4, device)
    if prior is not None:
        U += prior
        T += prior
    return U.to(torch.bfloat16).contiguous(), T.to(torch.bfloat16).contiguous()


def markov_rejection(device="cpu", R=256, gamma=7, V=129280, rank=256, seed=1003,
                     temperature=1.0) -> Workload:
    """DSpark Markov sampling + lossless rejection, bf16, T = 1. Uniforms from seeded streams
    (seed 2003 family) for the draft draw, the acceptance test and the final draw."""
    U, T = _bf16_pair(R, gamma, V, seed, device)
    W1, W2 = _markov_weights(V, rank, 0.02, seed, device, torch.bfloat16)
    useed = seed + 1000
    return Workload("markov_rejection", R, gamma, V, rank, temperature, U, T, W1, W2,
                    _anchors(R, V, seed * 10 + 6, device),
                    u_draft=_uniform((R, gamma), useed * 10 + 1, device),
                    u_accept=_uniform((R, gamma), useed * 10 + 2, device),
                    u_resid=_uniform((R,), useed * 10 + 3, device))


def confidence_scheduling(device="cpu", R=512, gamma=16, V=129280, rank=256, seed=1004,
                          temperature=1.0, Bmax=None) -> Workload:
    """Confidence + scheduling: logits as markov_rejection; Markov-sampled drafts (uniforms
    supplied); SPS table over B in [0, R*(gamma+1)] (8704 at the default size)."""
    wl = markov_rejection(device, R, gamma, V, rank, seed, temperature)
    wl.name = "confidence_scheduling"
    wl.sps = sps_table(R * (gamma + 1) if Bmax is None else Bmax)
    return wl


def zipf_prior(V, s=1.1, device="cpu"):
    """Token-frequency prior -s * ln(v + 1) (token id = frequency rank)."""
    return -s * torch.log(torch.arange(V, device=device, dtype=torch.float32) + 1.0)


def shuffled_zipf_prior(V, s=1.1, seed=7, device="cpu"):
    """Zipf(s) prior -s * ln(rank + 1) with the frequency ranks dealt to token ids by a seeded
    random permutation (so frequent tokens are scattered over the vocabulary)."""
    rank = torch.randperm(V, generator=_gen(device, seed), device=device).to(torch.float32)
    return -s * torch.log(rank + 1.0)


def truncate_rows(logits, top_k=None, top_p=None):
    """Target-side truncation of each row's distribution (the row's own softmax at T = 1): keep
    the top_k largest logits, or the smallest set of largest logits whose probability reaches
    top_p, and set every other logit to -inf. Computed with torch in fp64 on a sorted copy;
    ties at the cut keep the lower token ids."""
    x = logits.double()
    flat = x.reshape(-1, x.shape[-1])
    # stable descending order: larger logit first, lower id first among equals
    order = torch.sort(flat, dim=-1, descending=True, stable=True).indices
    keep = torch.zeros_like(flat, dtype=torch.bool)
    if top_k is not None:
        keep.scatter_(1, order[:, :top_k], True)
    else:
        srt = torch.gather(flat, 1, order)
        p = torch.softmax(srt, dim=-1)
        before = torch.cumsum(p, dim=-1) - p            # mass of the larger logits
        keep_sorted = before < top_p                    # includes the one that reaches top_p
        keep.scatter_(1, order, keep_sorted)
    out = torch.where(keep, flat, torch.full_like(flat, float("-inf")))
    return out.reshape(logits.shape).to(logits.dtype).contiguous()


def sparse_targets(device="cpu", R=256, gamma=7, V=129280, rank=256, seed=1006,
                   temperature=1.0, top_k=None, top_p=None, zipf_seed=1106) -> Workload:
    """Markov sampling + rejection verify on a vocab-shuffled Zipf(1.1) prior (added to U and to
    the target in fp32 before the bf16 cast) with top-k or top-p truncated target rows (every
    target row keeps only its nucleus; other target logits are -inf). The draft side is not
    truncated, so draft tokens outside the nucleus occur and must be rejected."""
    U, T = _bf16_pair(R, gamma, V, seed, device, prior=shuffled_zipf_prior(V, 1.1, zipf_seed,
                                                                              device))
    if top_k is not None or top_p is not None:
        T = truncate_rows(T, top_k=top_k, top_p=top_p)
    W1, W2 = _markov_weights(V, rank, 0.02, seed, device, torch.bfloat16)
    useed = seed + 1000
    wl = Workload("sparse_targets", R, gamma, V, rank, temperature, U, T, W1, W2,
                  _anchors(R, V, seed * 10 + 6, device),
                  u_draft=_uniform((R, gamma), useed * 10 + 1, device),
                  u_accept=_uniform((R, gamma), useed * 10 + 2, device),
                  u_resid=_uniform((R,), useed * 10 + 3, device))
    wl.extra.update(top_k=top_k, top_p=top_p)
    return wl


def full_loop(device="cpu", R=1024, gamma=16, V=129280, rank=256, iterations=20, seed=1005,
              temperature=0.7, Bmax=None) -> Workload:
    """Full draft -> verify loop: bf16 logits with a Zipf(1.1) prior added to U and target,
    T = 0.7, `iterations` chained iterations with per-iteration uniforms [iters, R, gamma] x 2
    and [iters, R], SPS table over B in [0, R*(gamma+1)] (17408 at the default size)."""
    U, T = _bf16_pair(R, gamma, V, seed, device, prior=zipf_prior(V, 1.1, device))
    W1, W2 = _markov_weights(V, rank, 0.02, seed, device, torch.bfloat16)
    useed = seed + 1000
    return Workload("full_loop", R, gamma, V, rank, temperature, U, T, W1, W2,
                    _anchors(R, V, seed * 10 + 6, device),
                    u_draft=_uniform((iterations, R, gamma), useed * 10 + 1, device),
                    u_accept=_uniform((iterations, R, gamma), useed * 10 + 2, device),
                    u_resid=_uniform((iterations, R), useed * 10 + 3, device),
                    sps=sps_table(R * (gamma + 1) if Bmax is None else Bmax),
                    iterations=iterations)


def random_survival(R, gamma, seed, device="cpu", low=0.05):
    """Scheduler input independent of either path: each row holds gamma draws from
    U[low, 1) sorted in decreasing order, so a_{r,j} is non-increasing in j as a survival
    row must be."""
    a = low + (1.0 - low) * _uniform((R, gamma), seed, device)
    return torch.sort(a, dim=1, descending=True).values.contiguous()


BY_NAME = {
    "greedy_toy": greedy_toy,
    "mtp_greedy": mtp_greedy,
    "markov_rejection": markov_rejection,
    "confidence_scheduling": confidence_scheduling,
    "full_loop": full_loop,
    "sparse_targets": sparse_targets,
}


def describe_sizes(wl: Workload) -> dict:
    d = dict(R=wl.R, gamma=wl.gamma, V=wl.V, rank=wl.rank, temperature=wl.temperature,
             iterations=wl.iterations)
    d["u_bytes"] = wl.U.numel() * wl.U.element_size()
    d["target_bytes"] = wl.target.numel() * wl.target.element_size()
    return d


__all__ = ["Workload", "greedy_toy", "mtp_greedy", "markov_rejection", "confidence_scheduling",
           "full_loop", "sps_table", "zipf_prior", "random_survival", "BY_NAME",
           "describe_sizes"]
