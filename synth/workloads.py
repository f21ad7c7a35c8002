"""Workload definitions and seeded generators.

Input distributions follow the configurations this library is measured on:

* checkpoint state S0 ~ N(0, 0.1^2), fp32, layout [n_slot, H, d_v, d_k];
* q, k ~ N(0, 1) drawn in fp32 and L2-normalised per (token, head) over d_k,
  then cast to the input dtype (bf16 round-to-nearest-even, or kept fp32);
* v ~ N(0, 1) cast the same way;
* g = -softplus(N(0, 1)) (so alpha = exp(g) lies in (0, 1)), beta = sigmoid(N(0, 1));
* the "edge" workload mixes in g = 0, g = -20, beta = 1e-4 and beta = 1 - 1e-4;
* accepted counts per sequence and step follow each workload's law.

The random numbers are drawn with ``torch.Generator`` on the CPU so the same
seed gives the same tensors on every machine.  Nothing here computes any part
of the recurrence; the normalisation of q and k is part of the input
distribution, not of the kernels (the kernels never re-normalise).
"""
from __future__ import annotations

import dataclasses
import math

import torch

BASE_SEED = 20261202


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    cfg_id: int
    B: int
    H: int
    dk: int
    dv: int
    T: int
    threshold: int
    in_dtype: str          # "bf16" or "fp32"
    steps: int
    layers: int
    accept_law: str        # "uniform", "geometric12", "forced"
    gate_law: str          # "normal" or "extreme"
    len0_law: str          # "fixed3" or "uniform"
    forced_flush: bool = False

    @property
    def cap(self) -> int:
        # With a flush of every sequence whose length reaches the threshold
        # after each accept, the length before a verify is at most
        # threshold - 1, so a verify needs threshold - 1 + T slots.
        return self.threshold - 1 + self.T

    @property
    def n_slot(self) -> int:
        # One spare slot per four sequences so the slot map is a real gather.
        return self.B + max(1, self.B // 4)

    @property
    def torch_in_dtype(self) -> torch.dtype:
        return torch.bfloat16 if self.in_dtype == "bf16" else torch.float32

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.dk)


WORKLOADS = {
    "tiny": Workload("tiny", 1, B=1, H=2, dk=64, dv=64, T=4, threshold=8,
                     in_dtype="fp32", steps=1, layers=1, accept_law="uniform",
                     gate_law="normal", len0_law="fixed3", forced_flush=True),
    "b8": Workload("b8", 2, B=8, H=16, dk=128, dv=128, T=16, threshold=32,
                   in_dtype="bf16", steps=64, layers=1, accept_law="geometric12",
                   gate_law="normal", len0_law="uniform"),
    "decode24": Workload("decode24", 3, B=32, H=16, dk=128, dv=128, T=16, threshold=32,
                         in_dtype="bf16", steps=64, layers=24, accept_law="geometric12",
                         gate_law="normal", len0_law="uniform"),
    "edge": Workload("edge", 4, B=12, H=16, dk=128, dv=128, T=16, threshold=64,
                     in_dtype="bf16", steps=64, layers=1, accept_law="forced",
                     gate_law="extreme", len0_law="uniform"),
    "large": Workload("large", 5, B=128, H=32, dk=128, dv=128, T=8, threshold=32,
                      in_dtype="bf16", steps=64, layers=1, accept_law="uniform",
                      gate_law="normal", len0_law="uniform"),
}

FORCED_ACCEPTS = (0, 1, 8, 15, 16)


def seed_for(wl: Workload, layer: int, step: int) -> int:
    """Seed of one (workload, layer, step); step -1 is the initial layer state."""
    return BASE_SEED + 1_000_000 * wl.cfg_id + 10_000 * layer + (step + 1)


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def _unit_rows(x: torch.Tensor) -> torch.Tensor:
    # L2-normalise the last axis in fp32 (eps 0): part of the input law.
    return x / x.norm(dim=-1, keepdim=True)


def _gates(wl: Workload, shape, gen: torch.Generator):
    g = -torch.nn.functional.softplus(torch.randn(shape, generator=gen))
    beta = torch.sigmoid(torch.randn(shape, generator=gen))
    if wl.gate_law == "extreme":
        u = torch.rand(shape, generator=gen)
        g = torch.where(u < 0.1, torch.zeros_like(g), g)
        g = torch.where((u >= 0.1) & (u < 0.2), torch.full_like(g, -20.0), g)
        w = torch.rand(shape, generator=gen)
        beta = torch.where(w < 0.1, torch.full_like(beta, 1e-4), beta)
        beta = torch.where((w >= 0.1) & (w < 0.2), torch.full_like(beta, 1.0 - 1e-4), beta)
    return g.float().contiguous(), beta.float().contiguous()


def _tokens(wl: Workload, lead, gen: torch.Generator):
    """k, v, g, beta (and q) for a block of tokens with leading shape ``lead``."""
    dt = wl.torch_in_dtype
    q = _unit_rows(torch.randn(*lead, wl.dk, generator=gen)).to(dt)
    k = _unit_rows(torch.randn(*lead, wl.dk, generator=gen)).to(dt)
    v = torch.randn(*lead, wl.dv, generator=gen).to(dt)
    g, beta = _gates(wl, tuple(lead), gen)
    return q.contiguous(), k.contiguous(), v.contiguous(), g, beta


def initial_layer(wl: Workload, layer: int = 0, B: int | None = None):
    """Checkpoint state, slot map and a pre-filled committed buffer for one layer.

    Returns a dict of CPU tensors:
      state    fp32  [n_slot, H, dv, dk]
      state_idx int32 [B]            (a seeded permutation of distinct slots)
      buf_k    in_dtype [n_slot, H, cap, dk]
      buf_v    in_dtype [n_slot, H, cap, dv]
      buf_g, buf_beta fp32 [n_slot, H, cap]
      buf_len  int32 [n_slot]       (unused slots hold length 0)
    ``B`` may shrink the batch for a bounded sample of a larger workload.
    """
    B = wl.B if B is None else B
    n_slot = B + max(1, B // 4)
    gen = _gen(seed_for(wl, layer, -1))
    state = (0.1 * torch.randn(n_slot, wl.H, wl.dv, wl.dk, generator=gen)).float().contiguous()
    state_idx = torch.randperm(n_slot, generator=gen)[:B].to(torch.int32).contiguous()
    cap = wl.cap
    _, k, v, g, beta = _tokens(wl, (n_slot, wl.H, cap), gen)
    if wl.len0_law == "fixed3":
        lens = torch.full((n_slot,), 3, dtype=torch.int32)
    else:
        lens = torch.randint(0, wl.threshold, (n_slot,), generator=gen, dtype=torch.int32)
    used = torch.zeros(n_slot, dtype=torch.bool)
    used[state_idx.long()] = True
    lens = torch.where(used, lens, torch.zeros_like(lens)).contiguous()
    return dict(state=state, state_idx=state_idx, buf_k=k, buf_v=v,
                buf_g=g, buf_beta=beta, buf_len=lens)


def accepted_counts(wl: Workload, layer: int, step: int, B: int | None = None,
                    gen: torch.Generator | None = None) -> torch.Tensor:
    B = wl.B if B is None else B
    if wl.accept_law == "forced":
        return torch.tensor([FORCED_ACCEPTS[(b + step) % len(FORCED_ACCEPTS)] for b in range(B)],
                            dtype=torch.int32)
    gen = gen if gen is not None else _gen(seed_for(wl, layer, step) ^ 0x5A5A)
    if wl.accept_law == "uniform":
        return torch.randint(0, wl.T + 1, (B,), generator=gen, dtype=torch.int32)
    # geometric with mean 12 on {1, 2, ...} (success probability 1/12), capped at T
    u = torch.rand(B, generator=gen, dtype=torch.float64)
    geo = torch.floor(torch.log1p(-u) / math.log1p(-1.0 / 12.0)) + 1
    return torch.clamp(geo, max=wl.T).to(torch.int32)


def draft_block(wl: Workload, layer: int, step: int, B: int | None = None):
    """Draft inputs of one step plus the accepted count per sequence.

    Returns a dict of CPU tensors:
      q, k   in_dtype [B, T, H, dk]
      v      in_dtype [B, T, H, dv]
      g, beta fp32    [B, T, H]
      accepted int32  [B]
    """
    B = wl.B if B is None else B
    gen = _gen(seed_for(wl, layer, step))
    q, k, v, g, beta = _tokens(wl, (B, wl.T, wl.H), gen)
    acc = accepted_counts(wl, layer, step, B)
    return dict(q=q, k=k, v=v, g=g, beta=beta, accepted=acc)
