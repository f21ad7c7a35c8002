"""Seeded inputs for the two GDN layer steps either side of the recurrence: the
causal convolution (ring of committed pre-convolution inputs, write positions,
draft blocks, accepted counts, weights) and the gated RMSNorm + FP8 quantisation
(GDN outputs, gates, norm weight).  Nothing here computes any part of either step.

Shapes follow the decode-loop sweep: the convolution covers q, k and v of every
head side by side (D = H (2 d_k + d_v) = 16 * 384 = 6144 channels), width 4, the
draft block of 16 tokens; the norm runs over the [B, T, H, d_v] outputs of the
verify (rows of d_v = 128).  Draws use torch.Generator on the CPU.
"""
from __future__ import annotations

import dataclasses

import torch

from .workloads import FORCED_ACCEPTS, WORKLOADS, accepted_counts

BASE_SEED = 20261203


@dataclasses.dataclass(frozen=True)
class ConvWorkload:
    name: str
    cfg_id: int
    B: int
    D: int
    W: int
    T: int
    cap: int
    act: int               # 0 identity, 1 SiLU
    in_dtype: str          # "bf16" or "fp32"
    out_dtype: str
    accept_law: str        # "geometric12", "uniform" or "forced"

    @property
    def n_slot(self) -> int:
        return self.B + max(1, self.B // 4)

    def torch_dtype(self, which: str) -> torch.dtype:
        return torch.bfloat16 if getattr(self, which) == "bf16" else torch.float32


CONV_WORKLOADS = {
    # the decode-loop sweep's layer: B=32, H=16 heads x (q, k, v) = 6144 channels
    "conv_decode": ConvWorkload("conv_decode", 11, B=32, D=6144, W=4, T=16, cap=32, act=1,
                                in_dtype="bf16", out_dtype="bf16", accept_law="geometric12"),
    # the tightest ring (cap = W - 1 + T) and the forced accepted counts {0, 1, 8, 15, 16}
    "conv_edge": ConvWorkload("conv_edge", 12, B=12, D=6144, W=4, T=16, cap=19, act=1,
                              in_dtype="bf16", out_dtype="fp32", accept_law="forced"),
    # narrower kernels, fp32 inputs, ragged grid (D not a multiple of the CTA's 1024 channels)
    "conv_w3_f32": ConvWorkload("conv_w3_f32", 13, B=5, D=200, W=3, T=7, cap=12, act=0,
                                in_dtype="fp32", out_dtype="fp32", accept_law="uniform"),
    "conv_w2_bf16": ConvWorkload("conv_w2_bf16", 14, B=3, D=136, W=2, T=1, cap=2, act=1,
                                 in_dtype="bf16", out_dtype="bf16", accept_law="uniform"),
    "conv_w1": ConvWorkload("conv_w1", 15, B=2, D=64, W=1, T=5, cap=5, act=1,
                            in_dtype="bf16", out_dtype="fp32", accept_law="uniform"),
}


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def conv_seed(wl: ConvWorkload, layer: int, step: int) -> int:
    return BASE_SEED + 1_000_000 * wl.cfg_id + 10_000 * layer + (step + 1)


def initial_conv_layer(wl: ConvWorkload, layer: int = 0):
    """Ring of committed inputs (N(0, 1)), write positions U[0, cap), a seeded slot
    permutation, weights N(0, 1/W) and bias N(0, 0.1^2).  CPU tensors:
      ring [n_slot, cap, D] in_dtype, pos int32 [n_slot], state_idx int32 [B],
      weight fp32 [D, W], bias fp32 [D]."""
    g = _gen(conv_seed(wl, layer, -1))
    n = wl.n_slot
    ring = torch.randn(n, wl.cap, wl.D, generator=g).to(wl.torch_dtype("in_dtype")).contiguous()
    pos = torch.randint(0, wl.cap, (n,), generator=g, dtype=torch.int32)
    state_idx = torch.randperm(n, generator=g)[:wl.B].to(torch.int32).contiguous()
    weight = (torch.randn(wl.D, wl.W, generator=g) / wl.W ** 0.5).float().contiguous()
    bias = (0.1 * torch.randn(wl.D, generator=g)).float().contiguous()
    return dict(ring=ring, pos=pos, state_idx=state_idx, weight=weight, bias=bias)


def conv_block(wl: ConvWorkload, layer: int, step: int):
    """Draft inputs x [B, T, D] (N(0, 1), in_dtype) and accepted counts int32 [B]."""
    g = _gen(conv_seed(wl, layer, step))
    x = torch.randn(wl.B, wl.T, wl.D, generator=g).to(wl.torch_dtype("in_dtype")).contiguous()
    if wl.accept_law == "forced":
        acc = torch.tensor([FORCED_ACCEPTS[(b + step) % len(FORCED_ACCEPTS)] for b in range(wl.B)],
                           dtype=torch.int32)
        acc = torch.clamp(acc, max=wl.T)
    elif wl.accept_law == "uniform":
        acc = torch.randint(0, wl.T + 1, (wl.B,), generator=g, dtype=torch.int32)
    else:
        dec = WORKLOADS["decode24"]
        acc = torch.clamp(accepted_counts(dec, layer, step, B=wl.B), max=wl.T)
    return dict(x=x, accepted=acc)


@dataclasses.dataclass(frozen=True)
class NormWorkload:
    name: str
    cfg_id: int
    rows: int
    d: int
    z_dtype: str
    eps: float
    inv_scale: float


NORM_WORKLOADS = {
    # the verify outputs of one decode24 layer-step: B*T*H = 32*16*16 rows of d_v = 128
    "norm_decode": NormWorkload("norm_decode", 21, rows=8192, d=128, z_dtype="bf16", eps=1e-6,
                                inv_scale=64.0),
    "norm_d64_f32": NormWorkload("norm_d64_f32", 22, rows=333, d=64, z_dtype="fp32", eps=1e-5,
                                 inv_scale=200.0),
    "norm_d256": NormWorkload("norm_d256", 23, rows=77, d=256, z_dtype="bf16", eps=1e-6,
                              inv_scale=90.0),
}


def norm_inputs(wl: NormWorkload, seed_offset: int = 0):
    """o fp32 [rows, d] with per-row scales spread over 2^-8 .. 2^8 (the norm removes
    them), gate z N(0, 2^2) in z_dtype, weight fp32 1 + N(0, 0.1^2)."""
    g = _gen(BASE_SEED + 1_000_000 * wl.cfg_id + seed_offset)
    scale = torch.exp2(torch.empty(wl.rows, 1).uniform_(-8, 8, generator=g))
    o = (torch.randn(wl.rows, wl.d, generator=g) * scale).float().contiguous()
    zt = torch.bfloat16 if wl.z_dtype == "bf16" else torch.float32
    z = (2.0 * torch.randn(wl.rows, wl.d, generator=g)).to(zt).contiguous()
    w = (1.0 + 0.1 * torch.randn(wl.d, generator=g)).float().contiguous()
    return dict(o=o, z=z, weight=w)
