"""Workload shapes and seeded input draws for the GLA forward and decode step.

Recipe (the same for every workload, only sizes and spreads differ):

* one ``torch.Generator`` seeded with ``seed`` (0 by default), on the device
  the tensors are made on;
* draw order: z, q, k, v, then h0 (when the workload has one);
* ``z ~ N(0, sigma_z^2)`` in fp32, and ``log_alpha = logsigmoid(z) / tau`` in
  fp32, i.e. the forget gate alpha = sigmoid(z)^(1/tau) lies in (0, 1);
* q, k, v ~ N(0, 1) drawn in fp32 and rounded to bf16;
* h0 ~ N(0, sigma_h^2) in fp32 when present, else no initial state (zero).

Layouts are head-first and contiguous: q, k, log_alpha ``[B, H, T, dk]``,
v ``[B, H, T, dv]``, h0 ``[B, H, dk, dv]`` (row index = key channel).

The backward of a chunked workload also draws the upstream gradients, from a
second generator seeded with ``seed + 1``: d_o ~ N(0, 1) in bf16
``[B, H, T, dv]``, then dhT ~ N(0, sigma_dhT^2) in fp32 ``[B, H, dk, dv]``
when the final state has a gradient.

For the decode workload the per-step tensors carry a leading step axis:
``[steps, B, H, dk]`` etc., and h0 is drawn before them.
"""

from __future__ import annotations

from dataclasses import dataclass

import torch
import torch.nn.functional as F


@dataclass(frozen=True)
class ChunkConfig:
    name: str
    B: int
    H: int
    T: int
    dk: int
    dv: int
    sigma_z: float = 1.0
    tau: float = 16.0
    sigma_h0: float | None = None  # None: no initial state

    @property
    def tokens(self) -> int:
        return self.B * self.H * self.T

    @property
    def scale(self) -> float:
        return self.dk ** -0.5


@dataclass(frozen=True)
class DecodeConfig:
    name: str
    B: int
    H: int
    dk: int
    dv: int
    steps: int
    check_every: int
    sigma_z: float = 1.0
    tau: float = 16.0
    sigma_h0: float = 0.1

    @property
    def scale(self) -> float:
        return self.dk ** -0.5


# The five workloads: four chunked forwards and one decode loop.
CHUNK_CONFIGS = {
    "small": ChunkConfig("B1-H2-T256-dk64-dv64", 1, 2, 256, 64, 64),
    "medium": ChunkConfig("B8-H16-T2048-dk128-dv128", 8, 16, 2048, 128, 128),
    "long": ChunkConfig("B2-H16-T32768-dk128-dv256", 2, 16, 32768, 128, 256,
                        sigma_z=2.0, sigma_h0=0.1),
    "very_long": ChunkConfig("B1-H32-T262144-dk128-dv128", 1, 32, 262144, 128, 128,
                             tau=32.0),
}
DECODE_CONFIG = DecodeConfig("decode-B256-H32-dk128-dv128-1024steps", 256, 32, 128, 128,
                             steps=1024, check_every=128)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_chunk_inputs(B: int, H: int, T: int, dk: int, dv: int, *, sigma_z: float = 1.0,
                      tau: float = 16.0, sigma_h0: float | None = None, seed: int = 0,
                      device="cpu"):
    """Draw (q, k, v, log_alpha, h0) for one chunked-forward workload.

    Returns bf16 q, k, v; fp32 log_alpha; fp32 h0 or None.
    """
    g = _gen(seed, device)
    z = torch.randn(B, H, T, dk, generator=g, device=device, dtype=torch.float32)
    if sigma_z != 1.0:
        z.mul_(sigma_z)
    q = torch.randn(B, H, T, dk, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    k = torch.randn(B, H, T, dk, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    v = torch.randn(B, H, T, dv, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    log_alpha = F.logsigmoid(z).div_(tau)
    del z
    h0 = None
    if sigma_h0 is not None:
        h0 = torch.randn(B, H, dk, dv, generator=g, device=device, dtype=torch.float32).mul_(sigma_h0)
    return q, k, v, log_alpha, h0


def make_config_inputs(cfg: ChunkConfig, seed: int = 0, device="cpu"):
    return make_chunk_inputs(cfg.B, cfg.H, cfg.T, cfg.dk, cfg.dv, sigma_z=cfg.sigma_z,
                             tau=cfg.tau, sigma_h0=cfg.sigma_h0, seed=seed, device=device)


def make_backward_grads(B: int, H: int, T: int, dk: int, dv: int, *,
                        sigma_dhT: float | None = None, seed: int = 0, device="cpu"):
    """Draw the upstream gradients (d_o bf16, dhT fp32 or None) of one backward call."""
    g = _gen(seed + 1, device)
    d_o = torch.randn(B, H, T, dv, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    dhT = None
    if sigma_dhT is not None:
        dhT = torch.randn(B, H, dk, dv, generator=g, device=device, dtype=torch.float32).mul_(sigma_dhT)
    return d_o, dhT


def make_decode_inputs(B: int, H: int, dk: int, dv: int, steps: int, *, sigma_z: float = 1.0,
                       tau: float = 16.0, sigma_h0: float = 0.1, seed: int = 0, device="cpu"):
    """Draw h0 and the per-step (q, k, v, log_alpha) of a decode loop.

    Returns h0 fp32 [B,H,dk,dv] and per-step tensors with a leading step axis.
    """
    g = _gen(seed, device)
    h0 = torch.randn(B, H, dk, dv, generator=g, device=device, dtype=torch.float32).mul_(sigma_h0)
    z = torch.randn(steps, B, H, dk, generator=g, device=device, dtype=torch.float32)
    if sigma_z != 1.0:
        z.mul_(sigma_z)
    q = torch.randn(steps, B, H, dk, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    k = torch.randn(steps, B, H, dk, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    v = torch.randn(steps, B, H, dv, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    log_alpha = F.logsigmoid(z).div_(tau)
    del z
    return h0, q, k, v, log_alpha


def make_gdn_inputs(B: int, H: int, T: int, dk: int, dv: int, *, sigma_z: float = 1.0,
                    tau: float = 16.0, sigma_h0: float | None = None, seed: int = 0,
                    device="cpu"):
    """Draw (q, k, v, g, beta, h0) for the gated delta rule: one generator seeded
    with ``seed``; draw order z, z_beta, q, k, v, h0; g = logsigmoid(z) / tau
    [B,H,T] fp32; beta = sigmoid(z_beta) [B,H,T] fp32; q, v ~ N(0, 1) and k ~ N(0, 1)
    normalised to unit L2 norm per token, all rounded to bf16; h0 ~ N(0, sigma_h0^2)."""
    gen = _gen(seed, device)
    z = torch.randn(B, H, T, generator=gen, device=device, dtype=torch.float32)
    if sigma_z != 1.0:
        z.mul_(sigma_z)
    zb = torch.randn(B, H, T, generator=gen, device=device, dtype=torch.float32)
    q = torch.randn(B, H, T, dk, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)
    k = torch.randn(B, H, T, dk, generator=gen, device=device, dtype=torch.float32)
    k = (k / k.norm(dim=-1, keepdim=True)).to(torch.bfloat16)
    v = torch.randn(B, H, T, dv, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)
    g = F.logsigmoid(z).div_(tau)
    beta = torch.sigmoid(zb)
    h0 = None
    if sigma_h0 is not None:
        h0 = torch.randn(B, H, dk, dv, generator=gen, device=device, dtype=torch.float32).mul_(sigma_h0)
    return q, k, v, g, beta, h0

