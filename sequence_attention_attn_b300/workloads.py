"""Seeded synthetic workloads for the DiT attention path.

This module only draws inputs: it holds the workload shapes and the seeded
random recipes, and none of the method's arithmetic.  Both the GPU path and the
CPU oracle are fed from it, so the same bf16 bits reach both sides.

Shapes follow the DiT families the pages speak of (image latents cut into 2x2
patches, MM-DiT joint text+image attention, video latents):

* ``tiny``          B=1, H=2,  S=256,   D=64,  Q/K/V ~ N(0,1)
* ``dit_xl2_512``   B=2, H=16, S=1024,  D=72,  Q/K/V ~ N(0,1) * 1/sqrt(72)
  (64x64 latent, 2x2 patches; B=2 is the cond/uncond pair of guidance)
* ``pixart_1024``   B=2, H=16, S=4096,  D=72,  Q/K/V ~ N(0,1) (128x128 latent)
* ``flux_mmdit``    B=1, H=24, S=4608,  D=128, 512 text tokens first (Q/K std 2),
  then 4096 image tokens (Q/K std 1); V std 1 everywhere
* ``video``         B=1, H=48, S=17550, D=64,  Q/K/V ~ N(0,1)
  (13 latent frames of 60x90, 2x2 patches)

Recipe: ``torch.Generator('cpu').manual_seed(seed)``; fp32 ``randn`` for Q,
then K, then V, each [B, H, S, D]; scale; round to bf16 (round-to-nearest-even,
torch's cast).  Default seed = 20261202 + the workload's index in ``CONFIGS``.
"""
from __future__ import annotations

import dataclasses
import math

import torch

SEED_BASE = 20261202


@dataclasses.dataclass(frozen=True)
class AttnConfig:
    name: str
    index: int
    B: int
    H: int
    S: int
    D: int
    chunk_counts: tuple
    text_tokens: int = 0          # leading text tokens (joint attention)
    text_qk_std: float = 1.0
    qkv_scale: float = 1.0        # multiplies N(0,1) before the bf16 cast
    cfg_shape: tuple | None = None  # (eps_c, eps_u) shape for the CFG combine
    cfg_w: float = 4.5
    merge_n: int | None = None    # partial count for the standalone merge

    @property
    def flops(self) -> float:
        """Algorithmic flops of one forward: 4 B H S^2 D (QK^T and PV)."""
        return 4.0 * self.B * self.H * self.S * self.S * self.D

    @property
    def rows(self) -> int:
        return self.B * self.H * self.S


CONFIGS = [
    AttnConfig("tiny", 0, 1, 2, 256, 64, (1, 2, 4), cfg_shape=(4, 32, 32)),
    AttnConfig("dit_xl2_512", 1, 2, 16, 1024, 72, (1, 2, 4, 8),
               qkv_scale=1.0 / math.sqrt(72.0)),
    AttnConfig("pixart_1024", 2, 2, 16, 4096, 72, (1, 4, 8), cfg_shape=(4, 128, 128)),
    AttnConfig("flux_mmdit", 3, 1, 24, 4608, 128, (1, 2, 4, 8), text_tokens=512,
               text_qk_std=2.0),
    AttnConfig("video", 4, 1, 48, 17550, 64, (1, 8, 16), merge_n=16),
]
BY_NAME = {c.name: c for c in CONFIGS}


def seed_for(cfg: AttnConfig, offset: int = 0) -> int:
    return SEED_BASE + cfg.index + offset


def make_qkv(cfg: AttnConfig, seed: int | None = None, generator_device: str = "cpu"):
    """Draw (q, k, v) bf16 tensors [B, H, S, D] on ``generator_device``."""
    seed = seed_for(cfg) if seed is None else seed
    g = torch.Generator(generator_device).manual_seed(seed)
    shape = (cfg.B, cfg.H, cfg.S, cfg.D)
    out = []
    for which in ("q", "k", "v"):
        x = torch.randn(shape, generator=g, dtype=torch.float32, device=generator_device)
        if cfg.qkv_scale != 1.0:
            x.mul_(cfg.qkv_scale)
        if cfg.text_tokens and which in ("q", "k"):
            x[:, :, :cfg.text_tokens, :].mul_(cfg.text_qk_std)
        out.append(x.to(torch.bfloat16))
    return tuple(out)


def make_random_qkv(B: int, H: int, S: int, D: int, seed: int, std: float = 1.0,
                    device: str = "cpu"):
    """Free-shape variant of ``make_qkv`` for edge-case tests."""
    g = torch.Generator(device).manual_seed(seed)
    out = []
    for _ in range(3):
        x = torch.randn((B, H, S, D), generator=g, dtype=torch.float32, device=device)
        out.append((x * std).to(torch.bfloat16))
    return tuple(out)


def make_cfg(shape, seed: int, device: str = "cpu"):
    """(eps_c, eps_u): fp32 N(0,1) noise predictions of the cond/uncond paths."""
    g = torch.Generator(device).manual_seed(seed)
    eps_c = torch.randn(shape, generator=g, dtype=torch.float32, device=device)
    eps_u = torch.randn(shape, generator=g, dtype=torch.float32, device=device)
    return eps_c, eps_u


def make_merge(n: int, rows: int, D: int, seed: int, device: str = "cpu",
               neg_inf_frac: float = 0.0):
    """(partials [n, rows, D], lses [n, rows]) fp32.

    Partials ~ N(0,1); LSEs ~ 7 + 2 N(0,1) (about ln of a 1097-key chunk, with
    spread so the weights differ between chunks).  With ``neg_inf_frac`` > 0 that
    fraction of (chunk, row) LSEs is set to -inf (empty chunks)."""
    g = torch.Generator(device).manual_seed(seed)
    partials = torch.randn((n, rows, D), generator=g, dtype=torch.float32, device=device)
    lses = 7.0 + 2.0 * torch.randn((n, rows), generator=g, dtype=torch.float32, device=device)
    if neg_inf_frac > 0.0:
        mask = torch.rand((n, rows), generator=g, device=device) < neg_inf_frac
        lses = lses.masked_fill(mask, float("-inf"))
    return partials, lses
