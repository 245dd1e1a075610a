"""Seeded synthetic inputs and the workload table.

This module holds no arithmetic of the method itself: it draws random
tensors, lays out per-unit token counts and turns them into block offsets.
Both the CUDA path's tests/benchmark and the CPU oracle take their inputs
from here, so the two see the same bytes.

Recipe
------
* Every tensor comes from its own ``torch.Generator('cpu')`` seeded with a
  64-bit value derived (SHA-256) from (workload seed, tensor name, index).
  Attention tensors (Q, K, V) are drawn per (head, unit), so any head or
  unit can be regenerated on its own, and a unit appended later holds the
  same keys a full-sequence prefill over the same timeline sees.
* Values are N(0, 1) * std in fp32 on the host, then rounded once to the
  workload dtype (round-to-nearest-even for bf16).  The rounded values are
  what both sides consume.
* Text tokens per unit (640x368 units) are uniform on 0..16 from the
  generator named "text".
* A streaming unit is one block: video-latent tokens, then audio, then text
  (the order only fixes which rows are latents; inside a block attention is
  bidirectional).
"""
from __future__ import annotations

import dataclasses
import hashlib
from typing import Optional

import numpy as np
import torch


def sub_seed(seed: int, name: str, index: int = 0) -> int:
    digest = hashlib.sha256(f"{seed}/{name}/{index}".encode()).digest()
    return int.from_bytes(digest[:8], "little") & ((1 << 63) - 1)


def generator(seed: int, name: str, index: int = 0) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(sub_seed(seed, name, index))
    return g


def normal(seed: int, name: str, index: int, shape, std: float = 1.0,
           dtype: torch.dtype = torch.float32) -> torch.Tensor:
    """N(0,1)*std drawn in fp32 on the host, rounded once to ``dtype``."""
    x = torch.randn(*shape, generator=generator(seed, name, index), dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def block_offsets(sizes) -> np.ndarray:
    """int32 offsets [n_blocks + 1]: 0, s0, s0+s1, ..."""
    out = np.zeros(len(sizes) + 1, dtype=np.int64)
    np.cumsum(np.asarray(sizes, dtype=np.int64), out=out[1:])
    if out[-1] > np.iinfo(np.int32).max:
        raise ValueError("too many tokens for int32 offsets")
    return out.astype(np.int32)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    heads: int
    head_dim: int
    dtype: str                   # "bf16" or "f32"
    std: float                   # std of Q/K/V entries
    video_tokens: int            # per unit
    audio_tokens: int            # per unit
    text_tokens: Optional[int]   # fixed per unit, or None for uniform 0..16
    history_units: int           # units already in the cache
    new_units: int               # units streamed (attention + append + Euler each)
    latent_tokens: int           # latent rows the Euler step updates per unit
    latent_channels: int
    euler_steps: int
    prefill: bool = False        # True: one full-sequence block-causal prefill

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    @property
    def n_units(self) -> int:
        return self.history_units + self.new_units

    def unit_sizes(self) -> list:
        n = self.n_units
        if self.text_tokens is None:
            text = torch.randint(0, 17, (n,), generator=generator(self.seed, "text")).tolist()
        else:
            text = [self.text_tokens] * n
        return [self.video_tokens + self.audio_tokens + t for t in text]

    def offsets(self) -> np.ndarray:
        return block_offsets(self.unit_sizes())

    def capacity(self) -> int:
        """Cache rows to allocate: every unit at its largest size."""
        most = self.video_tokens + self.audio_tokens + (16 if self.text_tokens is None else self.text_tokens)
        return self.n_units * most

    # Timeline tensors, one (head, unit) at a time -------------------------
    def unit_tensor(self, name: str, h: int, u: int, sizes=None) -> torch.Tensor:
        """Rows of tensor ``name`` ("q", "k" or "v") for head h, unit u: [n_u, D]."""
        n = (sizes if sizes is not None else self.unit_sizes())[u]
        return normal(self.seed, name, h * 1_000_000 + u, (n, self.head_dim), self.std, self.torch_dtype)

    def head_timeline(self, name: str, h: int, n_units: int, sizes=None) -> torch.Tensor:
        """Tensor ``name`` for head h over units 0..n_units-1: [T, D]."""
        sizes = sizes if sizes is not None else self.unit_sizes()
        parts = [self.unit_tensor(name, h, u, sizes) for u in range(n_units)]
        if not parts:
            return torch.empty(0, self.head_dim, dtype=self.torch_dtype)
        return torch.cat(parts, dim=0)

    def token_major(self, name: str, u: int, sizes=None) -> torch.Tensor:
        """Tensor ``name`` for unit u, all heads, token-major [n_u, H, D]."""
        sizes = sizes if sizes is not None else self.unit_sizes()
        out = torch.empty(sizes[u], self.heads, self.head_dim, dtype=self.torch_dtype)
        for h in range(self.heads):
            out[:, h, :] = self.unit_tensor(name, h, u, sizes)
        return out

    def token_major_range(self, name: str, u0: int, u1: int, sizes=None) -> torch.Tensor:
        """Units u0..u1-1 concatenated, token-major [n, H, D]."""
        sizes = sizes if sizes is not None else self.unit_sizes()
        return torch.cat([self.token_major(name, u, sizes) for u in range(u0, u1)], dim=0)

    # Flow-matching latents ------------------------------------------------
    def latent_shape(self):
        return (self.latent_tokens, self.latent_channels)

    def z0(self, unit: int) -> torch.Tensor:
        return normal(self.seed, "z0", unit, self.latent_shape(), 1.0, torch.float32)

    def eps(self, unit: int) -> torch.Tensor:
        return normal(self.seed, "eps", unit, self.latent_shape(), 1.0, torch.float32)

    def velocity_input(self, unit: int, step: int) -> torch.Tensor:
        """Stand-in for the velocity network's output at one solver step."""
        vdt = torch.float32 if self.dtype == "f32" else torch.bfloat16
        return normal(self.seed, "vel", unit * 64 + step, self.latent_shape(), 1.0, vdt)


WORKLOADS = {
    # 1 head, D 64, fp32, 8 blocks of 16 tokens; prefill + per-block
    # incremental attention; one Euler step on a 16 x 64 latent.
    "tiny_fp32": Workload("tiny_fp32", seed=0, heads=1, head_dim=64, dtype="f32", std=1.0,
                          video_tokens=16, audio_tokens=0, text_tokens=0,
                          history_units=7, new_units=1, latent_tokens=16,
                          latent_channels=64, euler_steps=1),
    # 192x336: 12x21 video latents + 8 audio + 4 text = 264 tokens per unit,
    # 32 history units, 24 heads; Euler over 260 x 3072 latents.
    "unit_192x336": Workload("unit_192x336", seed=1, heads=24, head_dim=128, dtype="bf16", std=0.5,
                             video_tokens=252, audio_tokens=8, text_tokens=4,
                             history_units=32, new_units=1, latent_tokens=260,
                             latent_channels=3072, euler_steps=4),
    # 640x368: 40x23 video latents + 8 audio + 0..16 text, 64 history units,
    # 40 heads; Euler over 928 x 5120 latents.
    "unit_640x368": Workload("unit_640x368", seed=2, heads=40, head_dim=128, dtype="bf16", std=0.5,
                             video_tokens=920, audio_tokens=8, text_tokens=None,
                             history_units=64, new_units=1, latent_tokens=928,
                             latent_channels=5120, euler_steps=4),
    # Full-sequence prefill: 128 units x 932 tokens, 40 heads.
    "prefill_128x932": Workload("prefill_128x932", seed=3, heads=40, head_dim=128, dtype="bf16", std=0.5,
                                video_tokens=920, audio_tokens=8, text_tokens=4,
                                history_units=0, new_units=128, latent_tokens=928,
                                latent_channels=5120, euler_steps=0, prefill=True),
    # Long session: 512 history units (~477k tokens), then 16 units streamed.
    "long_session_640x368": Workload("long_session_640x368", seed=4, heads=40, head_dim=128, dtype="bf16",
                                     std=0.5, video_tokens=920, audio_tokens=8, text_tokens=None,
                                     history_units=512, new_units=16, latent_tokens=928,
                                     latent_channels=5120, euler_steps=4),
}
