"""Shared helpers for the GPU parity tests: build seeded cases on the host,
move them to the device, run the oracle on the same bytes, compare."""
from __future__ import annotations

import numpy as np
import torch

from oracle import block_causal as bc
from streaming_block_causal_flash_b300.inputs import Workload, block_offsets

BF16_REL = 1e-2          # bf16 path: max|gpu - ref| <= 1e-2 * max|ref|
F32_ABS = 1e-5           # fp32 path: max|gpu - ref| <= 1e-5
LSE_REL = 1e-4           # LSE: |gpu - ref| <= 1e-4 * max(1, |ref|)


def custom_workload(seed, heads, head_dim, dtype="bf16", std=0.5):
    return Workload(name="case", seed=seed, heads=heads, head_dim=head_dim, dtype=dtype, std=std,
                    video_tokens=0, audio_tokens=0, text_tokens=0, history_units=0, new_units=0,
                    latent_tokens=1, latent_channels=8, euler_steps=0)


class Case:
    """A token timeline cut into blocks, its Q/K/V on the host and the device."""

    def __init__(self, w: Workload, sizes, n_units=None, cap_extra=0, device="cuda",
                 q_units=None, canary=None):
        self.w = w
        self.sizes = list(sizes)
        n_units = len(self.sizes) if n_units is None else n_units
        self.offsets = block_offsets(self.sizes[:n_units])
        self.T = int(self.offsets[-1])
        self.cap = self.T + cap_extra
        H, D, dt = w.heads, w.head_dim, w.torch_dtype
        fill = 0.0 if canary is None else canary
        self.k_host = torch.full((H, self.cap, D), fill, dtype=dt)
        self.v_host = torch.full((H, self.cap, D), fill, dtype=dt)
        for h in range(H):
            self.k_host[h, :self.T] = w.head_timeline("k", h, n_units, self.sizes)
            self.v_host[h, :self.T] = w.head_timeline("v", h, n_units, self.sizes)
        q_units = range(n_units) if q_units is None else q_units
        self.q_units = list(q_units)
        self.q_host = torch.cat([w.token_major("q", u, self.sizes) for u in self.q_units], 0) \
            if self.q_units else torch.empty(0, H, D, dtype=dt)
        self.device = device
        self.k = self.k_host.to(device)
        self.v = self.v_host.to(device)
        self.q = self.q_host.to(device)
        self.offs_dev = torch.from_numpy(self.offsets.astype(np.int32)).to(device)

    def q_rows_global(self):
        rows = []
        for u in self.q_units:
            rows += list(range(int(self.offsets[u]), int(self.offsets[u + 1])))
        return np.array(rows, dtype=np.int64)

    def oracle(self, row_sel=None, scale=None):
        """Oracle output/lse for query rows (indices into q) or all of them."""
        rows = self.q_rows_global()
        sel = np.arange(rows.size) if row_sel is None else np.asarray(row_sel)
        q = self.q_host[sel].float().numpy()
        out, lse = bc.attention_rows(q, rows[sel], self.k_host.float().numpy(),
                                     self.v_host.float().numpy(), self.offsets, scale)
        return sel, out, lse


def assert_close_bf16(gpu, ref, what=""):
    gpu = np.asarray(gpu, dtype=np.float64)
    bound = BF16_REL * np.abs(ref).max()
    err = np.abs(gpu - ref).max()
    assert np.isfinite(gpu).all(), f"{what}: non-finite output"
    assert err <= bound, f"{what}: max err {err:.3e} > {bound:.3e} (max|ref| {np.abs(ref).max():.3e})"
    return err, bound


def assert_close_abs(gpu, ref, tol, what=""):
    gpu = np.asarray(gpu, dtype=np.float64)
    err = np.abs(gpu - ref).max()
    assert np.isfinite(gpu).all(), f"{what}: non-finite output"
    assert err <= tol, f"{what}: max err {err:.3e} > {tol:.3e}"
    return err


def assert_lse(gpu, ref, what=""):
    gpu = np.asarray(gpu, dtype=np.float64)
    err = (np.abs(gpu - ref) / np.maximum(1.0, np.abs(ref))).max()
    assert err <= LSE_REL, f"{what}: LSE rel err {err:.3e}"
