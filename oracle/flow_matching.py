"""Conditional flow matching: interpolant, velocity and the Euler update.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

"全双工语音模型精读⑫：Wan-Streamer" (alwayszhang.cn), section 3.2 (混合生成目标),
defines for each continuous modality m (audio, video)
    z_tau = (1 - tau) z_0 + tau * eps,      dz_tau/dtau = eps - z_0,
with tau = 1 pure noise and tau = 0 the clean latent.  The performer runs a
flow-matching solver over these latents ("阿里通义万相发布亚秒级同步AI视频通话基础模型"
(youleyou.com), 3.3).  The solver, its grid and its step count are not
published (same page 七、局限 4); the reading taken here is the plain Euler
method on a uniform grid from tau = 1 down to tau = 0:
    z_{tau - dtau} = z_tau - dtau * v(z_tau, tau).
All arithmetic is fp64; callers round once to their own dtype to compare.

Classifier-free guidance: the same page (五、训练, item 3) says the
low-latency student is distilled from a teacher that samples with CFG and
more solver steps.  The pages give no formula; the reading taken here is the
standard guidance combination applied to the velocity,
    v = v_uncond + w * (v_cond - v_uncond),
followed by the same Euler update.  w = 0 gives the unconditional velocity,
w = 1 the conditional one.
"""
from __future__ import annotations

import numpy as np


def interpolant(z0, eps, tau: float):
    """z_tau = (1 - tau) z_0 + tau eps."""
    z0 = np.asarray(z0, dtype=np.float64)
    eps = np.asarray(eps, dtype=np.float64)
    return (1.0 - tau) * z0 + tau * eps


def velocity(z0, eps):
    """dz_tau / dtau = eps - z_0 (constant along the straight path)."""
    return np.asarray(eps, dtype=np.float64) - np.asarray(z0, dtype=np.float64)


def euler_step(z, v, dtau: float):
    """One Euler step towards tau = 0: z - dtau * v."""
    return np.asarray(z, dtype=np.float64) - float(dtau) * np.asarray(v, dtype=np.float64)


def uniform_grid(n_steps: int):
    """tau_0 = 1 > tau_1 > ... > tau_n = 0, equally spaced."""
    if n_steps < 1:
        raise ValueError("need at least one step")
    return np.linspace(1.0, 0.0, n_steps + 1)


def euler_solve(z1, velocity_fn, n_steps: int):
    """Integrate from tau = 1 to 0; velocity_fn(z, tau) gives v at (z, tau)."""
    z = np.asarray(z1, dtype=np.float64)
    grid = uniform_grid(n_steps)
    for a, b in zip(grid[:-1], grid[1:]):
        z = euler_step(z, velocity_fn(z, a), a - b)
    return z


def cfg_velocity(v_uncond, v_cond, w: float):
    """Guided velocity v_uncond + w * (v_cond - v_uncond)."""
    vu = np.asarray(v_uncond, dtype=np.float64)
    vc = np.asarray(v_cond, dtype=np.float64)
    return vu + float(w) * (vc - vu)


def cfg_euler_step(z, v_uncond, v_cond, w: float, dtau: float):
    """One Euler step with the guided velocity: z - dtau * cfg_velocity."""
    return euler_step(z, cfg_velocity(v_uncond, v_cond, w), dtau)
