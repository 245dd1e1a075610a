"""Full-history KV cache and the per-unit KV-slice append (plain copy).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The performer appends each KV slice it receives to its own full-history cache
before it runs the solver for the next unit ("全双工语音模型精读⑫：Wan-Streamer"
(alwayszhang.cn), 四、推理, steps 2-3; "阿里通义万相发布亚秒级同步AI视频通话基础模型"
(youleyou.com), 3.3 -- both ends share one KV-cache context).

Layouts: a slice is token-major ``[n, H, D]`` (as a projection emits it); the
cache is head-major ``[H, capacity, D]``.  The append is a bit copy:
    cache[h, cache_len + t, :] = slice[t, h, :]
for 0 <= t < n and every head h.  Nothing else in the cache changes.
"""
from __future__ import annotations

import numpy as np


def kv_append(k_cache, v_cache, k_new, v_new, cache_len: int):
    """Return copies of both caches with the slice written at ``cache_len``."""
    k_cache = np.array(k_cache, copy=True)
    v_cache = np.array(v_cache, copy=True)
    n, H, D = np.shape(k_new)
    if np.shape(v_new) != (n, H, D):
        raise ValueError("K and V slices differ in shape")
    if k_cache.shape[0] != H or k_cache.shape[2] != D:
        raise ValueError("cache shape does not match the slice")
    if cache_len < 0 or cache_len + n > k_cache.shape[1]:
        raise ValueError("append past capacity")
    for t in range(n):
        k_cache[:, cache_len + t, :] = np.asarray(k_new)[t]
        v_cache[:, cache_len + t, :] = np.asarray(v_new)[t]
    return k_cache, v_cache
