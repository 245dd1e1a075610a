"""Block-causal softmax attention, written out from its definition in fp64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

What the method computes
------------------------
The token sequence is cut into consecutive blocks (one streaming unit of
about 160 ms each).  A token attends to every token of its own block, in both
directions, and to every token of every earlier block; it never attends to a
later block.  [Wan Streamer real-time AV explainer (xiaohu-jiedu.pages.dev),
section "怎么做到边听边说、随时能打断"; "阿里通义万相发布亚秒级同步AI视频通话基础模型"
(youleyou.com), section 3.1.]

Blocks are given by ``offsets`` (length n_blocks + 1, offsets[0] = 0,
non-decreasing); block b holds tokens offsets[b] <= i < offsets[b+1].  An
empty block (equal offsets) holds no token.

Readings taken where the pages are silent:
* softmax scale s = 1/sqrt(D) unless given;
* K/V heads equal Q heads (plain multi-head attention);
* the log-sum-exp is natural-log: LSE_i = m_i + ln(sum_j exp(x_ij - m_i)).

Layouts used here: Q rows ``[R, H, D]`` with their global token indices,
K and V caches ``[H, N, D]`` (N >= the largest visible prefix).
"""
from __future__ import annotations

import math

import numpy as np


def block_index(offsets, i: int) -> int:
    """Block b with offsets[b] <= i < offsets[b+1] (token i must exist)."""
    offs = np.asarray(offsets, dtype=np.int64)
    if not (0 <= i < offs[-1]):
        raise IndexError(f"token {i} outside [0, {offs[-1]})")
    # The last b whose start is <= i; empty blocks before it are skipped
    # because their start equals the next block's start.
    b = int(np.searchsorted(offs, i, side="right")) - 1
    assert offs[b] <= i < offs[b + 1]
    return b


def row_limit(offsets, i: int) -> int:
    """e(i): token i sees exactly the keys j < e(i) = end of its own block."""
    return int(np.asarray(offsets)[block_index(offsets, i) + 1])


def visibility_mask(offsets) -> np.ndarray:
    """Explicit N x N mask built from block membership (brute force).

    mask[i, j] is True iff block(j) <= block(i): own block both ways, every
    earlier block, no later block.  This is a second, independent statement
    of the rule that ``row_limit`` states as a prefix length.
    """
    offs = np.asarray(offsets, dtype=np.int64)
    n = int(offs[-1])
    blk = np.empty(n, dtype=np.int64)
    for b in range(len(offs) - 1):
        blk[offs[b]:offs[b + 1]] = b
    return blk[None, :] <= blk[:, None]


def default_scale(head_dim: int) -> float:
    return 1.0 / math.sqrt(head_dim)


def attention_rows(q_rows, row_ids, k_cache, v_cache, offsets, scale=None):
    """Block-causal attention for the given query rows, every head.

    q_rows  : [R, H, D] query vectors of tokens ``row_ids`` (global indices)
    k_cache : [H, N, D] keys of tokens 0..N-1, v_cache likewise
    returns (out [R, H, D] float64, lse [H, R] float64)

    For each head h and row i, with e = e(i):
        x_j  = s * <q_i, k_j>            j < e
        m    = max_j x_j
        l    = sum_j exp(x_j - m)
        O_i  = sum_j exp(x_j - m) v_j / l
        LSE  = m + ln l
    Two passes over the logits (max, then sums).  Rows that share the same
    limit e are evaluated together with one matrix product per head; nothing
    else is blocked or reordered.
    """
    q = np.asarray(q_rows, dtype=np.float64)
    k = np.asarray(k_cache)       # converted to fp64 one head at a time
    v = np.asarray(v_cache)
    rows = np.asarray(row_ids, dtype=np.int64)
    R, H, D = q.shape
    if k.shape[0] != H or v.shape[0] != H or k.shape[2] != D:
        raise ValueError("cache shape does not match q")
    s = default_scale(D) if scale is None else float(scale)
    out = np.zeros((R, H, D), dtype=np.float64)
    lse = np.zeros((H, R), dtype=np.float64)
    limits = np.array([row_limit(offsets, int(i)) for i in rows], dtype=np.int64)
    if R and limits.max() > k.shape[1]:
        raise ValueError("cache shorter than the visible prefix")
    if R == 0:
        return out, lse
    e_max = int(limits.max())
    for h in range(H):
        kh = k[h, :e_max, :].astype(np.float64)
        vh = v[h, :e_max, :].astype(np.float64)
        for e in np.unique(limits):
            sel = np.nonzero(limits == e)[0]
            x = s * (q[sel, h, :] @ kh[:e].T)                  # [r, e]
            m = x.max(axis=1, keepdims=True)                   # pass 1
            w = np.exp(x - m)                                  # pass 2
            l = w.sum(axis=1, keepdims=True)
            out[sel, h, :] = (w @ vh[:e]) / l
            lse[h, sel] = (m + np.log(l))[:, 0]
    return out, lse


def block_causal_attention(q, k_cache, v_cache, offsets, scale=None):
    """Full-sequence (prefill) block-causal attention over all T tokens.

    q : [T, H, D] with T = offsets[-1]; caches [H, >=T, D].
    """
    T = int(np.asarray(offsets)[-1])
    if q.shape[0] != T:
        raise ValueError("q must hold one row per token")
    return attention_rows(q, np.arange(T), k_cache, v_cache, offsets, scale)


def unit_attention(q_unit, k_cache, v_cache, offsets, scale=None):
    """Attention of the last block's tokens against the cache (one streaming step).

    The cache already holds every block up to and including the last one
    (the performer appends the received slice first, then solves:
    "全双工语音模型精读⑫" (alwayszhang.cn), 四、推理, step 3).
    q_unit : [offsets[-1] - offsets[-2], H, D].
    """
    offs = np.asarray(offsets, dtype=np.int64)
    rows = np.arange(offs[-2], offs[-1])
    if q_unit.shape[0] != rows.size:
        raise ValueError("q_unit must hold the last block's tokens")
    return attention_rows(q_unit, rows, k_cache, v_cache, offs, scale)

