"""Ulysses-style context parallelism for one streaming unit's attention.

The chooseai.io news item on Wan-Streamer v0.2 (summary bullet 2, and the
paragraph on the performer) says the performer's video generation runs on
several GPUs through Ulysses context parallelism: each GPU holds a slice of
the unit's long token sequence, and for attention the slices are regrouped so
that each GPU holds every token of a subset of the heads.  Attention is
independent per head, so each GPU then runs the block-causal attention of its
heads over its own head-sharded KV cache, and the inverse regrouping returns
each GPU's slice of the output for all heads.

Partitioning (N ranks, H heads, N divides H):
  * sequence shards: rank r holds tokens [lo_r, hi_r) of the unit, all heads
    ([n_r, H, D]); the token ranges are contiguous and in rank order, the
    first n % N ranks holding one token more;
  * head shards: rank r holds heads [r H/N, (r+1) H/N) of every token;
  * the K/V cache is sharded by head: rank r keeps [H/N, capacity, D] and
    appends only its heads of each unit's slice -- no exchange beyond the two
    all-to-alls of the unit's own tokens;
  * the latents of the flow-matching Euler step stay sequence-sharded (the
    update is elementwise): no exchange at all.

Both regroupings are one all_to_all_single of local buffers (NCCL on the
device, gloo on the CPU): every rank sends and receives into memory it owns,
no kernel reads a peer's memory.  With one rank they are plain reshapes.
"""
from __future__ import annotations

from typing import Callable, List, Optional, Sequence, Tuple

import torch


def shard_bounds(n: int, world: int) -> List[Tuple[int, int]]:
    """Token range [lo, hi) of each rank's sequence shard of an n-token unit."""
    if world < 1:
        raise ValueError("world must be >= 1")
    base, extra = divmod(int(n), world)
    out, lo = [], 0
    for r in range(world):
        hi = lo + base + (1 if r < extra else 0)
        out.append((lo, hi))
        lo = hi
    return out


def _world(group) -> Tuple[int, int]:
    if group is None and not torch.distributed.is_initialized():
        return 0, 1
    return torch.distributed.get_rank(group), torch.distributed.get_world_size(group)


def seq_to_head(x_seq: torch.Tensor, n_total: int, group=None) -> torch.Tensor:
    """[n_r, H, D] (this rank's tokens, all heads) -> [n_total, H/N, D] (every
    token, this rank's heads), by one all-to-all."""
    rank, world = _world(group)
    n_r, H, D = x_seq.shape
    if H % world:
        raise ValueError(f"{H} heads do not split over {world} ranks")
    bounds = shard_bounds(n_total, world)
    if n_r != bounds[rank][1] - bounds[rank][0]:
        raise ValueError(f"rank {rank} holds {n_r} tokens; its shard has "
                         f"{bounds[rank][1] - bounds[rank][0]}")
    hs = H // world
    if world == 1:
        return x_seq.contiguous()
    # send buffer ordered by destination rank: [world][n_r][hs][D]
    send = x_seq.reshape(n_r, world, hs, D).permute(1, 0, 2, 3).contiguous()
    recv = torch.empty(n_total, hs, D, dtype=x_seq.dtype, device=x_seq.device)
    in_splits = [n_r * hs * D] * world
    out_splits = [(hi - lo) * hs * D for lo, hi in bounds]
    torch.distributed.all_to_all_single(recv.view(-1), send.view(-1), out_splits, in_splits,
                                        group=group)
    return recv


def head_to_seq(x_head: torch.Tensor, group=None) -> torch.Tensor:
    """[n_total, H/N, D] (every token, this rank's heads) -> [n_r, H, D] (this
    rank's tokens, all heads): the inverse of seq_to_head."""
    rank, world = _world(group)
    n_total, hs, D = x_head.shape
    bounds = shard_bounds(n_total, world)
    if world == 1:
        return x_head.contiguous()
    lo, hi = bounds[rank]
    n_r = hi - lo
    # the send buffer, in token order, is already ordered by destination rank
    send = x_head.contiguous()
    recv = torch.empty(world, n_r, hs, D, dtype=x_head.dtype, device=x_head.device)
    in_splits = [(b - a) * hs * D for a, b in bounds]
    out_splits = [n_r * hs * D] * world
    torch.distributed.all_to_all_single(recv.view(-1), send.view(-1), out_splits, in_splits,
                                        group=group)
    # recv[j] holds heads [j hs, (j+1) hs) of this rank's tokens
    return recv.permute(1, 0, 2, 3).reshape(n_r, world * hs, D)


def head_range(num_heads: int, group=None) -> Tuple[int, int]:
    """Heads [lo, hi) held by this rank's head shard (and its KV cache)."""
    rank, world = _world(group)
    if num_heads % world:
        raise ValueError(f"{num_heads} heads do not split over {world} ranks")
    hs = num_heads // world
    return rank * hs, (rank + 1) * hs


AttnFn = Callable[[torch.Tensor, torch.Tensor, torch.Tensor, torch.Tensor, torch.Tensor,
                   Sequence[int]], torch.Tensor]


def native_unit_attention(q_h, k_new_h, v_new_h, k_cache, v_cache, offsets,
                          offsets_dev: Optional[torch.Tensor] = None, workspace=None,
                          stream=None) -> torch.Tensor:
    """This rank's heads of the unit: append the unit's K/V slice to the
    head-sharded cache, then block-causal attention of the unit's queries
    against it, through the C ABI (ws_kv_append, ws_block_causal_attn)."""
    from streaming_block_causal_flash_b300 import ws
    import numpy as np
    offs = np.asarray(offsets, dtype=np.int32)
    ws.ws_kv_append(k_new_h, v_new_h, k_cache, v_cache, int(offs[-2]), stream=stream)
    if offsets_dev is None:
        offsets_dev = torch.from_numpy(offs).to(q_h.device)
    out = torch.empty_like(q_h)
    H, _, D = k_cache.shape
    if workspace is None:
        workspace = ws.workspace_for(int(offs[-1] - offs[-2]), int(offs[-1]), H, D, device=q_h.device)
    ws.ws_block_causal_attn(q_h, k_cache, v_cache, out, offs, offsets_dev, workspace=workspace,
                            stream=stream)
    return out


def ulysses_unit_attention(q_seq: torch.Tensor, k_seq: torch.Tensor, v_seq: torch.Tensor,
                           k_cache: torch.Tensor, v_cache: torch.Tensor, offsets: Sequence[int],
                           group=None, attn: Optional[Callable] = None) -> torch.Tensor:
    """One unit's attention under Ulysses context parallelism.

    q_seq, k_seq, v_seq: this rank's sequence shard of the unit ([n_r, H, D]);
    k_cache, v_cache: this rank's head shard of the cache ([H/N, capacity, D]),
    holding blocks 0 .. n_blocks-2 of its heads; offsets: the block offsets of
    the whole timeline (host), the unit being the last block.

    Returns this rank's sequence shard of the output, all heads ([n_r, H, D]).
    `attn(q_h, k_h, v_h, k_cache, v_cache, offsets)` runs the head-sharded
    append and attention; by default the native kernels."""
    n_total = int(offsets[-1]) - int(offsets[-2])
    q_h = seq_to_head(q_seq, n_total, group)
    k_h = seq_to_head(k_seq, n_total, group)
    v_h = seq_to_head(v_seq, n_total, group)
    fn = native_unit_attention if attn is None else attn
    o_h = fn(q_h, k_h, v_h, k_cache, v_cache, offsets)
    return head_to_seq(o_h, group)
