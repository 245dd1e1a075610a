"""Ulysses head-sharded attention for one streaming unit (CPU, world size 2
on gloo): the sequence-to-head regrouping and its inverse are bit-exact
against direct slicing, and the sharded unit step (each rank appending and
attending with its heads only, over its head-sharded cache) reassembles to the
unsharded result.  The per-rank attention here is the fp64 oracle, standing in
for the native kernels, which need a GPU per rank; the oracle is only the
checker of the sharding logic."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from streaming_block_causal_flash_b300 import ulysses
from streaming_block_causal_flash_b300.inputs import block_offsets
from tests.gpu_cases import custom_workload


def test_shard_bounds_cover_the_unit_in_rank_order():
    for n in (0, 1, 7, 934, 933):
        for world in (1, 2, 3, 4, 8):
            b = ulysses.shard_bounds(n, world)
            assert b[0][0] == 0 and b[-1][1] == n and len(b) == world
            assert all(b[i][1] == b[i + 1][0] for i in range(world - 1))
            sizes = [hi - lo for lo, hi in b]
            assert max(sizes) - min(sizes) <= 1 and sizes == sorted(sizes, reverse=True)
    with pytest.raises(ValueError):
        ulysses.shard_bounds(5, 0)


def test_single_rank_is_the_identity():
    x = torch.randn(9, 4, 8)
    assert torch.equal(ulysses.seq_to_head(x, 9), x)
    assert torch.equal(ulysses.head_to_seq(x), x)
    assert ulysses.head_range(4) == (0, 4)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _regroup_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out = []
        for n, H in ((934, 40), (933, 8), (5, 4), (1, 2), (3, 4)):
            if H % world:
                continue                  # heads must divide over the ranks
            g = torch.Generator().manual_seed(n * 100 + H)
            full = torch.randn(n, H, 16, generator=g).to(torch.bfloat16)
            lo, hi = ulysses.shard_bounds(n, world)[rank]
            h0, h1 = ulysses.head_range(H)
            heads = ulysses.seq_to_head(full[lo:hi].clone(), n)
            ok_fwd = torch.equal(heads, full[:, h0:h1])
            back = ulysses.head_to_seq(heads)
            ok_back = torch.equal(back, full[lo:hi])
            # the inverse alone, from a head shard built by slicing
            ok_inv = torch.equal(ulysses.head_to_seq(full[:, h0:h1].clone()), full[lo:hi])
            out.append((n, H, ok_fwd, ok_back, ok_inv))
        q.put((rank, out))
    finally:
        torch.distributed.destroy_process_group()


def _run(worker, world=2, extra=()):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=worker, args=(r, world, port, q, *extra)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=300) for _ in procs]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    return dict(res)


@pytest.mark.parametrize("world", [2, 4])
def test_regrouping_both_directions_bit_exact(world):
    res = _run(_regroup_worker, world=world)
    assert len(res) == world
    for rank, rows in res.items():
        for n, H, ok_fwd, ok_back, ok_inv in rows:
            assert ok_fwd, f"rank {rank}: sequence->head differs from slicing (n={n}, H={H})"
            assert ok_back, f"rank {rank}: head->sequence does not invert (n={n}, H={H})"
            assert ok_inv, f"rank {rank}: head->sequence differs from slicing (n={n}, H={H})"


SIZES = [300, 257, 400, 190, 301]     # four history units, then the streamed unit
HEADS = 4


def _oracle_attention(q_h, k_h, v_h, k_cache, v_cache, offsets):
    """Per-rank stand-in for the native append + attention: the oracle on this
    rank's heads (test infrastructure only)."""
    from oracle import block_causal as bc
    from oracle import kv_cache as kc
    offs = np.asarray(offsets)
    kc_new, vc_new = kc.kv_append(k_cache.float().numpy(), v_cache.float().numpy(),
                                  k_h.float().numpy(), v_h.float().numpy(), int(offs[-2]))
    k_cache.copy_(torch.from_numpy(kc_new))
    v_cache.copy_(torch.from_numpy(vc_new))
    o, _ = bc.unit_attention(q_h.double().numpy(), kc_new[:, :int(offs[-1])], vc_new[:, :int(offs[-1])], offs)
    return torch.from_numpy(o)


def _step_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = custom_workload(81, HEADS, 128)
        offs = block_offsets(SIZES)
        u = len(SIZES) - 1
        T_hist = int(offs[u])
        h0, h1 = ulysses.head_range(HEADS)
        cap = int(offs[-1]) + 16
        # this rank's head shard of the cache, history only
        k_cache = torch.zeros(h1 - h0, cap, 128, dtype=torch.float64)
        v_cache = torch.zeros_like(k_cache)
        for i, h in enumerate(range(h0, h1)):
            k_cache[i, :T_hist] = w.head_timeline("k", h, u, SIZES).double()
            v_cache[i, :T_hist] = w.head_timeline("v", h, u, SIZES).double()
        lo, hi = ulysses.shard_bounds(SIZES[u], world)[rank]
        q_u, k_u, v_u = (w.token_major(name, u, SIZES) for name in ("q", "k", "v"))
        o_seq = ulysses.ulysses_unit_attention(q_u[lo:hi].double(), k_u[lo:hi].double(),
                                               v_u[lo:hi].double(), k_cache, v_cache, offs,
                                               attn=_oracle_attention)
        # the appended rows of this rank's heads are the slice's rows
        appended = torch.equal(k_cache[:, T_hist:T_hist + SIZES[u]], k_u[:, h0:h1].transpose(0, 1).double())
        q.put((rank, (lo, hi, o_seq.numpy(), appended)))
    finally:
        torch.distributed.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_sharded_unit_step_matches_unsharded(world):
    from oracle import block_causal as bc
    res = _run(_step_worker, world=world)
    w = custom_workload(81, HEADS, 128)
    offs = block_offsets(SIZES)
    u = len(SIZES) - 1
    k = torch.stack([w.head_timeline("k", h, len(SIZES), SIZES) for h in range(HEADS)]).double().numpy()
    v = torch.stack([w.head_timeline("v", h, len(SIZES), SIZES) for h in range(HEADS)]).double().numpy()
    ref, _ = bc.unit_attention(w.token_major("q", u, SIZES).double().numpy(), k, v, offs)
    got = np.zeros_like(ref)
    covered = 0
    for rank, (lo, hi, o, appended) in res.items():
        assert appended, f"rank {rank} appended the wrong rows"
        got[lo:hi] = o
        covered += hi - lo
    assert covered == SIZES[u]
    # same per-head arithmetic on both sides: equal up to BLAS blocking order
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12 * np.abs(ref).max())
