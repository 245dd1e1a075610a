"""GPU parity at the full workload sizes, in the launch configuration the
benchmark times (``bench.UnitSession`` / ``bench.run_unit``: KV append, then
ws_block_causal_attn with the session's workspace, then the Euler steps).

* unit_192x336 -- every head and row against the fp64 oracle;
* unit_640x368 -- one head in full, every head on sampled rows, the appended
  slice bit-exact, four Euler steps in full;
* prefill_128x932 -- the full-sequence prefill on sampled rows of every head,
  and the streaming invariant: units attended one at a time over the cache
  agree with the prefill's rows;
* long_session_640x368 -- 16 consecutive units over a ~479k-token history:
  sampled heads and rows of three units, the cache after all appends, the
  Euler result of the last unit.

Sampled rows always include the first and last row of the query block and
the rows on both sides of every 128-row tile boundary the kernels use."""
import numpy as np
import pytest
import torch

import bench
from oracle import block_causal as bc
from oracle import flow_matching as fm
from streaming_block_causal_flash_b300 import build as ws_build
from streaming_block_causal_flash_b300 import ws
from streaming_block_causal_flash_b300.inputs import WORKLOADS
from tests.gpu_cases import Case, assert_close_bf16, assert_lse

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def native():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    ws_build.build()
    ws.load()
    ws.ws_clear_device_error()
    yield
    code, info = ws.ws_get_device_error()
    assert code == 0, f"device error word set: {info:#x}"


def sample_rows(n_rows: int, seed: int, n_random: int = 16, tile_step: int = 1) -> np.ndarray:
    """Local row indices 0..n_rows-1 to check: ends, tile boundaries, random."""
    rows = {0, n_rows - 1}
    for b in range(128, n_rows, 128 * tile_step):
        rows.update((b - 1, b))
    rng = np.random.default_rng(seed)
    rows.update(rng.integers(0, n_rows, size=n_random).tolist())
    return np.array(sorted(r for r in rows if 0 <= r < n_rows), dtype=np.int64)


def session_head_cache(sess, heads, upto_unit):
    """fp32 K/V of the given heads over units 0..upto_unit (history plus the
    new units' slices), as the cache holds them after those appends."""
    e = int(sess.offsets_all[upto_unit + 1])
    k = sess.k_host[heads, :e].float().numpy()
    v = sess.v_host[heads, :e].float().numpy()
    for u in sess.units:
        if u > upto_unit:
            break
        lo, hi = int(sess.offsets_all[u]), int(sess.offsets_all[u + 1])
        k_new, v_new = sess.kv_host[u]
        k[:, lo:hi] = k_new[:, heads].transpose(0, 1).float().numpy()
        v[:, lo:hi] = v_new[:, heads].transpose(0, 1).float().numpy()
    return k, v


def check_unit(sess, u, heads, rows_local, what):
    """The session's last attention output (unit u) against the oracle."""
    offs = sess.offsets_all[:u + 2]
    lo, hi = int(offs[-2]), int(offs[-1])
    k, v = session_head_cache(sess, heads, u)
    q = sess.q_host[u][rows_local][:, heads].float().numpy()
    ref, _ = bc.attention_rows(q, lo + rows_local, k, v, offs)
    got = sess.out[:hi - lo][rows_local][:, heads].float().cpu().numpy()
    return assert_close_bf16(got, ref, what)


def check_euler(sess, u, what):
    z = sess.eps_host[u].numpy().astype(np.float64)
    for s in range(sess.w.euler_steps):
        z = fm.euler_step(z, sess.vel_host[u][s].float().numpy(), 1.0 / sess.w.euler_steps)
    got = sess.z[u].cpu().numpy().astype(np.float64)
    err = np.abs(got - z).max()
    assert err <= 1e-6 * max(1.0, np.abs(z).max()), f"{what}: Euler err {err:.3e}"


def test_unit_192x336_every_head_and_row():
    w = WORKLOADS["unit_192x336"]
    sess = bench.UnitSession(w, torch.device("cuda"))
    u = sess.units[0]
    bench.run_unit(sess, u, torch.cuda.current_stream())
    torch.cuda.synchronize()
    n = sess.sizes[u]
    check_unit(sess, u, list(range(w.heads)), np.arange(n), "unit_192x336 all rows")
    check_euler(sess, u, "unit_192x336")


def test_unit_640x368_head_in_full_and_sampled_rows():
    w = WORKLOADS["unit_640x368"]
    sess = bench.UnitSession(w, torch.device("cuda"))
    u = sess.units[0]
    stream = torch.cuda.current_stream()
    bench.run_unit(sess, u, stream)
    torch.cuda.synchronize()
    n = sess.sizes[u]
    lo = int(sess.offsets_all[u])
    # the slice the step appended, bit for bit
    k_new, v_new = sess.kv_host[u]
    assert torch.equal(sess.k[:, lo:lo + n].cpu(), k_new.transpose(0, 1))
    assert torch.equal(sess.v[:, lo:lo + n].cpu(), v_new.transpose(0, 1))
    check_unit(sess, u, [17], np.arange(n), "unit_640x368 head 17, all rows")
    check_unit(sess, u, list(range(w.heads)), sample_rows(n, 3), "unit_640x368 sampled rows")
    check_euler(sess, u, "unit_640x368")
    # LSE of the same call shape (the benchmark passes none)
    lse = torch.empty(w.heads, n, dtype=torch.float32, device="cuda")
    offs = sess.offsets_all[:u + 2]
    ws.ws_block_causal_attn(sess.q[u], sess.k, sess.v, sess.out[:n], offs, sess.offs_dev[u],
                            lse=lse, workspace=sess.workspace)
    torch.cuda.synchronize()
    heads = [0, 17, 39]
    rows = sample_rows(n, 4)
    k, v = session_head_cache(sess, heads, u)
    _, ref_lse = bc.attention_rows(sess.q_host[u][rows][:, heads].float().numpy(), lo + rows, k, v,
                                   offs)
    assert_lse(lse[heads][:, rows].cpu().numpy(), ref_lse, "unit_640x368 LSE")


def test_prefill_128x932_sampled_rows_and_streaming_invariant():
    w = WORKLOADS["prefill_128x932"]
    sizes = w.unit_sizes()
    case = Case(w, sizes)
    H, T = w.heads, case.T
    out = torch.empty_like(case.q)
    lse = torch.empty(H, T, dtype=torch.float32, device="cuda")
    ws.ws_block_causal_prefill(case.q, case.k, case.v, out, case.offsets, case.offs_dev, lse=lse)
    torch.cuda.synchronize()
    rows = sample_rows(T, 5, n_random=24, tile_step=61)
    for b in (0, 1, 63, 127):                  # first/last row of some units
        rows = np.union1d(rows, [int(case.offsets[b]), int(case.offsets[b + 1]) - 1])
    sel, ref, ref_lse = case.oracle(row_sel=rows)
    assert_close_bf16(out[rows].float().cpu().numpy(), ref, "prefill sampled rows")
    assert_lse(lse[:, rows].cpu().numpy(), ref_lse, "prefill LSE")
    # Streaming invariant: unit b attended over blocks 0..b of the same cache.
    for b in (0, 64, 127):
        lo, hi = int(case.offsets[b]), int(case.offsets[b + 1])
        offs_b = case.offsets[:b + 2]
        q_b = case.q[lo:hi]
        out_b = torch.empty_like(q_b)
        wsp = ws.workspace_for(hi - lo, hi, H, w.head_dim)
        ws.ws_block_causal_attn(q_b, case.k, case.v, out_b, offs_b, case.offs_dev[:b + 2],
                                workspace=wsp)
        torch.cuda.synchronize()
        r = sample_rows(hi - lo, 6 + b)
        _, ref_b, _ = case.oracle(row_sel=lo + r)
        assert_close_bf16(out_b[r].float().cpu().numpy(), ref_b, f"unit {b} incremental")
        full_rows = out[lo:hi].float().cpu().numpy().astype(np.float64)
        assert_close_bf16(out_b.float().cpu().numpy(), full_rows, f"unit {b}: incremental vs prefill")


def test_long_session_16_units():
    w = WORKLOADS["long_session_640x368"]
    sess = bench.UnitSession(w, torch.device("cuda"))
    stream = torch.cuda.current_stream()
    heads = [0, 19, 39]
    checked = {sess.units[0], sess.units[7], sess.units[-1]}
    for u in sess.units:
        bench.run_unit(sess, u, stream)
        if u in checked:
            torch.cuda.synchronize()
            check_unit(sess, u, heads, sample_rows(sess.sizes[u], u, n_random=8, tile_step=2),
                       f"long session unit {u}")
    torch.cuda.synchronize()
    e = int(sess.offsets_all[sess.units[-1] + 1])
    for h in heads:
        k, v = session_head_cache(sess, [h], sess.units[-1])
        assert np.array_equal(sess.k[h, :e].float().cpu().numpy(), k[0]), f"K cache head {h}"
        assert np.array_equal(sess.v[h, :e].float().cpu().numpy(), v[0]), f"V cache head {h}"
    check_euler(sess, sess.units[-1], "long session last unit")
