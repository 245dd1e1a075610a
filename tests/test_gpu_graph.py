"""The per-unit step (KV append, block-causal attention with split-KV
workspace, four Euler steps) is capturable in a CUDA graph: every call is
asynchronous on the given stream, allocates nothing and never synchronises.
A replay of the captured step gives bit-identical results to the eager step
(the kernels are deterministic for fixed sizes and launch shapes)."""
import numpy as np
import pytest
import torch

import bench
from streaming_block_causal_flash_b300 import build as ws_build
from streaming_block_causal_flash_b300 import ws
from streaming_block_causal_flash_b300.inputs import WORKLOADS

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


def test_unit_step_graph_replay_matches_eager():
    w = WORKLOADS["unit_192x336"]
    sess = bench.UnitSession(w, torch.device("cuda"))
    u = sess.units[0]
    n = sess.sizes[u]
    stream = torch.cuda.current_stream()
    z_start = sess.eps_host[u].cuda()
    # eager step
    sess.z[u].copy_(z_start)
    bench.run_unit(sess, u, stream)
    torch.cuda.synchronize()
    out_eager, z_eager = sess.out[:n].clone(), sess.z[u].clone()
    k_eager = sess.k.clone()
    # captured step, replayed twice from the same starting z
    sess.out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        bench.run_unit(sess, u, torch.cuda.current_stream())
    for _ in range(2):
        sess.z[u].copy_(z_start)
        sess.out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(sess.out[:n], out_eager)
        assert torch.equal(sess.z[u], z_eager)
        assert torch.equal(sess.k, k_eager)
    assert np.isfinite(out_eager.float().cpu().numpy()).all()


def _ragged_session():
    """A small ragged timeline: 6 history units, then 4 streamed units whose
    sizes straddle 128-row tile boundaries; 4 heads, D = 128."""
    from tests.gpu_cases import custom_workload
    w = custom_workload(71, 4, 128)
    sizes = [300, 257, 400, 128, 333, 190, 301, 255, 129, 287]
    return w, sizes, 6


def test_one_graph_replayed_over_consecutive_units_with_device_sizes():
    """One captured unit step -- append, attention, four Euler steps, then the
    device-side state advance -- replayed for unit k, k+1, ...: each replay
    reads the unit's cache length and size from device memory.  Every unit's
    O and LSE match the oracle, its z matches the oracle's Euler steps, and
    after the last unit the cache holds the timeline bit for bit (rows past it
    untouched).  Query and slice rows past each unit are filled with junk
    (finite, as the entry point asks, and NaN for the slices, which are never
    read past the unit) to show that no result depends on them."""
    from oracle import block_causal as bc
    from oracle import flow_matching as fm
    from streaming_block_causal_flash_b300.inputs import block_offsets
    from tests.gpu_cases import assert_close_bf16, assert_lse

    w, sizes, hist = _ragged_session()
    H, D = w.heads, w.head_dim
    offs = block_offsets(sizes)
    T_hist, T = int(offs[hist]), int(offs[-1])
    cap = T + 200
    q_max = max(sizes[hist:])
    dev = torch.device("cuda")
    k_host = torch.zeros(H, cap, D, dtype=torch.bfloat16)
    v_host = torch.zeros_like(k_host)
    for h in range(H):
        k_host[h, :T_hist] = w.head_timeline("k", h, hist, sizes)
        v_host[h, :T_hist] = w.head_timeline("v", h, hist, sizes)
    k_cache, v_cache = k_host.to(dev), v_host.to(dev)
    nan = float("nan")
    q_buf = torch.zeros((q_max, H, D), dtype=torch.bfloat16, device=dev)
    kn_buf, vn_buf = torch.full_like(q_buf, nan), torch.full_like(q_buf, nan)
    torch.manual_seed(5)
    out = torch.full_like(q_buf, nan)
    lse = torch.full((H, q_max), nan, dtype=torch.float32, device=dev)
    n_lat, C = 16, 256
    z = torch.empty(n_lat * C, dtype=torch.float32, device=dev)
    vel = [torch.empty(n_lat * C, dtype=torch.bfloat16, device=dev) for _ in range(4)]
    state = ws.unit_state(T_hist, sizes[hist], hist, device=dev)
    sizes_dev = torch.tensor(sizes, dtype=torch.int32, device=dev)
    wsp = torch.empty(ws.ws_block_causal_attn_dev_workspace_size(q_max, cap, H, D), dtype=torch.uint8,
                      device=dev)
    wsp.fill_(0xFF)

    def step(st):
        ws.ws_kv_append_dev(kn_buf, vn_buf, k_cache, v_cache, state, stream=st)
        ws.ws_block_causal_attn_dev(q_buf, k_cache, v_cache, out, state, lse=lse, workspace=wsp, stream=st)
        for s_ in range(4):
            ws.ws_fm_euler_step(z, vel[s_], 0.25, stream=st)
        ws.ws_unit_state_advance(state, sizes_dev, stream=st)

    # capture with the state parked at an empty unit (n_new = 0), so that the
    # warm-up call and the capture itself leave the cache untouched
    saved = state.clone()
    state.copy_(ws.unit_state(T_hist, 0, hist - 1, device=dev))
    step(torch.cuda.current_stream())
    torch.cuda.synchronize()
    state.copy_(ws.unit_state(T_hist, 0, hist - 1, device=dev))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert torch.equal(k_cache.cpu(), k_host), "warm-up or capture wrote the cache"
    state.copy_(saved)

    k_full = torch.stack([w.head_timeline("k", h, len(sizes), sizes) for h in range(H)]).float().numpy()
    v_full = torch.stack([w.head_timeline("v", h, len(sizes), sizes) for h in range(H)]).float().numpy()
    for u in range(hist, len(sizes)):
        n = sizes[u]
        q_buf.normal_(0.0, 3.0), kn_buf.fill_(nan), vn_buf.fill_(nan), out.fill_(nan), lse.fill_(nan)
        q_u = w.token_major("q", u, sizes)
        q_buf[:n].copy_(q_u.to(dev))
        kn_buf[:n].copy_(w.token_major("k", u, sizes).to(dev))
        vn_buf[:n].copy_(w.token_major("v", u, sizes).to(dev))
        eps = torch.randn(n_lat * C, generator=torch.Generator().manual_seed(7000 + u))
        z.copy_(eps.to(dev))
        vel_h = [torch.randn(n_lat * C, generator=torch.Generator().manual_seed(1000 * u + s_)).to(torch.bfloat16)
                 for s_ in range(4)]
        for s_ in range(4):
            vel[s_].copy_(vel_h[s_].to(dev))
        g.replay()
        torch.cuda.synchronize()
        code, info = ws.ws_get_device_error()
        assert code == 0, f"device error word {code}/{info:#x} at unit {u}"
        e = int(offs[u + 1])
        ref_o, ref_lse = bc.unit_attention(q_u.float().numpy(), k_full[:, :e], v_full[:, :e], offs[:u + 2])
        assert_close_bf16(out[:n].float().cpu().numpy(), ref_o, f"unit {u} O")
        assert_lse(lse[:, :n].cpu().numpy(), ref_lse, f"unit {u} LSE")
        assert torch.isnan(out[n:].float()).all(), "rows past the unit were written"
        zr = eps.numpy().astype(np.float64)
        for s_ in range(4):
            zr = fm.euler_step(zr, vel_h[s_].float().numpy(), 0.25)
        zerr = np.abs(z.cpu().numpy() - zr).max()
        assert zerr <= 1e-6 * max(1.0, np.abs(zr).max()), f"unit {u} Euler err {zerr:.3e}"
        assert state.cpu().tolist() == [e, sizes[u + 1] if u + 1 < len(sizes) else 0, u + 1]
    k_end = k_cache.cpu()
    assert torch.equal(k_end[:, :T].float(), torch.from_numpy(k_full)), "K cache differs from the timeline"
    assert torch.equal(v_cache.cpu()[:, :T].float(), torch.from_numpy(v_full)), "V cache differs"
    assert not k_end[:, T:].any(), "rows past the timeline were written"


def test_device_sizes_out_of_range_write_nothing_and_report():
    """A device-resident state whose unit is larger than the launch's maximum
    (or does not fit the capacity) makes the kernels write nothing and report
    WS_ERR_CAPACITY through the device error word; the context stays usable."""
    w, sizes, hist = _ragged_session()
    H, D = w.heads, w.head_dim
    dev = torch.device("cuda")
    cap, q_max = 1024, 300
    k_cache = torch.zeros(H, cap, D, dtype=torch.bfloat16, device=dev)
    v_cache = torch.zeros_like(k_cache)
    slab = torch.ones(q_max, H, D, dtype=torch.bfloat16, device=dev)
    out = torch.zeros_like(slab)
    wsp = torch.empty(ws.ws_block_causal_attn_dev_workspace_size(q_max, cap, H, D), dtype=torch.uint8,
                      device=dev)
    ws.ws_clear_device_error()
    for bad in ([0, q_max + 1, 0], [cap - 10, 100, 0], [-1, 5, 0]):
        state = torch.tensor(bad, dtype=torch.int64, device=dev)
        ws.ws_kv_append_dev(slab, slab, k_cache, v_cache, state)
        ws.ws_block_causal_attn_dev(slab, k_cache, v_cache, out, state, workspace=wsp)
        code, info = ws.ws_get_device_error()
        assert code == 2 and info in (1, 2), (bad, code, info)
        with pytest.raises(ws.WsError) as ei:
            ws._check(ws.load().ws_get_device_error(*(ws.ctypes.byref(ws.ctypes.c_int()) for _ in range(2))))
        assert ei.value.status == ws.WS_ERR_CAPACITY
        ws.ws_clear_device_error()
        assert not k_cache.any() and not out.any(), f"state {bad} wrote memory"
    assert ws.ws_get_device_error() == (0, 0)
