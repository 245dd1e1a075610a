"""ws_block_causal_attn_side: the newest unit's queries against the cache
(blocks before the last) plus the unit's own K/V from token-major side
buffers, without touching the cache.  Checked against the fp64 oracle of the
same attention with the slice appended (oracle.kv_cache.kv_append, then
oracle.block_causal.unit_attention).  The cache rows the last unit would
occupy are filled with NaN, so any read of them would poison the output."""
import numpy as np
import pytest
import torch

import bench
from oracle import block_causal as bc
from oracle import kv_cache as kvc
from streaming_block_causal_flash_b300 import build as ws_build
from streaming_block_causal_flash_b300 import ws
from streaming_block_causal_flash_b300.inputs import WORKLOADS, normal
from tests.gpu_cases import Case, assert_close_bf16, assert_lse, custom_workload

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


def side_case(seed, heads, sizes, cap_extra=11):
    """Case whose cache holds blocks 0..n-2; the last block's cache rows are NaN."""
    w = custom_workload(seed, heads, 128)
    case = Case(w, sizes, q_units=[len(sizes) - 1], cap_extra=cap_extra)
    lo, hi = int(case.offsets[-2]), int(case.offsets[-1])
    case.k_side = w.token_major("k", len(sizes) - 1, case.sizes).cuda()
    case.v_side = w.token_major("v", len(sizes) - 1, case.sizes).cuda()
    case.k[:, lo:hi] = float("nan")
    case.v[:, lo:hi] = float("nan")
    return case


def run_side(case, k_side=None, v_side=None, with_lse=True):
    H = case.w.heads
    q_len = case.q.shape[0]
    out = torch.full_like(case.q, float("nan"))
    lse = torch.full((H, q_len), float("nan"), device="cuda") if with_lse else None
    wsp = ws.workspace_for(q_len, case.T, H, 128)
    if wsp is not None:
        wsp.fill_(0xFF)
    ws.ws_block_causal_attn_side(case.q, case.k, case.v,
                                 case.k_side if k_side is None else k_side,
                                 case.v_side if v_side is None else v_side,
                                 out, case.offsets, case.offs_dev, lse=lse, workspace=wsp)
    torch.cuda.synchronize()
    return out, lse


def oracle_with_side(case, k_side, v_side):
    """Oracle: append the side slice to the history, then attend."""
    lo = int(case.offsets[-2])
    k, v = kvc.kv_append(case.k_host.float().numpy(), case.v_host.float().numpy(),
                         k_side.float().cpu().numpy(), v_side.float().cpu().numpy(), lo)
    return bc.unit_attention(case.q_host.float().numpy(), k, v, case.offsets)


SIDE_CASES = [
    (41, 1, [128, 128]),
    (42, 2, [300, 77]),
    (43, 3, [1000, 1000, 600]),
    (44, 4, [0, 130, 0, 260]),
    (45, 1, [40]),                 # first unit: no history in the cache
    (46, 2, [8000, 300]),          # split key range
    (47, 1, [129, 127, 256, 1, 255]),
    (48, 2, [5000, 1]),            # one-token unit
]


@pytest.mark.parametrize("seed,heads,sizes", SIDE_CASES)
def test_side_attention_matches_oracle(seed, heads, sizes):
    case = side_case(seed, heads, sizes)
    out, lse = run_side(case)
    ref, ref_lse = oracle_with_side(case, case.k_side, case.v_side)
    assert_close_bf16(out.float().cpu().numpy(), ref, f"side {sizes}")
    assert_lse(lse.cpu().numpy(), ref_lse, f"side {sizes}")


def test_solver_steps_then_commit():
    """Four solver steps re-attend with fresh (noisy) unit K/V from the side
    buffers; the final slice is then committed with ws_kv_append and the
    plain call over the cache agrees with the last side call."""
    case = side_case(49, 2, [3000, 2000, 934])
    n = case.q.shape[0]
    for step in range(4):
        ks = normal(49, "k_noisy", step, (n, 2, 128), 0.5, torch.bfloat16).cuda()
        vs = normal(49, "v_noisy", step, (n, 2, 128), 0.5, torch.bfloat16).cuda()
        out, _ = run_side(case, ks, vs, with_lse=False)
        ref, _ = oracle_with_side(case, ks, vs)
        assert_close_bf16(out.float().cpu().numpy(), ref, f"solver step {step}")
    ws.ws_kv_append(ks, vs, case.k, case.v, int(case.offsets[-2]))
    plain = torch.empty_like(case.q)
    ws.ws_block_causal_attn(case.q, case.k, case.v, plain, case.offsets, case.offs_dev,
                            workspace=ws.workspace_for(n, case.T, 2, 128))
    torch.cuda.synchronize()
    assert_close_bf16(plain.float().cpu().numpy(), ref, "committed")
    assert_close_bf16(out.float().cpu().numpy(), plain.float().cpu().numpy().astype(np.float64),
                      "side vs committed")


def test_side_unit_640x368_sampled_rows():
    w = WORKLOADS["unit_640x368"]
    sess = bench.UnitSession(w, torch.device("cuda"))
    u = sess.units[0]
    n = sess.sizes[u]
    offs = sess.offsets_all[:u + 2]
    k_side, v_side = sess.kv[u]
    out = torch.empty(n, w.heads, w.head_dim, dtype=torch.bfloat16, device="cuda")
    ws.ws_block_causal_attn_side(sess.q[u], sess.k, sess.v, k_side, v_side, out, offs,
                                 sess.offs_dev[u], workspace=sess.workspace)
    torch.cuda.synchronize()
    lo = int(offs[-2])
    rows = np.unique(np.concatenate([[0, n - 1, 127, 128, 255, 256, 511, 512],
                                     np.random.default_rng(5).integers(0, n, 12)]))
    heads = [0, 21, 39]
    k = sess.k_host[heads, :lo].float().numpy()
    v = sess.v_host[heads, :lo].float().numpy()
    k, v = kvc.kv_append(np.concatenate([k, np.zeros((3, n, 128), np.float32)], 1),
                         np.concatenate([v, np.zeros((3, n, 128), np.float32)], 1),
                         k_side[:, heads].float().cpu().numpy(), v_side[:, heads].float().cpu().numpy(), lo)
    ref, _ = bc.attention_rows(sess.q_host[u][rows][:, heads].float().numpy(), lo + rows, k, v, offs)
    assert_close_bf16(out[rows][:, heads].float().cpu().numpy(), ref, "640x368 side")


# ------------------------------------------------- fused commit (append fused in)

@pytest.mark.parametrize("seed,heads,sizes", [
    (51, 2, [300, 77]),
    (52, 3, [1000, 1000, 600]),
    (53, 1, [40]),                  # no history
    (54, 2, [8000, 300]),           # split key range: several groups share the head
    (55, 4, [0, 130, 0, 260]),
    (56, 1, [129, 127, 256, 1, 255]),
])
def test_side_commit_writes_the_slice_and_nothing_else(seed, heads, sizes):
    case = side_case(seed, heads, sizes, cap_extra=37)
    lo, hi = int(case.offsets[-2]), int(case.offsets[-1])
    case.k[:, hi:] = 7.0            # canary rows past the unit
    case.v[:, hi:] = -3.0
    k_before, v_before = case.k.clone(), case.v.clone()
    H, q_len = heads, case.q.shape[0]
    out = torch.full_like(case.q, float("nan"))
    wsp = ws.workspace_for(q_len, case.T, H, 128)
    ws.ws_block_causal_attn_side(case.q, case.k, case.v, case.k_side, case.v_side, out, case.offsets,
                                 case.offs_dev, workspace=wsp, commit=True)
    torch.cuda.synchronize()
    # the unit's rows hold the slice, bit for bit; every other row is as before
    assert torch.equal(case.k[:, lo:hi], case.k_side.transpose(0, 1))
    assert torch.equal(case.v[:, lo:hi], case.v_side.transpose(0, 1))
    for t, before in ((case.k, k_before), (case.v, v_before)):
        assert torch.equal(t[:, :lo], before[:, :lo])
        assert torch.equal(t[:, hi:], before[:, hi:])
    ref, _ = oracle_with_side(case, case.k_side, case.v_side)
    assert_close_bf16(out.float().cpu().numpy(), ref, f"side+commit {sizes}")


def test_solver_steps_then_fused_commit():
    """Three noisy steps through side buffers, the last one commits its slice
    in the same call; the plain attention over the cache then agrees."""
    case = side_case(57, 2, [3000, 2000, 934])
    n = case.q.shape[0]
    lo, hi = int(case.offsets[-2]), int(case.offsets[-1])
    wsp = ws.workspace_for(n, case.T, 2, 128)
    for step in range(3):
        ks = normal(57, "k_noisy", step, (n, 2, 128), 0.5, torch.bfloat16).cuda()
        vs = normal(57, "v_noisy", step, (n, 2, 128), 0.5, torch.bfloat16).cuda()
        out = torch.empty_like(case.q)
        ws.ws_block_causal_attn_side(case.q, case.k, case.v, ks, vs, out, case.offsets, case.offs_dev,
                                     workspace=wsp, commit=(step == 2))
    torch.cuda.synchronize()
    assert torch.equal(case.k[:, lo:hi], ks.transpose(0, 1))
    plain = torch.empty_like(case.q)
    ws.ws_block_causal_attn(case.q, case.k, case.v, plain, case.offsets, case.offs_dev, workspace=wsp)
    torch.cuda.synchronize()
    ref, _ = oracle_with_side(case, ks, vs)
    assert_close_bf16(out.float().cpu().numpy(), ref, "last side step")
    assert_close_bf16(plain.float().cpu().numpy(), ref, "after fused commit")


@pytest.mark.parametrize("workload", ["unit_640x368", "unit_192x336"])
def test_side_commit_full_size_matches_append(workload):
    """At full size the fused commit writes exactly what ws_kv_append writes
    (640x368: four query-tile pairs per group; 192x336: one pair and solo
    CTAs for the unpaired third tile, which store nothing)."""
    w = WORKLOADS[workload]
    sess = bench.UnitSession(w, torch.device("cuda"))
    u = sess.units[0]
    n = sess.sizes[u]
    offs = sess.offsets_all[:u + 2]
    lo = int(offs[-2])
    k_side, v_side = sess.kv[u]
    k_ref, v_ref = sess.k.clone(), sess.v.clone()
    ws.ws_kv_append(k_side, v_side, k_ref, v_ref, lo)
    out = torch.empty(n, w.heads, w.head_dim, dtype=torch.bfloat16, device="cuda")
    ws.ws_block_causal_attn_side(sess.q[u], sess.k, sess.v, k_side, v_side, out, offs,
                                 sess.offs_dev[u], workspace=sess.workspace, commit=True)
    torch.cuda.synchronize()
    assert torch.equal(sess.k, k_ref)
    assert torch.equal(sess.v, v_ref)
