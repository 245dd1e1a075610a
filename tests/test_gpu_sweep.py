"""Seeded random-shape sweep of the bf16 attention against the fp64 oracle.

Each case draws a head count and a block layout (history blocks, then the
query block) from its seed: query blocks of 1 to 9 tiles (odd counts get
solo CTAs, even ones pairs only), ragged tails, empty history blocks and key
ranges split over several CTA groups.  Every case runs five ways through the
C ABI: the unit call, the side-buffer call with the fused commit (cache rows
of the unit checked bit for bit, rows past it untouched), the call with
device-resident sizes (a query buffer sized for the largest unit), the
no-alloc call, and the prefill of the whole sequence."""
import numpy as np
import pytest
import torch

from oracle import block_causal as bc
from oracle import kv_cache as kvc
from streaming_block_causal_flash_b300 import build as ws_build
from streaming_block_causal_flash_b300 import ws
from tests.gpu_cases import Case, assert_close_bf16, assert_lse, custom_workload

pytestmark = pytest.mark.gpu

SEEDS = list(range(200, 216))


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


def draw(seed):
    """(heads, block sizes): 0-4 history blocks of 0-2000 tokens, then a query
    block of 1-1100 tokens."""
    rng = np.random.default_rng(seed)
    heads = int(rng.integers(1, 7))
    n_hist = int(rng.integers(0, 5))
    hist = [int(x) for x in rng.integers(0, 2001, size=n_hist)]
    q = int(rng.integers(1, 1101))
    return heads, hist + [q]


@pytest.mark.parametrize("seed", SEEDS)
def test_random_layout_every_entry_point(seed):
    heads, sizes = draw(seed)
    w = custom_workload(seed, heads, 128)
    case = Case(w, sizes, q_units=[len(sizes) - 1], cap_extra=29)
    H, q_len = heads, case.q.shape[0]
    lo, hi = int(case.offsets[-2]), int(case.offsets[-1])
    _, ref, ref_lse = case.oracle()

    # unit call
    out = torch.full_like(case.q, float("nan"))
    lse = torch.full((H, q_len), float("nan"), device="cuda")
    wsp = ws.workspace_for(q_len, case.T, H, 128)
    if wsp is not None:
        wsp.fill_(0xFF)
    ws.ws_block_causal_attn(case.q, case.k, case.v, out, case.offsets, case.offs_dev, lse=lse,
                            workspace=wsp)
    torch.cuda.synchronize()
    assert_close_bf16(out.float().cpu().numpy(), ref, f"unit {sizes}")
    assert_lse(lse.cpu().numpy(), ref_lse, f"unit {sizes}")

    # side buffers with the fused commit: the unit's cache rows start as NaN
    k_side = w.token_major("k", len(sizes) - 1, case.sizes).cuda()
    v_side = w.token_major("v", len(sizes) - 1, case.sizes).cuda()
    kc, vc = case.k.clone(), case.v.clone()
    kc[:, lo:hi] = float("nan")
    vc[:, lo:hi] = float("nan")
    kc[:, hi:] = 5.0                   # canary rows past the unit
    vc[:, hi:] = -5.0
    out_s = torch.full_like(case.q, float("nan"))
    if wsp is not None:
        wsp.fill_(0xFF)
    ws.ws_block_causal_attn_side(case.q, kc, vc, k_side, v_side, out_s, case.offsets,
                                 case.offs_dev, workspace=wsp, commit=True)
    torch.cuda.synchronize()
    assert torch.equal(kc[:, lo:hi], k_side.transpose(0, 1))
    assert torch.equal(vc[:, lo:hi], v_side.transpose(0, 1))
    assert torch.equal(kc[:, :lo], case.k[:, :lo]) and torch.equal(vc[:, :lo], case.v[:, :lo])
    assert bool((kc[:, hi:] == 5.0).all()) and bool((vc[:, hi:] == -5.0).all())
    k_o, v_o = kvc.kv_append(case.k_host.float().numpy(), case.v_host.float().numpy(),
                             k_side.float().cpu().numpy(), v_side.float().cpu().numpy(), lo)
    ref_s, _ = bc.unit_attention(case.q_host.float().numpy(), k_o, v_o, case.offsets)
    assert_close_bf16(out_s.float().cpu().numpy(), ref_s, f"side+commit {sizes}")

    # device-resident sizes (the graph path): the unit's queries in a buffer
    # sized for the largest unit, the sizes read from a device state
    q_max = min(1152, case.cap)        # a unit never exceeds the cache
    q_buf = torch.zeros(q_max, H, 128, dtype=torch.bfloat16, device="cuda")
    q_buf[:q_len] = case.q
    out_d = torch.full_like(q_buf, float("nan"))
    lse_d = torch.full((H, q_max), float("nan"), device="cuda")
    wsd = torch.empty(ws.ws_block_causal_attn_dev_workspace_size(q_max, case.cap, H, 128),
                      dtype=torch.uint8, device="cuda").fill_(0xFF)
    state = ws.unit_state(lo, q_len, len(sizes) - 1)
    ws.ws_block_causal_attn_dev(q_buf, case.k, case.v, out_d, state, lse=lse_d, workspace=wsd)
    torch.cuda.synchronize()
    assert_close_bf16(out_d[:q_len].float().cpu().numpy(), ref, f"device sizes {sizes}")
    assert_lse(lse_d[:, :q_len].cpu().numpy(), ref_lse, f"device sizes {sizes}")

    # no-alloc entry point (library scratch instead of a workspace)
    out_n = torch.full_like(case.q, float("nan"))
    ws.ws_block_causal_attn_noalloc(case.q, case.k, case.v, out_n, case.offsets, case.offs_dev)
    torch.cuda.synchronize()
    assert_close_bf16(out_n.float().cpu().numpy(), ref, f"no-alloc {sizes}")

    # prefill of the whole sequence (every block's rows)
    full = Case(w, sizes, cap_extra=3)
    out_p = torch.full_like(full.q, float("nan"))
    lse_p = torch.full((H, full.T), float("nan"), device="cuda")
    ws.ws_block_causal_prefill(full.q, full.k, full.v, out_p, full.offsets, full.offs_dev,
                               lse=lse_p)
    torch.cuda.synchronize()
    _, ref_p, ref_lse_p = full.oracle()
    assert_close_bf16(out_p.float().cpu().numpy(), ref_p, f"prefill {sizes}")
    assert_lse(lse_p.cpu().numpy(), ref_lse_p, f"prefill {sizes}")
