"""GPU parity of the bf16 tcgen05 attention against the fp64 oracle on small
and ragged shapes: tails shorter than a tile, odd query-tile counts, empty
blocks, one-token units, pure causal and pure bidirectional block layouts,
heavy split-KV, LSE output, and peaky softmax stress inputs."""
import numpy as np
import pytest
import torch

from streaming_block_causal_flash_b300 import build as ws_build
from streaming_block_causal_flash_b300 import ws
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


def run_unit(case, with_lse=True, scale=0.0):
    """ws_block_causal_attn for the last block of the case."""
    H, D = case.w.heads, case.w.head_dim
    q_len = case.q.shape[0]
    out = torch.full_like(case.q, float("nan"))
    lse = torch.full((H, q_len), float("nan"), device="cuda") if with_lse else None
    wsp = ws.workspace_for(q_len, case.T, H, D)
    if wsp is not None:
        wsp.fill_(0xFF)          # contents on entry must not matter
    ws.ws_block_causal_attn(case.q, case.k, case.v, out, case.offsets, case.offs_dev, lse=lse,
                            softmax_scale=scale, workspace=wsp)
    torch.cuda.synchronize()
    return out, lse


def run_prefill(case, with_lse=True, scale=0.0):
    H = case.w.heads
    out = torch.full_like(case.q, float("nan"))
    lse = torch.full((H, case.T), float("nan"), device="cuda") if with_lse else None
    ws.ws_block_causal_prefill(case.q, case.k, case.v, out, case.offsets, case.offs_dev, lse=lse,
                               softmax_scale=scale)
    torch.cuda.synchronize()
    return out, lse


UNIT_CASES = [
    # (seed, heads, block sizes) -- the last block is the query block
    (1, 1, [128, 128]),            # exact tiles
    (2, 2, [300, 77]),             # q shorter than a tile, ragged key tail
    (3, 3, [1000, 1000, 600]),     # 5 query tiles: odd count, 3 pairs
    (4, 1, [5000, 1]),             # one-token unit
    (5, 2, [8000, 300]),           # many groups per head: heavy split-KV
    (6, 4, [0, 130, 0, 260]),      # empty blocks around
    (7, 1, [40]),                  # first unit, no history
    (8, 2, [2000, 513]),           # q tile boundary + 1
]


@pytest.mark.parametrize("seed,heads,sizes", UNIT_CASES)
def test_unit_attention_matches_oracle(seed, heads, sizes):
    w = custom_workload(seed, heads, 128)
    case = Case(w, sizes, q_units=[len(sizes) - 1], cap_extra=17)
    out, lse = run_unit(case)
    _, ref, ref_lse = case.oracle()
    assert_close_bf16(out.float().cpu().numpy(), ref, f"unit {sizes}")
    assert_lse(lse.cpu().numpy(), ref_lse, f"unit {sizes}")


PREFILL_CASES = [
    (11, 2, [100, 37, 200, 0, 300]),   # ragged, one empty block
    (12, 1, [16] * 40),                # many small blocks
    (13, 1, [1] * 300),                # block size 1: causal attention
    (14, 2, [700]),                    # one block: full bidirectional attention
    (15, 3, [932] * 3),                # three 640x368-sized units
    (16, 1, [129, 127, 256, 1, 255]),  # straddling tile boundaries
    (17, 2, [90, 60]),                 # one query-tile pair: a couple of one
]


@pytest.mark.parametrize("seed,heads,sizes", PREFILL_CASES)
def test_prefill_matches_oracle(seed, heads, sizes):
    w = custom_workload(seed, heads, 128)
    case = Case(w, sizes, cap_extra=3)
    out, lse = run_prefill(case)
    _, ref, ref_lse = case.oracle()
    assert_close_bf16(out.float().cpu().numpy(), ref, f"prefill {sizes}")
    assert_lse(lse.cpu().numpy(), ref_lse, f"prefill {sizes}")


def test_prefill_rows_equal_incremental_units():
    """Streaming invariant on the GPU: each unit's rows from the prefill agree
    with that unit attended incrementally over a cache holding blocks 0..b."""
    w = custom_workload(17, 2, 128)
    sizes = [300, 250, 400, 130]
    full = Case(w, sizes)
    out_full, _ = run_prefill(full, with_lse=False)
    for b in range(len(sizes)):
        inc = Case(w, sizes, n_units=b + 1, q_units=[b], cap_extra=64)
        out_b, _ = run_unit(inc, with_lse=False)
        lo, hi = int(full.offsets[b]), int(full.offsets[b + 1])
        _, ref, _ = inc.oracle()
        assert_close_bf16(out_b.float().cpu().numpy(), ref, f"unit {b}")
        assert_close_bf16(out_full[lo:hi].float().cpu().numpy(), ref, f"prefill rows {b}")


def test_explicit_softmax_scale():
    w = custom_workload(18, 2, 128)
    case = Case(w, [600, 300], q_units=[1])
    out, lse = run_unit(case, scale=0.3)
    _, ref, ref_lse = case.oracle(scale=0.3)
    assert_close_bf16(out.float().cpu().numpy(), ref, "scale 0.3")
    assert_lse(lse.cpu().numpy(), ref_lse, "scale 0.3")


@pytest.mark.parametrize("std", [2.0, 4.0])
def test_stress_peaky_softmax(std):
    """Inputs x4/x8 the default scale: logits with std ~4-16 force many
    running-max rescales."""
    w = custom_workload(19, 2, 128, std=std)
    case = Case(w, [3000, 500], q_units=[1])
    out, lse = run_unit(case)
    _, ref, ref_lse = case.oracle()
    assert_close_bf16(out.float().cpu().numpy(), ref, f"std {std}")
    assert_lse(lse.cpu().numpy(), ref_lse, f"std {std}")


def test_stress_late_spike_key_forces_rescale():
    """One key per head late in the history with a huge logit: the running max
    jumps after many tiles have been accumulated."""
    w = custom_workload(20, 2, 128)
    case = Case(w, [4000, 256], q_units=[1])
    j = 3500
    for h in range(2):
        qm = case.q_host[:, h].float().mean(0)
        case.k_host[h, j] = (qm / qm.norm() * 400.0).to(torch.bfloat16)
        case.v_host[h, j] = torch.full((128,), 3.0, dtype=torch.bfloat16)
    case.k = case.k_host.cuda()
    case.v = case.v_host.cuda()
    out, lse = run_unit(case)
    _, ref, ref_lse = case.oracle()
    assert_close_bf16(out.float().cpu().numpy(), ref, "spike")
    assert_lse(lse.cpu().numpy(), ref_lse, "spike")


def test_workspace_too_small_is_rejected():
    w = custom_workload(22, 2, 128)
    case = Case(w, [8000, 300], q_units=[1])
    need = ws.ws_block_causal_attn_workspace_size(300, case.T, 2, 128)
    assert need > 0
    small = torch.empty(need // 2, dtype=torch.uint8, device="cuda")
    out = torch.zeros_like(case.q)
    with pytest.raises(ws.WsError) as ei:
        ws.ws_block_causal_attn(case.q, case.k, case.v, out, case.offsets, case.offs_dev,
                                workspace=small)
    assert ei.value.status == ws.WS_ERR_INVALID_ARGUMENT
    assert int(torch.count_nonzero(out)) == 0
