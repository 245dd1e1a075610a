"""ws_block_causal_attn_noalloc: the attention entry point for callers that
cannot allocate device memory (no cudaMalloc, no torch allocation inside the
call), which uses the library's static device scratch instead of a caller
workspace.

It must give the results of ws_block_causal_attn with a caller workspace and
match the fp64 oracle, on consecutive calls that reuse the scratch left by
the previous one, and the calls must leave the device's free memory
unchanged (they allocate nothing).

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes when run alone."""
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


def _outputs(case):
    H = case.w.heads
    out = torch.full_like(case.q, float("nan"))
    lse = torch.full((H, case.q.shape[0]), float("nan"), device="cuda")
    return out, lse


def _with_workspace(case):
    H, D = case.w.heads, case.w.head_dim
    q_len = case.q.shape[0]
    out, lse = _outputs(case)
    wsp = ws.workspace_for(q_len, case.T, H, D)
    ws.ws_block_causal_attn(case.q, case.k, case.v, out, case.offsets, case.offs_dev, lse=lse,
                            workspace=wsp)
    torch.cuda.synchronize()
    return out, lse


def _no_alloc(case, out, lse):
    out.fill_(float("nan"))
    lse.fill_(float("nan"))
    ws.ws_block_causal_attn_noalloc(case.q, case.k, case.v, out, case.offsets, case.offs_dev,
                                    lse=lse)
    torch.cuda.synchronize()
    return out, lse


def test_no_alloc_matches_workspace_entry_point_and_oracle_on_consecutive_calls():
    # Two cases whose key ranges are split across CTA groups, so the scratch
    # holds partial results that the combine step reads back.
    a = Case(custom_workload(31, 2, 128), [8000, 300], q_units=[1], cap_extra=5)
    b = Case(custom_workload(32, 3, 128), [5000, 2000, 934], q_units=[2], cap_extra=9)
    for c in (a, b):
        assert ws.ws_block_causal_attn_workspace_size(c.q.shape[0], c.T, c.w.heads, 128) > 0
    ref = {id(c): _with_workspace(c) for c in (a, b)}
    oracle = {id(c): c.oracle() for c in (a, b)}
    bufs = {id(c): _outputs(c) for c in (a, b)}
    # a, then b on the scratch a left behind, then a again on b's leftovers
    for c in (a, b, a):
        out, lse = _no_alloc(c, *bufs[id(c)])
        got = out.float().cpu().numpy()
        ref_out, ref_lse = ref[id(c)]
        assert_close_bf16(got, ref_out.float().cpu().numpy().astype(np.float64),
                          "no-alloc vs workspace call")
        assert_lse(lse.cpu().numpy(), ref_lse.cpu().numpy().astype(np.float64), "no-alloc LSE")
        _, o_ref, l_ref = oracle[id(c)]
        assert_close_bf16(got, o_ref, "no-alloc vs oracle")
        assert_lse(lse.cpu().numpy(), l_ref, "no-alloc LSE vs oracle")


def test_no_alloc_calls_leave_free_device_memory_unchanged():
    # After one warm-up call (which may load the library's module on this
    # device and so reserve the static scratch), further calls must not
    # change the device's free memory: they allocate nothing.
    c = Case(custom_workload(33, 2, 128), [6000, 500], q_units=[1], cap_extra=3)
    out, lse = _outputs(c)
    _no_alloc(c, out, lse)
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        ws.ws_block_causal_attn_noalloc(c.q, c.k, c.v, out, c.offsets, c.offs_dev, lse=lse)
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before, f"free device memory changed by {free_before - free_after} B"
    _, o_ref, _ = c.oracle()
    assert_close_bf16(out.float().cpu().numpy(), o_ref, "no-alloc after repeated calls")
