"""ws_block_causal_attn_noalloc: the attention entry point for callers that
cannot allocate device memory (no cudaMalloc, no torch allocation inside the
call), which uses the library's static device scratch instead of a caller
workspace.  It must give the results of ws_block_causal_attn with a caller
workspace, on consecutive calls that reuse the scratch left by the previous
one.

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


def _with_workspace(case):
    H, D = case.w.heads, case.w.head_dim
    q_len = case.q.shape[0]
    out = torch.full_like(case.q, float("nan"))
    lse = torch.full((H, q_len), float("nan"), device="cuda")
    wsp = ws.workspace_for(q_len, case.T, H, D)
    ws.ws_block_causal_attn(case.q, case.k, case.v, out, case.offsets, case.offs_dev, lse=lse,
                            workspace=wsp)
    torch.cuda.synchronize()
    return out, lse


def _no_alloc(case):
    H = case.w.heads
    out = torch.full_like(case.q, float("nan"))
    lse = torch.full((H, case.q.shape[0]), float("nan"), device="cuda")
    ws.ws_block_causal_attn_noalloc(case.q, case.k, case.v, out, case.offsets, case.offs_dev,
                                    lse=lse)
    torch.cuda.synchronize()
    return out, lse


def test_no_alloc_matches_workspace_entry_point_on_consecutive_calls():
    # Two cases whose key ranges are split across CTA groups, so the scratch
    # holds partial results that the combine step reads back.
    a = Case(custom_workload(31, 2, 128), [8000, 300], q_units=[1], cap_extra=5)
    b = Case(custom_workload(32, 3, 128), [5000, 2000, 934], q_units=[2], cap_extra=9)
    for c in (a, b):
        assert ws.ws_block_causal_attn_workspace_size(c.q.shape[0], c.T, c.w.heads, 128) > 0
    ref = {id(c): _with_workspace(c) for c in (a, b)}
    # a, then b on the scratch a left behind, then a again on b's leftovers
    for c in (a, b, a):
        out, lse = _no_alloc(c)
        ref_out, ref_lse = ref[id(c)]
        r = ref_out.float().cpu().numpy().astype(np.float64)
        assert_close_bf16(out.float().cpu().numpy(), r, "no-alloc vs workspace call")
        assert_lse(lse.cpu().numpy(), ref_lse.cpu().numpy().astype(np.float64), "no-alloc LSE")
