"""Failure detection on the GPU without a fault: every in-kernel wait of the
tensor-core attention has a wall-clock limit.  The test hook
ws_debug_force_wait_timeout makes one MMA issuer wait on a barrier that
nothing completes; with a 20 ms limit that wait gives up, the kernel records
the site in its device error word, every role drains its own copies and
MMAs, frees its tensor memory and returns.  The host reads WS_ERR_TIMEOUT,
and the context stays usable: the next call is correct."""
import numpy as np
import pytest
import torch

from streaming_block_causal_flash_b300 import build as ws_build
from streaming_block_causal_flash_b300 import ws
from tests.gpu_cases import Case, assert_close_bf16, custom_workload

pytestmark = pytest.mark.gpu

DEFAULT_LIMIT_NS = 2_000_000_000


@pytest.fixture(scope="module", autouse=True)
def native():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    ws_build.build()
    ws.load()
    ws.ws_clear_device_error()
    yield
    ws.ws_debug_force_wait_timeout(False)
    ws.ws_set_wait_timeout_ns(DEFAULT_LIMIT_NS)
    ws.ws_clear_device_error()


def _call(case, wsp):
    out = torch.zeros_like(case.q)
    ws.ws_block_causal_attn(case.q, case.k, case.v, out, case.offsets, case.offs_dev, workspace=wsp)
    return out


def test_wait_limit_reports_timeout_and_context_survives():
    case = Case(custom_workload(40, 2, 128), [3000, 300], q_units=[1])
    wsp = ws.workspace_for(300, case.T, 2, 128)
    torch.cuda.synchronize()
    ws.ws_set_wait_timeout_ns(20_000_000)
    ws.ws_debug_force_wait_timeout(True)
    try:
        _call(case, wsp)
        code, info = ws.ws_get_device_error()      # synchronises
    finally:
        ws.ws_debug_force_wait_timeout(False)
        ws.ws_set_wait_timeout_ns(DEFAULT_LIMIT_NS)
    assert code == 1, "the stalled wait must give up"
    site, block = info >> 16, info & 0xFFFF
    assert 1 <= site <= 13, f"unknown wait site {site}"
    assert block < 148 * 4
    with pytest.raises(ws.WsError) as ei:
        ws._check(ws.load().ws_get_device_error(*(ws.ctypes.byref(ws.ctypes.c_int()) for _ in range(2))))
    assert ei.value.status == ws.WS_ERR_TIMEOUT
    ws.ws_clear_device_error()
    assert ws.ws_get_device_error() == (0, 0)
    # the same context runs the next call correctly
    out = _call(case, wsp)
    torch.cuda.synchronize()
    assert ws.ws_get_device_error()[0] == 0
    _, ref, _ = case.oracle()
    assert_close_bf16(out.float().cpu().numpy(), ref, "after a timed-out call")
