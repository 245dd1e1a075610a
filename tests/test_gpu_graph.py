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
