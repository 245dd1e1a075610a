"""The Ulysses layer's native path on one GPU (one rank: the regroupings are
reshapes): its head-sharded append and attention run the library's kernels
and give what ws_kv_append + ws_block_causal_attn give, bit for bit, and
match the oracle."""
import numpy as np
import pytest
import torch

from streaming_block_causal_flash_b300 import build as ws_build
from streaming_block_causal_flash_b300 import ulysses, ws
from streaming_block_causal_flash_b300.inputs import block_offsets
from tests.gpu_cases import assert_close_bf16, custom_workload

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


def test_single_rank_ulysses_step_runs_the_native_kernels():
    from oracle import block_causal as bc
    sizes = [700, 650, 934]
    w = custom_workload(91, 8, 128)
    offs = block_offsets(sizes)
    u = len(sizes) - 1
    T_hist, T = int(offs[u]), int(offs[-1])
    dev = torch.device("cuda")

    def cache():
        k = torch.zeros(w.heads, T + 8, 128, dtype=torch.bfloat16)
        v = torch.zeros_like(k)
        for h in range(w.heads):
            k[h, :T_hist] = w.head_timeline("k", h, u, sizes)
            v[h, :T_hist] = w.head_timeline("v", h, u, sizes)
        return k.to(dev), v.to(dev)

    q, kn, vn = (w.token_major(name, u, sizes).to(dev) for name in ("q", "k", "v"))
    k1, v1 = cache()
    o_u = ulysses.ulysses_unit_attention(q, kn, vn, k1, v1, offs)
    k2, v2 = cache()
    ws.ws_kv_append(kn, vn, k2, v2, T_hist)
    o_ref = torch.empty_like(q)
    ws.ws_block_causal_attn(q, k2, v2, o_ref, offs, torch.from_numpy(offs.astype(np.int32)).to(dev),
                            workspace=ws.workspace_for(sizes[u], T, w.heads, 128))
    torch.cuda.synchronize()
    assert torch.equal(o_u, o_ref) and torch.equal(k1, k2) and torch.equal(v1, v2)
    k_t = torch.stack([w.head_timeline("k", h, len(sizes), sizes) for h in range(w.heads)]).float().numpy()
    v_t = torch.stack([w.head_timeline("v", h, len(sizes), sizes) for h in range(w.heads)]).float().numpy()
    ref, _ = bc.unit_attention(q.float().cpu().numpy(), k_t, v_t, offs)
    assert_close_bf16(o_u.float().cpu().numpy(), ref, "Ulysses native step")
