"""Run by tests/test_gpu_debug_build.py in a child process with WS_DEBUG=1:
one small pass of every kernel of the debug build (bounds-checked indices),
checked against the oracle; the device error word must stay clean.  Prints
"debug build ok" on success."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def main():
    import numpy as np
    import torch

    from oracle import block_causal as bc
    from streaming_block_causal_flash_b300 import build as ws_build
    from streaming_block_causal_flash_b300 import ws
    from tests.gpu_cases import Case, assert_close_bf16, custom_workload

    assert os.environ.get("WS_DEBUG") == "1" and ws.LIB_PATH.endswith("libws_b300_debug.so")
    ws_build.build(debug=True)
    ws.load()
    ws.ws_clear_device_error()
    dev = torch.device("cuda")
    # split-KV unit attention, prefill, side buffers with the fused commit
    c = Case(custom_workload(61, 3, 128), [3000, 1700, 301], q_units=[2], cap_extra=40)
    out = torch.empty_like(c.q)
    ws.ws_block_causal_attn(c.q, c.k, c.v, out, c.offsets, c.offs_dev,
                            workspace=ws.workspace_for(c.q.shape[0], c.T, 3, 128))
    _, ref, _ = c.oracle()
    assert_close_bf16(out.float().cpu().numpy(), ref, "debug build unit attention")
    p = Case(custom_workload(62, 2, 128), [200, 130, 77])
    pout = torch.empty_like(p.q)
    ws.ws_block_causal_prefill(p.q, p.k, p.v, pout, p.offsets, p.offs_dev)
    _, pref, _ = p.oracle()
    assert_close_bf16(pout.float().cpu().numpy(), pref, "debug build prefill")
    w = c.w
    ks, vs = (w.token_major(n, 2, c.sizes).to(dev) for n in ("k", "v"))
    k2, v2 = c.k.clone(), c.v.clone()
    k2[:, int(c.offsets[2]):] = 0
    v2[:, int(c.offsets[2]):] = 0
    sout = torch.empty_like(c.q)
    ws.ws_block_causal_attn_side(c.q, k2, v2, ks, vs, sout, c.offsets, c.offs_dev, commit=True,
                                 workspace=ws.workspace_for(c.q.shape[0], c.T, 3, 128))
    torch.cuda.synchronize()
    assert_close_bf16(sout.float().cpu().numpy(), ref, "debug build side attention")
    assert torch.equal(k2[:, :c.T], c.k[:, :c.T]) and torch.equal(v2[:, :c.T], c.v[:, :c.T])
    # device-resident sizes: append and attention of the last unit
    k3, v3 = c.k.clone(), c.v.clone()
    k3[:, int(c.offsets[2]):] = 0
    v3[:, int(c.offsets[2]):] = 0
    state = ws.unit_state(int(c.offsets[2]), c.q.shape[0], 2, device=dev)
    dout = torch.empty_like(c.q)
    cap = c.k.shape[1]
    wsp = torch.empty(ws.ws_block_causal_attn_dev_workspace_size(c.q.shape[0], cap, 3, 128),
                      dtype=torch.uint8, device=dev)
    ws.ws_kv_append_dev(ks, vs, k3, v3, state)
    ws.ws_block_causal_attn_dev(c.q, k3, v3, dout, state, workspace=wsp)
    torch.cuda.synchronize()
    assert_close_bf16(dout.float().cpu().numpy(), ref, "debug build device-resident attention")
    assert torch.equal(k3, c.k) and torch.equal(v3, c.v)
    # Euler
    z = torch.randn(4099, device=dev)
    v = torch.randn(4099, device=dev).to(torch.bfloat16)
    zr = z.double().cpu().numpy() - 0.25 * v.double().cpu().numpy()
    ws.ws_fm_euler_step(z, v, 0.25)
    torch.cuda.synchronize()
    assert np.abs(z.cpu().numpy() - zr).max() <= 1e-6 * max(1.0, np.abs(zr).max())
    code, info = ws.ws_get_device_error()
    assert code == 0, f"debug build reported device error {code}/{info:#x}"
    print("debug build ok", flush=True)


if __name__ == "__main__":
    main()
