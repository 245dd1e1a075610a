"""GPU parity: KV append (bit-exact), flow-matching Euler step and the fp32
attention path, each against the fp64 CPU oracle through the C ABI."""
import numpy as np
import pytest
import torch

from oracle import flow_matching as fm
from oracle import kv_cache as kvc
from streaming_block_causal_flash_b300 import build as ws_build
from streaming_block_causal_flash_b300 import ws
from streaming_block_causal_flash_b300.inputs import WORKLOADS, normal
from tests.gpu_cases import F32_ABS, Case, assert_close_abs, assert_lse, custom_workload

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


# --------------------------------------------------------------------- Euler

def test_euler_one_step_closed_form_tiny_fp32():
    w = WORKLOADS["tiny_fp32"]
    z0, eps = w.z0(0), w.eps(0)
    v = eps - z0                                    # exact velocity, fp32
    z = eps.clone().cuda()
    ws.ws_fm_euler_step(z, v.cuda(), 1.0)
    got = z.cpu().numpy().astype(np.float64)
    ref = fm.euler_step(eps.numpy(), v.numpy(), 1.0)
    assert_close_abs(got, ref, F32_ABS, "euler vs oracle")
    assert_close_abs(got, z0.numpy(), F32_ABS, "euler vs closed form z0")
    # one fp32 rounding of the fp64 result
    assert np.array_equal(got.astype(np.float32), ref.astype(np.float32))


@pytest.mark.parametrize("name,extra", [("unit_192x336", 0), ("unit_640x368", 0), ("unit_192x336", 5)])
def test_euler_four_bf16_steps(name, extra):
    w = WORKLOADS[name]
    n = w.latent_tokens * w.latent_channels + extra
    z_init = torch.cat([w.eps(0).flatten(), normal(9, "z_tail", 0, (extra,))])
    vs = [torch.cat([w.velocity_input(0, s).flatten(),
                     normal(9, "v_tail", s, (extra,), 1.0, torch.bfloat16)]) for s in range(4)]
    z = z_init.clone().cuda()
    zb = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    ref = z_init.numpy().astype(np.float64)
    for s in range(4):
        ws.ws_fm_euler_step(z, vs[s].cuda(), 0.25, z_bf16_out=zb)
        ref = fm.euler_step(ref, vs[s].float().numpy(), 0.25)
        got = z.cpu().numpy().astype(np.float64)
        assert_close_abs(got, ref, 1e-6 * max(1.0, np.abs(ref).max()), f"step {s}")
        # the bf16 copy is the round-to-nearest-even image of the new fp32 z
        assert torch.equal(zb.cpu(), z.cpu().to(torch.bfloat16)), "bf16 copy"


def test_euler_exact_velocity_recovers_z0_in_four_steps():
    w = WORKLOADS["unit_640x368"]
    z0, eps = w.z0(1), w.eps(1)
    v = (eps - z0).cuda()
    z = eps.clone().cuda()
    for _ in range(4):
        ws.ws_fm_euler_step(z, v, 0.25)
    np.testing.assert_allclose(z.cpu().numpy(), z0.numpy(), rtol=0, atol=1e-5)


@pytest.mark.parametrize("guidance", [0.0, 1.0, 3.0])
def test_euler_cfg_four_bf16_steps(guidance):
    """Guided step against the oracle.  Bound from the fp32 arithmetic: per
    step the kernel rounds d = v_c - v_u, v = fma(w, d, v_u) and
    z = fma(-dtau, v, z) once each, an error of at most
    2^-24 (|z| + dtau (|v| + |w| |d|)) per step (taken as 2^-23 for margin),
    accumulated over the steps.  The bf16 copy must be the exact
    round-to-nearest-even image of the fp32 result."""
    w = WORKLOADS["unit_640x368"]
    n = w.latent_tokens * w.latent_channels + 5
    z_init = normal(7, "z_cfg", 0, (n,))
    vus = [normal(7, "vu", s, (n,), 1.0, torch.bfloat16) for s in range(4)]
    vcs = [normal(7, "vc", s, (n,), 1.0, torch.bfloat16) for s in range(4)]
    z = z_init.clone().cuda()
    zb = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    ref = z_init.numpy().astype(np.float64)
    bound = 0.0
    for s in range(4):
        ws.ws_fm_euler_cfg_step(z, vus[s].cuda(), vcs[s].cuda(), guidance, 0.25, z_bf16_out=zb)
        vu, vc = vus[s].float().numpy(), vcs[s].float().numpy()
        v = fm.cfg_velocity(vu, vc, guidance)
        ref = fm.cfg_euler_step(ref, vu, vc, guidance, 0.25)
        bound += 2.0 ** -23 * (np.abs(ref).max() + 0.25 * (np.abs(v).max() + abs(guidance) * np.abs(vc - vu).max()))
        got = z.cpu().numpy().astype(np.float64)
        assert_close_abs(got, ref, bound, f"guided step {s}")
        assert torch.equal(zb.cpu(), z.cpu().to(torch.bfloat16)), "bf16 copy"


def test_euler_cfg_with_exact_velocity_recovers_z0():
    w = WORKLOADS["unit_192x336"]
    z0, eps = w.z0(3), w.eps(3)
    v = (eps - z0).cuda()
    z = eps.clone().cuda()
    ws.ws_fm_euler_cfg_step(z, v, v, 2.5, 1.0)
    np.testing.assert_allclose(z.cpu().numpy(), z0.numpy(), rtol=0, atol=F32_ABS)


# ----------------------------------------------------------------- KV append

@pytest.mark.parametrize("name", ["tiny_fp32", "unit_192x336", "unit_640x368"])
def test_kv_append_bit_exact_with_canaries(name):
    w = WORKLOADS[name]
    sizes = w.unit_sizes()
    offs = w.offsets()
    u = w.n_units - 1
    k_new, v_new = w.token_major("k", u, sizes), w.token_major("v", u, sizes)
    cap = w.capacity()
    canary_k = torch.full((w.heads, cap, w.head_dim), 7.0, dtype=w.torch_dtype)
    canary_v = torch.full((w.heads, cap, w.head_dim), -3.0, dtype=w.torch_dtype)
    kc, vc = canary_k.cuda(), canary_v.cuda()
    cache_len = int(offs[u])
    ws.ws_kv_append(k_new.cuda(), v_new.cuda(), kc, vc, cache_len)
    ref_k, ref_v = kvc.kv_append(canary_k.float().numpy(), canary_v.float().numpy(),
                                 k_new.float().numpy(), v_new.float().numpy(), cache_len)
    assert torch.equal(kc.cpu(), torch.from_numpy(ref_k).to(w.torch_dtype))
    assert torch.equal(vc.cpu(), torch.from_numpy(ref_v).to(w.torch_dtype))
    # bit-level: the bytes of the written rows are the slice's bytes
    assert torch.equal(kc[:, cache_len:cache_len + k_new.shape[0]].cpu().view(torch.int16 if w.dtype == "bf16" else torch.int32),
                       k_new.transpose(0, 1).contiguous().view(torch.int16 if w.dtype == "bf16" else torch.int32))


def test_kv_append_unit_by_unit_rebuilds_timeline():
    w = WORKLOADS["unit_192x336"]
    sizes = w.unit_sizes()
    offs = w.offsets()
    kc = torch.zeros(w.heads, w.capacity(), w.head_dim, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    for u in range(w.n_units):
        k, v = w.token_major("k", u, sizes), w.token_major("v", u, sizes)
        ws.ws_kv_append(k.cuda(), v.cuda(), kc, vc, int(offs[u]))
    for h in (0, 7, w.heads - 1):
        assert torch.equal(kc[h, :offs[-1]].cpu(), w.head_timeline("k", h, w.n_units, sizes))
        assert torch.equal(vc[h, :offs[-1]].cpu(), w.head_timeline("v", h, w.n_units, sizes))


def test_kv_append_capacity_error_touches_nothing():
    kc = torch.zeros(2, 16, 128, dtype=torch.bfloat16, device="cuda")
    k = torch.ones(4, 2, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ws.WsError) as ei:
        ws.ws_kv_append(k, k, kc, kc.clone(), 13)
    assert ei.value.status == ws.WS_ERR_CAPACITY
    assert int(torch.count_nonzero(kc)) == 0


# ------------------------------------------------------- fp32 attention (tiny)

def test_fp32_tiny_prefill_and_incremental():
    w = WORKLOADS["tiny_fp32"]
    sizes = w.unit_sizes()
    case = Case(w, sizes)
    out = torch.empty_like(case.q)
    lse = torch.empty(w.heads, case.T, dtype=torch.float32, device="cuda")
    ws.ws_block_causal_prefill(case.q, case.k, case.v, out, case.offsets, case.offs_dev, lse=lse)
    _, ref, ref_lse = case.oracle()
    assert_close_abs(out.cpu().numpy(), ref, F32_ABS, "fp32 prefill")
    assert_lse(lse.cpu().numpy(), ref_lse, "fp32 prefill")
    # incremental: cache grows block by block; unit b attends to blocks 0..b
    for b in range(len(sizes)):
        inc = Case(w, sizes, n_units=b + 1, q_units=[b], cap_extra=w.capacity() - int(case.offsets[b + 1]))
        o = torch.empty_like(inc.q)
        ws.ws_block_causal_attn(inc.q, inc.k, inc.v, o, inc.offsets, inc.offs_dev)
        _, r, _ = inc.oracle()
        assert_close_abs(o.cpu().numpy(), r, F32_ABS, f"fp32 unit {b}")
        lo, hi = int(case.offsets[b]), int(case.offsets[b + 1])
        assert_close_abs(o.cpu().numpy(), ref[lo:hi], F32_ABS, f"incremental == prefill rows, unit {b}")


@pytest.mark.parametrize("D", [64, 128])
def test_fp32_ragged_blocks(D):
    w = custom_workload(21, heads=3, head_dim=D, dtype="f32", std=1.0)
    sizes = [5, 0, 40, 1, 77, 3]
    case = Case(w, sizes)
    out = torch.empty_like(case.q)
    ws.ws_block_causal_prefill(case.q, case.k, case.v, out, case.offsets, case.offs_dev)
    _, ref, _ = case.oracle()
    assert_close_abs(out.cpu().numpy(), ref, F32_ABS, "fp32 ragged prefill")
