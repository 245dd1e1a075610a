"""Pins for the fp64 CPU oracle: checks against what the pages and the
mathematics fix, never against the oracle's own code retyped.

Every test here runs on the CPU (no ``gpu`` mark).  The last group plants a
mistake in a copy of the oracle and shows that a pin above catches it.
"""
import os

import numpy as np
import pytest
import scipy.special
import torch

from oracle import block_causal as bc
from oracle import flow_matching as fm
from oracle import kv_cache as kvc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _random_offsets(rng, n_blocks, max_size, allow_empty=True):
    lo = 0 if allow_empty else 1
    sizes = rng.integers(lo, max_size + 1, size=n_blocks)
    if sizes.sum() == 0:
        sizes[0] = 1
    return np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)


def _qkv(rng, T, H, D):
    q = rng.standard_normal((T, H, D))
    k = rng.standard_normal((H, T, D))
    v = rng.standard_normal((H, T, D))
    return q, k, v


def _bruteforce(q, k, v, mask, scale):
    """Textbook masked softmax attention, one head, whole logit matrix."""
    x = scale * (q @ k.T)
    x = np.where(mask, x, -np.inf)
    w = np.exp(x - x.max(axis=1, keepdims=True))
    return (w / w.sum(axis=1, keepdims=True)) @ v


def _block_ids_by_scan(offsets):
    """Block id of each token by walking the sizes (no searchsorted)."""
    ids = []
    for b in range(len(offsets) - 1):
        ids += [b] * int(offsets[b + 1] - offsets[b])
    return np.array(ids, dtype=np.int64)


# ----------------------------------------------------------------------------
# Visibility rule
# ----------------------------------------------------------------------------

def test_golden_block_visibility_from_explainer_example():
    golden = np.loadtxt(os.path.join(GOLDEN, "block_visibility_explainer.txt"), dtype=np.int64)
    offsets = np.array([0, 3, 4, 8, 10])          # four blocks of sizes 3, 1, 4, 2
    mask = bc.visibility_mask(offsets)
    ids = _block_ids_by_scan(offsets)
    for a in range(4):
        for b in range(4):
            sub = mask[np.ix_(ids == a, ids == b)]
            assert sub.all() if golden[a, b] else not sub.any(), (a, b)
    # the prefix-length statement of the rule agrees token by token
    for i in range(offsets[-1]):
        e = bc.row_limit(offsets, i)
        assert mask[i, :e].all() and not mask[i, e:].any()


@pytest.mark.parametrize("seed", range(6))
def test_row_limit_matches_mask_with_empty_blocks(seed):
    rng = _rng(seed)
    offsets = _random_offsets(rng, n_blocks=9, max_size=5, allow_empty=True)
    mask = bc.visibility_mask(offsets)
    ids = _block_ids_by_scan(offsets)
    assert np.array_equal(mask, ids[None, :] <= ids[:, None])
    for i in range(offsets[-1]):
        assert bc.block_index(offsets, i) == ids[i]
        e = bc.row_limit(offsets, i)
        assert e == np.nonzero(mask[i])[0].max() + 1
        assert e >= i + 1                      # a token always sees itself


def test_special_case_masks():
    T = 12
    full = bc.visibility_mask([0, T])
    assert full.all()
    causal = bc.visibility_mask(np.arange(T + 1))
    assert np.array_equal(causal, np.tril(np.ones((T, T), dtype=bool)))


# ----------------------------------------------------------------------------
# Attention values
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(5))
def test_attention_matches_bruteforce_mask(seed):
    rng = _rng(100 + seed)
    offsets = _random_offsets(rng, n_blocks=7, max_size=6, allow_empty=True)
    T, H, D = int(offsets[-1]), 3, 8
    q, k, v = _qkv(rng, T, H, D)
    scale = 0.37
    out, lse = bc.block_causal_attention(q, k, v, offsets, scale)
    # explicit N x N mask built from token block ids, independent of row_limit
    ids = _block_ids_by_scan(offsets)
    mask = ids[None, :] <= ids[:, None]
    for h in range(H):
        ref = _bruteforce(q[:, h], k[h], v[h], mask, scale)
        np.testing.assert_allclose(out[:, h], ref, rtol=1e-12, atol=1e-12)
        x = np.where(mask, scale * q[:, h] @ k[h].T, -np.inf)
        np.testing.assert_allclose(lse[h], scipy.special.logsumexp(x, axis=1), rtol=1e-12, atol=1e-12)


from hypothesis import given, settings, strategies as st


@settings(max_examples=60, deadline=None, derandomize=True)
@given(sizes=st.lists(st.integers(0, 9), min_size=1, max_size=8),
       heads=st.integers(1, 3), head_dim=st.sampled_from([1, 4, 8]),
       scale=st.floats(0.05, 2.0), seed=st.integers(0, 2 ** 16))
def test_attention_matches_scipy_softmax_for_random_layouts(sizes, heads, head_dim, scale, seed):
    """Random block layouts (empty blocks included): every row of the oracle
    equals scipy's softmax over the keys of its own and earlier blocks, with
    the block of each token found by walking the sizes; the unit call on the
    last block gives the same rows as the full sequence."""
    if sum(sizes) == 0:
        sizes = sizes + [1]
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    T = int(offsets[-1])
    rng = _rng(seed)
    q, k, v = _qkv(rng, T, heads, head_dim)
    out, lse = bc.block_causal_attention(q, k, v, offsets, scale)
    ids = _block_ids_by_scan(offsets)
    for i in range(T):
        vis = ids <= ids[i]
        for h in range(heads):
            x = scale * (k[h][vis] @ q[i, h])
            w = scipy.special.softmax(x)
            np.testing.assert_allclose(out[i, h], w @ v[h][vis], rtol=1e-10, atol=1e-12)
            np.testing.assert_allclose(lse[h, i], scipy.special.logsumexp(x), rtol=1e-12, atol=1e-12)
    lo = int(offsets[-2])
    if T > lo:
        out_u, lse_u = bc.unit_attention(q[lo:], k, v, offsets, scale)
        np.testing.assert_array_equal(out_u, out[lo:])
        np.testing.assert_array_equal(lse_u, lse[:, lo:])


def test_one_block_is_full_attention_sdpa():
    rng = _rng(7)
    T, H, D = 37, 4, 16
    q, k, v = _qkv(rng, T, H, D)
    out, _ = bc.block_causal_attention(q, k, v, [0, T])      # default scale 1/sqrt(D)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q).permute(1, 0, 2), torch.from_numpy(k), torch.from_numpy(v))
    np.testing.assert_allclose(out, ref.permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-12)


def test_unit_blocks_are_causal_attention_sdpa():
    rng = _rng(8)
    T, H, D = 29, 2, 8
    q, k, v = _qkv(rng, T, H, D)
    out, _ = bc.block_causal_attention(q, k, v, np.arange(T + 1))
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q).permute(1, 0, 2), torch.from_numpy(k), torch.from_numpy(v), is_causal=True)
    np.testing.assert_allclose(out, ref.permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-12)


def test_zero_query_gives_mean_of_visible_values():
    rng = _rng(9)
    offsets = np.array([0, 4, 4, 9, 11, 16])
    T, H, D = 16, 2, 5
    _, k, v = _qkv(rng, T, H, D)
    q = np.zeros((T, H, D))
    out, lse = bc.block_causal_attention(q, k, v, offsets)
    for i in range(T):
        e = bc.row_limit(offsets, i)
        for h in range(H):
            np.testing.assert_allclose(out[i, h], v[h, :e].mean(axis=0), rtol=1e-13, atol=1e-13)
            np.testing.assert_allclose(lse[h, i], np.log(e), rtol=1e-13)


def test_constant_values_pass_through():
    rng = _rng(10)
    offsets = np.array([0, 3, 10, 12])
    T, H, D = 12, 3, 6
    q, k, _ = _qkv(rng, T, H, D)
    row = rng.standard_normal(D)
    v = np.broadcast_to(row, (H, T, D)).copy()
    out, _ = bc.block_causal_attention(q * 3.0, k, v, offsets)
    np.testing.assert_allclose(out, np.broadcast_to(row, (T, H, D)), rtol=1e-13, atol=1e-13)


def test_default_scale_matches_sdpa_convention():
    assert bc.default_scale(128) == pytest.approx(1 / np.sqrt(128), rel=1e-15)


def test_streaming_invariant_incremental_equals_prefill_exactly():
    rng = _rng(11)
    offsets = _random_offsets(rng, n_blocks=6, max_size=7, allow_empty=False)
    T, H, D = int(offsets[-1]), 2, 8
    q, k, v = _qkv(rng, T, H, D)
    full, full_lse = bc.block_causal_attention(q, k, v, offsets)
    for b in range(len(offsets) - 1):
        lo, hi = offsets[b], offsets[b + 1]
        # the cache holds blocks 0..b (appended before attending); rows past
        # it hold garbage that must never be read
        kc = np.full((H, T + 5, D), np.nan)
        vc = np.full((H, T + 5, D), np.nan)
        kc[:, :hi], vc[:, :hi] = k[:, :hi], v[:, :hi]
        out, lse = bc.unit_attention(q[lo:hi], kc, vc, offsets[:b + 2])
        assert np.array_equal(out, full[lo:hi])
        assert np.array_equal(lse, full_lse[:, lo:hi])


def test_appending_future_blocks_leaves_past_rows_unchanged():
    rng = _rng(12)
    offsets = _random_offsets(rng, n_blocks=8, max_size=6, allow_empty=False)
    T, H, D = int(offsets[-1]), 2, 4
    q, k, v = _qkv(rng, T, H, D)
    B = 5
    past, _ = bc.block_causal_attention(q[:offsets[B]], k[:, :offsets[B]], v[:, :offsets[B]], offsets[:B + 1])
    longer, _ = bc.block_causal_attention(q, k, v, offsets)
    assert np.array_equal(past, longer[:offsets[B]])


# ----------------------------------------------------------------------------
# KV append
# ----------------------------------------------------------------------------

def test_kv_append_rebuilds_timeline_and_touches_nothing_else():
    rng = _rng(13)
    H, D, cap = 3, 4, 40
    sizes = [5, 1, 7, 3]
    T = sum(sizes)
    k_tl = rng.standard_normal((T, H, D))
    v_tl = rng.standard_normal((T, H, D))
    canary = 12345.0
    kc = np.full((H, cap, D), canary)
    vc = np.full((H, cap, D), -canary)
    pos = 0
    for n in sizes:
        kc, vc = kvc.kv_append(kc, vc, k_tl[pos:pos + n], v_tl[pos:pos + n], pos)
        pos += n
    assert np.array_equal(kc[:, :T], k_tl.transpose(1, 0, 2))
    assert np.array_equal(vc[:, :T], v_tl.transpose(1, 0, 2))
    assert (kc[:, T:] == canary).all() and (vc[:, T:] == -canary).all()
    too_many = rng.standard_normal((cap - T + 1, H, D))
    with pytest.raises(ValueError):
        kvc.kv_append(kc, vc, too_many, too_many, T)


# ----------------------------------------------------------------------------
# Flow matching
# ----------------------------------------------------------------------------

def _latents(seed, shape=(16, 64)):
    g = torch.Generator().manual_seed(seed)
    z0 = torch.randn(*shape, generator=g).numpy()          # fp32 values
    eps = torch.randn(*shape, generator=g).numpy()
    return z0, eps


def test_interpolant_endpoints_and_velocity_sign():
    z0, eps = _latents(1)
    assert np.array_equal(fm.interpolant(z0, eps, 1.0), eps.astype(np.float64))
    assert np.array_equal(fm.interpolant(z0, eps, 0.0), z0.astype(np.float64))
    # velocity is the tau-derivative of the interpolant (finite difference
    # of a straight line is exact up to rounding)
    d = (fm.interpolant(z0, eps, 0.75) - fm.interpolant(z0, eps, 0.25)) / 0.5
    np.testing.assert_allclose(d, fm.velocity(z0, eps), rtol=0, atol=1e-14)


def test_one_euler_step_from_noise_recovers_clean_latent_exactly():
    z0, eps = _latents(2)
    z1 = fm.interpolant(z0, eps, 1.0)
    z = fm.euler_step(z1, fm.velocity(z0, eps), 1.0)
    # fp32 inputs: eps - z0 and eps - (eps - z0) are exact in fp64
    assert np.array_equal(z, z0.astype(np.float64))


@pytest.mark.parametrize("n_steps", [2, 4, 7])
def test_uniform_euler_solve_with_exact_velocity_recovers_z0(n_steps):
    z0, eps = _latents(3)
    v = fm.velocity(z0, eps)
    z = fm.euler_solve(eps, lambda z, tau: v, n_steps)
    np.testing.assert_allclose(z, z0, rtol=0, atol=1e-13)


def test_single_step_moves_along_the_straight_path():
    z0, eps = _latents(4)
    v = fm.velocity(z0, eps)
    for tau, dtau in [(1.0, 0.25), (0.75, 0.5), (0.6, 0.1)]:
        z = fm.euler_step(fm.interpolant(z0, eps, tau), v, dtau)
        np.testing.assert_allclose(z, fm.interpolant(z0, eps, tau - dtau), rtol=0, atol=1e-14)


def test_cfg_endpoints_are_the_plain_velocities():
    rng = np.random.default_rng(11)
    vu, vc, z = rng.standard_normal((3, 6, 5))
    # w = 0 is exact; w = 1 computes v_u + (v_c - v_u), equal to v_c up to one
    # fp64 rounding of the difference
    np.testing.assert_array_equal(fm.cfg_velocity(vu, vc, 0.0), vu)
    np.testing.assert_allclose(fm.cfg_velocity(vu, vc, 1.0), vc, rtol=0, atol=1e-15)
    np.testing.assert_array_equal(fm.cfg_euler_step(z, vu, vc, 0.0, 0.25), fm.euler_step(z, vu, 0.25))
    np.testing.assert_allclose(fm.cfg_euler_step(z, vu, vc, 1.0, 0.25), fm.euler_step(z, vc, 0.25),
                               rtol=0, atol=1e-15)


@pytest.mark.parametrize("w", [0.0, 1.0, 3.5, -2.0])
def test_cfg_with_exact_velocity_recovers_z0_for_any_guidance(w):
    # both branches predict the exact velocity eps - z0: guidance changes nothing
    rng = np.random.default_rng(12)
    z0, eps = rng.standard_normal((2, 16, 64))
    v = fm.velocity(z0, eps)
    z = fm.interpolant(z0, eps, 1.0)
    np.testing.assert_allclose(fm.cfg_euler_step(z, v, v, w, 1.0), z0, rtol=0, atol=1e-14)


def test_cfg_velocity_is_affine_in_guidance():
    # v(w) on the line through v(0) = v_u and v(1) = v_c: v(w) = (1 - w) v_u + w v_c
    rng = np.random.default_rng(13)
    vu, vc = rng.standard_normal((2, 7, 3))
    for w in (-1.5, 0.25, 2.0, 7.5):
        np.testing.assert_allclose(fm.cfg_velocity(vu, vc, w), (1 - w) * vu + w * vc, rtol=0, atol=1e-12)


def test_uniform_grid():
    assert np.allclose(fm.uniform_grid(4), [1.0, 0.75, 0.5, 0.25, 0.0])


# ----------------------------------------------------------------------------
# Planted mistakes: a wrong oracle must fail a pin
# ----------------------------------------------------------------------------

def test_planted_mistake_own_block_dropped_is_caught(monkeypatch):
    # a plausible slip: limit = start of own block (strictly causal over blocks)
    def wrong_limit(offsets, i):
        return max(int(np.asarray(offsets)[bc.block_index(offsets, i)]), i + 1)
    monkeypatch.setattr(bc, "row_limit", wrong_limit)
    with pytest.raises(AssertionError):
        test_golden_block_visibility_from_explainer_example()


def test_planted_mistake_transposed_operand_is_caught(monkeypatch):
    orig = bc.attention_rows

    def wrong(q_rows, row_ids, k_cache, v_cache, offsets, scale=None):
        # V read through K's storage (swapped operand)
        return orig(q_rows, row_ids, k_cache, k_cache, offsets, scale)
    monkeypatch.setattr(bc, "attention_rows", wrong)
    with pytest.raises(AssertionError):
        test_attention_matches_bruteforce_mask(0)


def test_planted_mistake_euler_sign_is_caught(monkeypatch):
    monkeypatch.setattr(fm, "euler_step",
                        lambda z, v, dtau: np.asarray(z, np.float64) + dtau * np.asarray(v, np.float64))
    with pytest.raises(AssertionError):
        test_one_euler_step_from_noise_recovers_clean_latent_exactly()


def test_planted_mistake_cfg_swapped_branches_is_caught(monkeypatch):
    # a guidance combination that swaps the branches fails the endpoint pin
    rng = np.random.default_rng(14)
    vu, vc = rng.standard_normal((2, 4, 4))
    monkeypatch.setattr(fm, "cfg_velocity", lambda a, b, w: np.asarray(b) + w * (np.asarray(a) - np.asarray(b)))
    with pytest.raises(AssertionError):
        np.testing.assert_array_equal(fm.cfg_velocity(vu, vc, 0.0), vu)


def test_planted_mistake_dropped_normalisation_is_caught(monkeypatch):
    orig = bc.attention_rows

    def unnormalised(q_rows, row_ids, k_cache, v_cache, offsets, scale=None):
        out, lse = orig(q_rows, row_ids, k_cache, v_cache, offsets, scale)
        lim = np.array([bc.row_limit(offsets, int(i)) for i in row_ids], dtype=np.float64)
        return out * lim[:, None, None], lse          # forgot to divide by l
    monkeypatch.setattr(bc, "attention_rows", unnormalised)
    with pytest.raises(AssertionError):
        test_zero_query_gives_mean_of_visible_values()
