"""Seeded input generators: determinism and workload shapes (CPU only)."""
import numpy as np
import torch

from streaming_block_causal_flash_b300.inputs import WORKLOADS, block_offsets, normal


def test_generator_is_deterministic_and_named():
    a = normal(5, "k", 3, (7, 8))
    b = normal(5, "k", 3, (7, 8))
    c = normal(5, "v", 3, (7, 8))
    assert torch.equal(a, b) and not torch.equal(a, c)


def test_bf16_rounding_happens_once_on_the_host():
    x = normal(1, "q", 0, (64, 128), 0.5, torch.bfloat16)
    ref = (normal(1, "q", 0, (64, 128), 1.0, torch.float32) * 0.5).to(torch.bfloat16)
    assert x.dtype == torch.bfloat16 and torch.equal(x, ref)


def test_offsets_shapes_of_every_workload():
    expect_unit = {"tiny_fp32": 16, "unit_192x336": 264, "prefill_128x932": 932}
    for name, w in WORKLOADS.items():
        sizes = w.unit_sizes()
        offs = w.offsets()
        assert offs.dtype == np.int32 and offs[0] == 0 and len(offs) == w.n_units + 1
        assert np.all(np.diff(offs) == sizes)
        assert offs[-1] <= w.capacity()
        if name in expect_unit:
            assert set(sizes) == {expect_unit[name]}
        else:   # 640x368 units: 920 video + 8 audio + 0..16 text
            assert min(sizes) >= 928 and max(sizes) <= 944 and len(set(sizes)) > 1


def test_unit_tensors_do_not_depend_on_what_else_is_drawn():
    w = WORKLOADS["unit_192x336"]
    sizes = w.unit_sizes()
    tl = w.head_timeline("k", 2, 3, sizes)
    assert torch.equal(tl[sizes[0]:sizes[0] + sizes[1]], w.unit_tensor("k", 2, 1, sizes))
    tm = w.token_major("v", 1, sizes)
    assert torch.equal(tm[:, 5, :], w.unit_tensor("v", 5, 1, sizes))


def test_block_offsets_rejects_int32_overflow():
    import pytest
    with pytest.raises(ValueError):
        block_offsets([2**30, 2**30])
