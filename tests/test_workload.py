"""The seeded generator: bf16 rounding, determinism and the planted structure."""
import numpy as np
import pytest
import torch

from sparse_long_context_tail_gb300 import workload as wl


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * s for s in (1e-3, 1, 1e3)])
    x = np.concatenate([x, np.float32([1.00390625, 1.01171875, -1.00390625, 0.0, -0.0])])  # ties
    ours = wl.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    np.testing.assert_array_equal(wl.bf16_bits_to_f32(ours), torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_generation_is_deterministic_and_shaped():
    spec = wl.scaled_spec(wl.named_spec("llama8b-L32768"), [1000, 333], planted=[3, 1])
    a, b = wl.generate(spec), wl.generate(spec)
    np.testing.assert_array_equal(a.k_bits, b.k_bits)
    np.testing.assert_array_equal(a.q_tail_bits, b.q_tail_bits)
    np.testing.assert_array_equal(a.hidden_bits(), b.hidden_bits())
    np.testing.assert_array_equal(a.slots(), b.slots())
    assert a.k_bits.shape == (1333, 8, 128)
    assert a.q_tail_bits.shape == (256, 32, 128)
    assert a.cu_seqlens.tolist() == [0, 1000, 1333]
    assert a.tail_rows.tolist() == list(range(872, 1000)) + list(range(1205, 1333))
    assert sorted(a.slots().tolist()) == list(range(1333))
    assert a.positions().tolist() == list(range(1000)) + list(range(333))
    assert a.hidden_bits().shape == (1333, 4096)


def test_planted_blocks_avoid_sink_and_tail():
    spec = wl.named_spec("small-L4096")
    w = wl.generate(spec)
    blocks = w.planted_blocks[0]
    assert len(blocks) == 4 and len(set(blocks.tolist())) == 4
    assert all(b * 64 >= 128 and (b + 1) * 64 <= 4096 - 128 for b in blocks)


@pytest.mark.parametrize("name", ["small-L4096", "llama8b-L131072", "llama8b-batch16",
                                  "qwen3next-G32-n512", "gemma3-G128-n32"])
def test_named_specs(name):
    s = wl.named_spec(name)
    assert s.num_q_heads % s.num_kv_heads == 0
    if name == "llama8b-batch16":
        assert len(s.lengths) == 16 and all(4096 <= L <= 131072 for L in s.lengths)
        assert s.planted == [max(1, round(64 * L / 131072)) for L in s.lengths]
    assert name in wl.NAMED


def test_q_full_layout_places_tail_rows():
    spec = wl.scaled_spec(wl.named_spec("small-L4096"), [300, 50], planted=[1, 0])
    w = wl.generate(spec)
    q = w.q_full_bits()
    np.testing.assert_array_equal(q[w.tail_rows], w.q_tail_bits)
    assert q.shape == (350, 8, 64)
