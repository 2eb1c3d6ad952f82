"""The seeded input generators: bf16 rounding, determinism, routing recipes."""
import numpy as np
import pytest

import moe_inputs as mi


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    r = np.random.default_rng(0)
    v = np.concatenate([r.standard_normal(100000).astype(np.float32) * 3,
                        np.array([0.0, -0.0, 1.0, 1.00390625, 1.01171875, 65504.0, 1e-30], np.float32)])
    ours = mi.f32_to_bf16_bits(v)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    np.testing.assert_array_equal(mi.bf16_bits_to_f32(ours), torch.from_numpy(v).to(torch.bfloat16).float().numpy())


def test_generators_are_deterministic():
    a, b = mi.make("tiny"), mi.make("tiny")
    np.testing.assert_array_equal(a.x, b.x)
    np.testing.assert_array_equal(a.topk_ids, b.topk_ids)
    np.testing.assert_array_equal(a.W1, b.W1)
    np.testing.assert_array_equal(a.expert_W2(3), b.W2[3])


def test_uniform_routing_distinct_and_in_range():
    p = mi.make("tiny")
    s = p.shape
    assert p.topk_ids.shape == (s.T, s.K)
    assert all(len(set(row)) == s.K for row in p.topk_ids.tolist())
    assert p.topk_ids.min() >= 0 and p.topk_ids.max() < s.E
    w = mi.bf16_bits_to_f32(p.topk_weights)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, atol=2e-2)


def test_zipf_routing_skew_and_empty_experts():
    r = np.random.default_rng(1)
    ids = mi.zipf_ids(np.random.default_rng(2), np.random.default_rng(3), 16384, 32, 8)
    assert all(len(set(row)) == 8 for row in ids[:500].tolist())
    counts = np.bincount(ids.reshape(-1), minlength=32)
    assert (counts == 0).sum() >= 3
    assert counts.max() > 8 * counts[counts > 0].min()
