"""Seeded generator: determinism, slicing, statistics (CPU only)."""
import numpy as np

from routing_predicted_experts_gb300 import synth as S


def test_generator_is_counter_based_and_sliceable():
    a = S.normal_f32(3, "t", (1000,), 0.02)
    b = S.normal_f32(3, "t", (400,), 0.02, offset=600)
    assert np.array_equal(a[600:], b)
    assert not np.array_equal(a, S.normal_f32(4, "t", (1000,), 0.02))
    assert not np.array_equal(a, S.normal_f32(3, "u", (1000,), 0.02))


def test_generator_statistics():
    a = S.normal_f32(0, "stats", (400_000,), 1.0).astype(np.float64)
    assert abs(a.mean()) < 0.01
    assert abs(a.std() - 1.0) < 0.01
    assert np.abs(a).max() <= 6.0
    # Irwin-Hall(12) kurtosis is 3 - 0.1 = 2.9
    k = np.mean(a ** 4) / np.mean(a ** 2) ** 2
    assert abs(k - 2.9) < 0.05


def test_uniform_and_bf16_helper():
    u = S.uniform_f64(1, "u", (100_000,))
    assert u.min() >= 0 and u.max() < 1 and abs(u.mean() - 0.5) < 0.01
    assert list(S.bf16_bits(np.array([1.0, 1.0 + 2 ** -8, -2.5], np.float32))) == [0x3F80, 0x3F80, 0xC020]


def test_zipf_logits_are_skewed():
    z = S.zipf_gumbel_logits(0, 512, 256)
    ids = np.argsort(-z, axis=1, kind="stable")[:, :8]
    counts = np.bincount(ids.ravel(), minlength=256)
    assert counts.sum() == 4096
    assert counts.max() > 200 and (counts <= 5).sum() > 50


def test_locality_trace_targets():
    tr = S.locality_trace(0, 3, 512, 256, 4)
    assert tr.shape == (512, 4)
    assert all(len(set(row)) == 4 for row in tr)
    overlap = np.mean([len(set(tr[t]) & set(tr[t - 1])) / 4 for t in range(1, 512)])
    assert 0.15 < overlap < 0.35
