"""The seeded input generator: deterministic, thread-count independent, and
drawing the distributions the model configurations name."""
import numpy as np

import synth


def test_deterministic_and_thread_independent(monkeypatch):
    a = synth.normal_f32(42, 3, (1000,), 0.0, 0.02)
    monkeypatch.setattr(synth, "_threads", lambda: 1)
    b = synth.normal_f32(42, 3, (1000,), 0.0, 0.02)
    q1, s1 = synth.int8_rows(42, 5, 17, 300)
    monkeypatch.setattr(synth, "_threads", lambda: 7)
    q2, s2 = synth.int8_rows(42, 5, 17, 300)
    assert np.array_equal(a, b) and np.array_equal(q1, q2) and np.array_equal(s1, s2)
    assert not np.array_equal(a, synth.normal_f32(43, 3, (1000,), 0.0, 0.02))


def test_normal_moments():
    x = synth.normal_f32(1, 1, (400000,), 0.0, 0.02).astype(np.float64)
    assert abs(x.mean()) < 1e-4 and abs(x.std() - 0.02) < 2e-4
    assert abs(((x / 0.02) ** 4).mean() - 3.0) < 0.05  # Gaussian kurtosis


def test_int8_rows_recipe():
    q, s = synth.int8_rows(2, 9, 64, 4096, 0.02)
    assert np.all(np.abs(q.astype(np.int32)).max(axis=1) == 127)
    # scale ~ max|w|/127 with max over 4096 draws of N(0, 0.02) ~ 3.5-4.5 sigma
    assert np.all((s > 0.02 * 3.0 / 127) & (s < 0.02 * 5.5 / 127))


def test_tokens_range_and_spread():
    t = synth.tokens(5, 100000, 1024)
    assert t.min() >= 0 and t.max() < 1024
    counts = np.bincount(t, minlength=1024)
    assert counts.min() > 50 and counts.max() < 160


def test_config_byte_counts():
    # int8 non-embedding bytes per configuration, from the layer shapes
    c = synth.CONFIGS
    assert c["tiny"].layer_bytes() * 4 == 3_407_872
    assert c["350m"].layer_bytes() * 24 == 377_487_360
    assert c["1b"].layer_bytes() * 16 == 973_078_528
    assert c["8b"].layer_bytes() * 32 == 6_979_321_856
