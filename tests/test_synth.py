"""The shared input generator: counter-mode determinism and distributions."""
import numpy as np

import synth


def test_counter_mode_slices_match():
    full = synth.normal_f16((1000,), 0, 7, 0.02)
    part = synth.normal_f16((300,), 0, 7, 0.02, offset=500)
    assert np.array_equal(full[500:800], part)


def test_streams_and_seeds_differ():
    a = synth.normal_f16((256,), 0, 1, 1.0)
    b = synth.normal_f16((256,), 0, 2, 1.0)
    c = synth.normal_f16((256,), 1, 1, 1.0)
    assert not np.array_equal(a, b) and not np.array_equal(a, c)
    assert np.array_equal(a, synth.normal_f16((256,), 0, 1, 1.0))


def test_normal_moments():
    w = synth.weights(256, 1024, 0, 3).view(np.float16).astype(np.float64)
    assert abs(w.mean()) < 3e-4
    assert abs(w.std() - 0.02) < 3e-4
    x = synth.activations(1 << 16, 0, 4).view(np.float16).astype(np.float64)
    assert abs(x.std() - 1.0) < 0.02
    # a Gaussian has about 4.55% of its mass beyond 2 sigma
    assert 0.04 < np.mean(np.abs(x) > 2.0) < 0.051


def test_small_integers_exact():
    v = synth.int_f16((4096,), 0, 5, -8, 8, -6).view(np.float16).astype(np.float64)
    k = v * 64.0
    assert np.array_equal(k, np.round(k)) and k.min() == -8 and k.max() == 8
    assert len(np.unique(k)) == 17


def test_sample_rows_cover_ends():
    ids = synth.sample_rows(57344, 64, 0, 9)
    assert ids[0] == 0 and ids[-1] == 57343 and len(ids) == 64 and len(set(ids)) == 64
