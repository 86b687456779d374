"""Seeded input generators: determinism, ranges and layout."""
import numpy as np

import datagen


def test_splitmix64_counter_form_matches_sequential_steps():
    state = 12345
    seq = []
    for _ in range(5):
        state, z = datagen.splitmix64_scalar(state)
        seq.append(z)
    assert [int(v) for v in datagen.splitmix64(12345, 0, 5)] == seq
    assert [int(v) for v in datagen.splitmix64(12345, 2, 3)] == seq[2:]


def test_streams_are_distinct_and_reproducible():
    a = datagen.uniform_pm1(1001, "A", 1000)
    b = datagen.uniform_pm1(1001, "B", 1000)
    assert not np.array_equal(a, b)
    assert np.array_equal(a, datagen.uniform_pm1(1001, "A", 1000))


def test_uniform_range_and_exactness():
    u = datagen.uniform_pm1(3, "A", 200000)
    assert u.dtype == np.float32
    assert u.min() >= -1.0 and u.max() < 1.0
    assert np.all(u * 2 ** 23 == np.round(u * 2 ** 23))
    assert abs(float(u.mean())) < 0.01 and abs(float(u.std()) - 1 / np.sqrt(3)) < 0.01


def test_normal_moments():
    z = datagen.normal01(4, "B", 400000).astype(np.float64)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1.0) < 0.01


def test_small_ints():
    v = datagen.small_ints(5, "C", 10000)
    assert set(np.unique(v).tolist()) == set(range(-8, 9))


def test_matrix_leading_dimension_gap_is_nan():
    m = datagen.matrix("uniform", 6, "A", 3, 5, ld=8).reshape(3, 8)
    assert np.isnan(m[:, 5:]).all() and np.isfinite(m[:, :5]).all()
    assert np.array_equal(m[:, :5].reshape(-1), datagen.uniform_pm1(6, "A", 15))


def test_chunked_generation_is_split_independent():
    n = (1 << 20) * 2 + 17
    whole = datagen.splitmix64(77, 0, n)
    parts = np.concatenate([datagen.splitmix64(77, 0, 1000), datagen.splitmix64(77, 1000, n - 1000)])
    assert np.array_equal(whole, parts)
