"""The seeded input generator: determinism, random access, distribution."""
import numpy as np

import synth


def test_known_words():
    # fmix32 is MurmurHash3's finaliser: fmix32(0) = 0 and fmix32(1) = 0x514E28B7
    assert int(synth.fmix32(np.array([0], np.uint32))[0]) == 0
    assert int(synth.fmix32(np.array([1], np.uint32))[0]) == 0x514E28B7


def test_random_access_matches_full_tensor():
    full = synth.normal(77, (37, 96), 0.02)
    rows = [0, 5, 36, 17]
    assert np.array_equal(synth.weight_rows(77, 37, 96, rows), full[rows])


def test_values_exact_in_binary32():
    z = synth.normal_z(3, np.arange(10000))
    assert np.array_equal(z * np.float32(65536.0), np.round(z * np.float32(65536.0)))
    assert np.abs(z).max() <= 6.0


def test_moments():
    z = synth.normal_z(9, np.arange(2_000_000)).astype(np.float64)
    assert abs(z.mean()) < 0.005
    assert abs(z.var() - 1.0) < 0.01
    # Irwin-Hall(12) kurtosis is 3 - 1.2/12 = 2.9
    k = ((z - z.mean()) ** 4).mean() / z.var() ** 2
    assert abs(k - 2.9) < 0.02


def test_outliers_exact_count():
    K = 3584
    x = synth.activation(5, 3, K, outlier_frac=0.001).astype(np.float64)
    base = synth.activation(5, 3, K).astype(np.float64)
    for m in range(3):
        changed = np.nonzero(x[m] != base[m])[0]
        assert changed.size <= synth.n_outliers(K, 0.001) == 4
    assert synth.n_outliers(18944, 0.001) == 19


def test_seeds_differ():
    a = synth.normal(1, (4, 64))
    b = synth.normal(2, (4, 64))
    assert not np.array_equal(a, b)
    assert np.array_equal(a, synth.normal(1, (4, 64)))


def test_host_twin_matches_numpy():
    """The C host twin draws the same bits as the numpy definition, whatever
    the thread split and the counter offset."""
    for seed, shape, sigma, offset, threads in [(3, (37, 96), 0.02, 0, 1), (1004, (5, 3584), 0.02, 12345, 3),
                                                (7, (1000,), 1.0, 2 ** 32 - 1000, 8), (0, (1, 1), 0.5, 0, 4)]:
        a = synth.normal_host(seed, shape, sigma, offset=offset, threads=threads)
        b = synth.normal(seed, shape, sigma, offset=offset)
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    rows = [0, 511, 1999]
    full = synth.normal_host(1006, (2000, 512), 0.02)
    assert np.array_equal(full[rows].view(np.uint32), synth.weight_rows(1006, 2000, 512, rows).view(np.uint32))
