"""The seeded token streams: determinism, ranges, and the laws they claim."""
import numpy as np

import synthdata


def test_splitmix64_reference_values():
    # First outputs of SplitMix64 seeded with 0 (published reference sequence
    # of Vigna's splitmix64.c): 0xe220a8397b1dcdaf, 0x6e789e6aa1b965f4.
    out = synthdata.splitmix64(0, np.arange(2, dtype=np.uint64))
    assert int(out[0]) == 0xE220A8397B1DCDAF
    assert int(out[1]) == 0x6E789E6AA1B965F4


def test_batches_are_deterministic_shifted_windows():
    for kind, V in (("zipf", 50257), ("markov", 65), ("uniform", 65)):
        x, y = synthdata.batch_for(kind, V, 3, 40, 1337)
        x2, y2 = synthdata.batch_for(kind, V, 3, 40, 1337)
        assert x.dtype == np.int32 and x.shape == (3, 40)
        assert np.array_equal(x, x2) and np.array_equal(y, y2)
        assert np.array_equal(x[:, 1:], y[:, :-1])  # targets are inputs shifted by one
        assert x.min() >= 0 and max(x.max(), y.max()) < V
        x3, _ = synthdata.batch_for(kind, V, 3, 40, 1338)
        assert not np.array_equal(x, x3)


def test_zipf_frequencies():
    V = 50257
    x, _ = synthdata.zipf_batch(V, 64, 1024, 7)
    p = synthdata.zipf_pmf(V)
    freq = np.bincount(x.reshape(-1), minlength=V) / x.size
    n = x.size
    for r in range(5):
        assert abs(freq[r] - p[r]) < 5 * np.sqrt(p[r] / n)
    assert 0.13 < p[0] < 0.15  # token 0 is ~13.9% of draws at s = 1.1


def test_markov_stationary_law_is_zipf():
    V = 65
    x, _ = synthdata.markov_batch(V, 2048, 256, 11)
    p = synthdata.zipf_pmf(V)
    freq = np.bincount(x.reshape(-1), minlength=V) / x.size
    assert np.abs(freq - p).max() < 0.02
    # it is a chain, not i.i.d.: repeats far above the i.i.d. rate sum p^2
    rep = np.mean(x[:, 1:] == x[:, :-1])
    assert rep > 2 * np.sum(p ** 2)
