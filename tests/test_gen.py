"""The seeded generator: determinism, index addressing, distributions and
the structure of masks, positions and pad rows."""
import numpy as np

import gen


def test_counter_based_and_deterministic():
    a = gen.uniform(3, 2, 1000)
    b = gen.uniform(3, 2, 100, offset=900)
    assert np.array_equal(a[900:], b)
    assert np.array_equal(gen.uniform(3, 2, 10), gen.uniform(3, 2, 10))
    assert not np.array_equal(gen.uniform(3, 2, 10), gen.uniform(3, 1, 10))
    assert not np.array_equal(gen.uniform(3, 2, 10), gen.uniform(4, 2, 10))


def test_splitmix64_known_word():
    # mix(key + 1*golden) for seed 0, stream 0 is the SplitMix64 finaliser
    # applied to 0x9E3779B97F4A7C15 (key = mix(0) = 0): 0xE220A8397B1DCDAF,
    # the first output of SplitMix64 seeded with 0.
    assert int(gen.splitmix64_stream(0, 0, 0)) == 0xE220A8397B1DCDAF


def test_normal_moments():
    z = gen.normal(0, 1, 200000)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1) < 0.01
    assert np.all(np.isfinite(z))


def test_workload_structure():
    w = gen.named_config("pi05")
    assert np.all(w.k()[968:] == 0) and np.all(w.v()[968:] == 0)
    m = w.mask()
    assert m.dtype == np.float16 and m.shape == (10, 1024)
    for t in range(10):
        p = w.pos()[t]
        assert np.all(m[t, :p + 1] == 0) and np.all(np.isneginf(m[t, p + 1:]))
    w3 = gen.named_config("c3")
    assert np.all(np.isneginf(w3.mask()).sum(axis=1) == 204)
    w4 = gen.named_config("long_decode")
    assert list(w4.pos()) == list(range(32752, 32768))
    assert gen.named_config("tiny").mask() is None
