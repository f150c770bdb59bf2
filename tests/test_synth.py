"""The seeded generator: reproducible, independent of the thread split, and
distributed as drawn (mean / variance within a few standard errors)."""
import numpy as np

import synth


def test_normal_moments_and_reproducible():
    a = synth.normal_bf16(0, 11, (1 << 20,), 0.02)
    b = synth.normal_bf16(0, 11, (1 << 20,), 0.02)
    assert np.array_equal(a, b)
    x = synth.bf16_to_f32(a).astype(np.float64)
    n = x.size
    assert abs(x.mean()) < 4 * 0.02 / np.sqrt(n)
    assert abs(x.var() / 0.02 ** 2 - 1) < 4 * np.sqrt(2 / n) + 2 ** -8
    # Box-Muller tails: about 0.27% beyond 3 sigma
    frac = np.mean(np.abs(x) > 3 * 0.02)
    assert 0.002 < frac < 0.0035


def test_streams_and_elements_independent_of_split():
    big = synth.normal_bf16(3, 12, (200000,))
    small = synth.normal_bf16(3, 12, (1000,))
    assert np.array_equal(big[:1000], small)
    other = synth.normal_bf16(3, 13, (1000,))
    assert not np.array_equal(other, small)
    f = synth.normal_f32(3, 12, (1000,))
    assert np.array_equal((f.view(np.uint32) + 0x7FFF + ((f.view(np.uint32) >> 16) & 1)) >> 16,
                          small.astype(np.uint32))


def test_uniform_int_range():
    t = synth.uniform_int(0, 4, 100000, 32000)
    assert t.min() >= 0 and t.max() < 32000
    assert abs(t.mean() - 16000) < 4 * 32000 / np.sqrt(12 * 100000)
