"""Pins for the oracle's counter-based random stream."""
import numpy as np

from conftest import golden_lines
from oracle import rng


def test_splitmix64_matches_published_reference_outputs():
    for line in golden_lines("splitmix64_reference.txt"):
        vals = [int(v) for v in line.split()]
        state, expected = vals[0], vals[1:]
        assert rng.splitmix64_sequence(state, len(expected)) == expected
        # counter form: the i-th output from state s is splitmix64(s + i*gamma)
        for i, e in enumerate(expected):
            assert rng.splitmix64((state + i * rng.GOLDEN_GAMMA) & rng.MASK64) == e


def test_uniform24_exact_range():
    assert rng.uniform24(0) == np.float32(0.0)
    top = rng.uniform24((1 << 64) - 1)
    assert top == np.float32(1.0 - 2.0 ** -24) and top < 1.0
    assert rng.uniform24(1 << 63) == np.float32(0.5)


def test_draw_slots_distinct_and_phase_layout():
    g = 4
    draws = rng.phase_draws(7, 0, 0, g)
    assert len(draws) == 2 * g + 1 and len(set(draws)) == len(draws)
    # phase p, slot s is counter p*(2g+1)+s: the first slot of phase 1 follows
    # the last slot of phase 0 on the same row
    assert rng.draw(7, 0, 1, 0, g) == rng.splitmix64(7 ^ rng.splitmix64(2 * g + 1))
    # rows are separated by 2**32 in the counter
    assert rng.draw(7, 1, 0, 0, g) == rng.splitmix64(7 ^ rng.splitmix64(1 << 32))


def test_uniforms_are_uniform():
    u = np.array([rng.uniform24(rng.draw(3, 0, p, 0, 2)) for p in range(20000)], dtype=np.float64)
    # mean 1/2 and variance 1/12 within 5 standard errors
    n = len(u)
    assert abs(u.mean() - 0.5) < 5 * np.sqrt(1 / 12 / n)
    assert abs(u.var() - 1 / 12) < 5 * np.sqrt(1 / 180 / n)
