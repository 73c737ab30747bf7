"""Pins for the oracle's token decisions (accept / resample / sampler).

The speculative-sampling rule is fixed by the works the EasySpec pages cite
for speculative decoding (Leviathan et al., "Fast Inference from
Transformers via Speculative Decoding"; Chen et al., "Accelerating Large
Language Model Decoding with Speculative Sampling"): the emitted token is
distributed exactly as p, and a draft token is accepted with total
probability sum_x min(p(x), q(x)).
"""
import numpy as np
import pytest
from scipy import stats

from oracle import rng
from oracle.sampling import (accept_resample, argmax_f32, quantise,
                             sample_quantised, softmax_f32)


def test_quantised_sampler_hand_cdf():
    # weights 1/4, 0, 1/2, 1/4 are exact; T = 2**40, so t = u64 >> 24
    w = np.array([0.25, 0.0, 0.5, 0.25], dtype=np.float32)
    assert list(quantise(w)) == [1 << 38, 0, 1 << 39, 1 << 38]
    cases = [(0, 0), ((1 << 62) - 1, 0), (1 << 62, 2), ((3 << 62) - 1, 2),
             (3 << 62, 3), ((1 << 64) - 1, 3)]
    for u, want in cases:
        assert sample_quantised(w, u) == want, (hex(u), want)
    assert sample_quantised(np.zeros(5, np.float32), 123) == -1


def test_quantised_sampler_is_order_free_exact_inverse_cdf():
    r = np.random.default_rng(0)
    w = r.random(1000).astype(np.float32)
    W = [int(x) for x in quantise(w)]
    T = sum(W)
    for _ in range(200):
        u = int(r.integers(0, 1 << 63)) * 2 + int(r.integers(0, 2))
        t = (u * T) >> 64
        # brute-force linear scan with Python integers
        acc, want = 0, None
        for i, x in enumerate(W):
            acc += x
            if acc > t:
                want = i
                break
        assert sample_quantised(w, u) == want


def test_argmax_lowest_index_on_ties():
    assert argmax_f32([1.0, 3.0, 3.0, -1.0]) == 1
    assert argmax_f32(np.float32([0.0, 0.0])) == 0


def test_softmax_matches_closed_form():
    p = softmax_f32(np.float32([0.0, np.log(3.0)]), 1.0)
    assert np.allclose(p, [0.25, 0.75], atol=1e-7)
    p2 = softmax_f32(np.float32([0.0, np.log(9.0)]), 2.0)
    assert np.allclose(p2, [0.25, 0.75], atol=1e-7)


def _rand_dist(r, V, sharp=1.0):
    z = r.normal(size=V) * sharp
    return softmax_f32(z.astype(np.float32), 1.0)


@pytest.mark.parametrize("V,seed", [(8, 1), (5, 2)])
def test_emitted_token_follows_p_and_accept_rate_closed_form(V, seed):
    r = np.random.default_rng(seed)
    p1 = _rand_dist(r, V)
    q1 = _rand_dist(r, V, 1.5)
    p2 = _rand_dist(r, V)  # bonus distribution (all accepted)
    n = 100_000
    counts = np.zeros(V)
    bonus = np.zeros(V)
    n_acc = 0
    for t in range(n):
        draws = rng.phase_draws(seed, 0, t, 1)
        d = sample_quantised(q1, draws[0])
        a, out = accept_resample(np.stack([p1, p2]), q1[None], [d], draws[1:2], draws[2], False)
        counts[out[0]] += 1
        if a == 1:
            bonus[out[1]] += 1
        n_acc += a
    # first emitted token ~ p1; the bonus token after full acceptance ~ p2
    for c, p in ((counts, p1), (bonus, p2)):
        pe = p.astype(np.float64)
        chi = stats.chisquare(c, c.sum() * pe / pe.sum())
        assert chi.pvalue > 1e-3, chi
    # P(accept) = sum_x min(p, q)
    pa = float(np.minimum(p1, q1).sum())
    assert abs(n_acc / n - pa) < 5 * np.sqrt(pa * (1 - pa) / n)


def test_greedy_rule():
    V = 6
    p = np.zeros((3, V), np.float32)
    q = np.zeros((2, V), np.float32)
    p[0, 2] = 5; p[1, 4] = 5; p[2, 1] = 5
    # both drafts agree with the base argmax -> bonus from p[2]
    assert accept_resample(p, q, [2, 4], None, None, True) == (2, [2, 4, 1])
    # second draft disagrees -> replaced by argmax p[1]
    assert accept_resample(p, q, [2, 3], None, None, True) == (1, [2, 4])
    # first draft disagrees
    assert accept_resample(p, q, [0, 4], None, None, True) == (0, [2])


def test_accept_boundary_is_strict_float32():
    V = 4
    q = np.full((1, V), 0.25, np.float32)
    p = np.zeros((2, V), np.float32)
    p[0, 1] = np.float32(0.125)
    p[1, 0] = 1.0
    # u = 0.5 exactly: u*q = 0.125 == p -> reject (strict <)
    u_half = 1 << 63
    a, out = accept_resample(p, q, [1], [u_half], 0, False)
    assert a == 0
    # u just below 0.5 -> accept
    u_lo = (1 << 63) - (1 << 40)
    a, out = accept_resample(p, q, [1], [u_lo], 0, False)
    assert a == 1 and out == [1, 0]


def test_residual_is_max_p_minus_q():
    # p = (0.5, 0.5, 0, 0), q = (0.5, 0, 0.5, 0): a rejected token must be 1
    p = np.float32([[0.5, 0.5, 0, 0], [1, 0, 0, 0]])
    q = np.float32([[0.5, 0, 0.5, 0]])
    for u in [0, 1 << 60, 1 << 63, (1 << 64) - 1]:
        a, out = accept_resample(p, q, [2], [u], u, False)
        assert a == 0 and out == [1]


def test_zero_residual_falls_back_to_p():
    # p <= q everywhere (only possible through rounding in real runs): a
    # rejection leaves an all-zero residual and the draw is taken from p.
    q = np.float32([[0.5, 0.5]])
    p = np.float32([[0.25, 0.5], [1.0, 0.0]])
    u_rej = (1 << 64) - 1                 # u*q(0) = 0.49999997 >= p(0): reject
    u_bonus = int(0.4 * 2 ** 64)          # from p: t = 0.4*T -> index 1; from q -> 0
    a, out = accept_resample(p, q, [0], [u_rej], u_bonus, False)
    assert a == 0 and out == [1]
