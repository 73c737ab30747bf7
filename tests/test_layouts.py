"""Layer-set layouts and the layout search (host logic, no GPU).

The default rule is pinned to the page's own 32-layer, N = 4 example
(OpenReview discussion page, reply on Table 4 / Appendix B.1;
tests/golden/grouping_L32_N4.txt) and to the oracle's independent
implementation of the same rule. The variants are checked against their
definitions on small cases written out by hand.
"""
import os

import pytest

from layer_drafting_draft_b300 import layouts as LY
from oracle import model as M

GOLD = os.path.join(os.path.dirname(__file__), "golden", "grouping_L32_N4.txt")


def _golden():
    with open(GOLD) as f:
        return [[int(x) for x in ln.split()] for ln in f if ln.strip() and not ln.startswith("#")]


def test_aligned_matches_the_pages_example():
    assert LY.aligned(32, 4) == _golden()


@pytest.mark.parametrize("L", [1, 2, 3, 5, 8, 16, 24, 28, 32, 80])
@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 8])
def test_aligned_agrees_with_the_oracle_rule(L, N):
    assert LY.aligned(L, N) == M.default_groups(L, N)


def test_variants_on_hand_written_cases():
    assert LY.from_one(32, 4)[:3] == [[0], [1, 2, 3, 4], [5, 6, 7, 8]]
    assert LY.from_one(32, 4)[-3:] == [[25, 26, 27, 28], [29, 30], [31]]
    assert LY.with_ends(10, 4) == [[0, 1, 2, 3], [4, 5, 6, 7], [8, 9]]
    assert LY.tapered(16, 4) == LY.by_sizes([1, 2, 4, 4, 2, 2, 1])
    assert LY.tapered(8, 4) == LY.by_sizes([1, 2, 2, 2, 1])
    assert LY.by_sizes([3, 1, 4]) == [[0, 1, 2], [3], [4, 5, 6, 7]]
    assert LY.starts(LY.by_sizes([3, 1, 4])) == [0, 3, 4]
    assert LY.name(LY.by_sizes([1, 3])) == "0|1-3"


@pytest.mark.parametrize("L", [4, 8, 16, 24, 28, 32])
def test_every_generated_layout_is_valid(L):
    for f in (LY.aligned, LY.from_one, LY.with_ends, LY.tapered):
        for N in (1, 2, 3, 4, 8):
            LY.check(f(L, N), L)
    c = LY.candidates(L)
    assert c["sequential"] == [[l] for l in range(L)]
    assert len({LY.name(s) for s in c.values()}) == len(c)


def test_check_rejects_bad_layouts():
    for bad in ([[0, 1], [3]], [[0], [0, 1], [2, 3]], [[1, 0], [2, 3]], [list(range(9)), [9]]):
        with pytest.raises(ValueError):
            LY.check(bad, 10 if bad[-1] == [9] else 4)


def test_search_ranks_by_decode_rate():
    # fake measurements: tokens per phase grows with the mean set size
    # less slowly than time per phase falls
    def measure(sets):
        k = 16 / len(sets)
        return {"tokens": 100 * (3.0 - 0.2 * k), "phases": 100, "ms": 100 * (2.0 / k + 1.0), "useful": 240}
    rows = LY.search(measure, LY.candidates(16, sizes=(2, 4)))
    rates = [r["tok_s"] for r in rows]
    assert rates == sorted(rates, reverse=True)
    assert rows[-1]["layout"] == "sequential"
    r = rows[0]
    assert r["tok_s"] == pytest.approx(240 / (r["ms_per_phase"] * 100 / 1e3))


# ------------------------------------------------ the library's own rule
# es_layer_sets returns the set starts the CUDA path's planner uses when no
# explicit sets are configured (host only, no GPU).

def test_library_rule_matches_the_pages_example():
    from layer_drafting_draft_b300.easyspec import layer_sets
    assert layer_sets(32, 4) == LY.starts(_golden())


@pytest.mark.parametrize("L", [1, 2, 3, 5, 8, 16, 24, 28, 32, 80])
@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 8])
def test_library_rule_agrees_with_the_oracle(L, N):
    from layer_drafting_draft_b300.easyspec import layer_sets
    assert layer_sets(L, N) == LY.starts(M.default_groups(L, N))


def test_library_rule_rejects_bad_arguments():
    from layer_drafting_draft_b300.easyspec import EasySpecError, layer_sets
    for L, N in ((0, 4), (8, 0), (8, 9)):
        with pytest.raises(EasySpecError):
            layer_sets(L, N)
