"""Pins for the oracle's speculative loop.

What the pages fix (OpenReview discussion page, first reply, and the arXiv
abstract page): speculative decoding is lossless, so
  * greedy speculative output equals greedy decoding with the base alone, and
  * sampled speculative output follows the base model's distribution;
and calibration replaces the fuzzy draft KV entries with exact ones (reply on
Figure 2), i.e. after calibration the draft cache equals a from-scratch
sequential prefill of the committed tokens.
"""
import copy
import multiprocessing as mp
import os

import numpy as np
import pytest
from scipy import stats

from oracle import model as M
from oracle import spec
from oracle_util import tiny_pair


def _perturbed(W, sigma, seed):
    r = np.random.default_rng(seed)
    out = copy.deepcopy(W)
    for lw in out["layers"]:
        for k, v in lw.items():
            if v.ndim == 2:
                v += r.normal(size=v.shape) * sigma * np.std(v)
    return out


CASES = [(k, mode, g) for k in (1, 2, 3) for mode in (M.ATTN_ONLY, M.FULL_LAYER) for g in (1, 4)]


@pytest.mark.parametrize("k,mode,gamma", CASES)
def test_greedy_speculative_equals_greedy_base(k, mode, gamma):
    Wd, sd, Wb, sb = tiny_pair(10, std=0.3, Ld=5)
    prompts = [[5, 6, 7, 8], [60, 1, 2]]
    want = [spec.seq_decode(Wb, sb, p, 20, 64) for p in prompts]
    dec = spec.SpecDecoder(Wd, sd, Wb, sb, k=k, mode=mode, max_len=64)
    assert dec.generate(prompts, 20, gamma, 0.0) == want


def test_greedy_selfdraft_takes_all_accepted_path():
    # draft = base with small noise: most drafts accepted, bonus path used
    _, _, Wb, sb = tiny_pair(11, std=0.3)
    Wd = _perturbed(Wb, 0.02, 1)
    dec = spec.SpecDecoder(Wd, sb, Wb, sb, k=2, mode=M.FULL_LAYER, max_len=64)
    prompt = [3, 1, 4, 1, 5]
    dec.prefill([prompt])
    accepted = []
    while len(dec.rows[0].tokens) < len(prompt) + 24:
        dec.draft_row(0, 4, 0.0, 0)
        a, _ = dec.verify_row(0, 4, 0.0, 0)
        accepted.append(a)
    assert 4 in accepted
    assert dec.rows[0].tokens[len(prompt):len(prompt) + 24] == spec.seq_decode(Wb, sb, prompt, 24, 64)


@pytest.mark.parametrize("mode,temp", [(M.FULL_LAYER, 0.0), (M.ATTN_ONLY, 1.0)])
def test_calibrated_draft_cache_equals_fresh_prefill(mode, temp):
    Wd, sd, Wb, sb = tiny_pair(12, std=0.3, Ld=5)
    dec = spec.SpecDecoder(Wd, sd, Wb, sb, k=3, mode=mode, max_len=64)
    dec.prefill([[9, 8, 7]])
    r = dec.rows[0]
    for phase in range(6):
        dec.draft_row(0, 4, temp, 5)
        n = r.draft_len  # calibrated prefix [0, n)
        fresh = M.KVCache(sd, 64)
        for pos, t in enumerate(r.tokens[:n]):
            M.forward_exact(Wd, sd, t, pos, fresh)
        assert np.array_equal(r.draft.K[:, :n], fresh.K[:, :n])
        assert np.array_equal(r.draft.V[:, :n], fresh.V[:, :n])
        if phase > 0:
            # the previous phase wrote fuzzy entries past its committed prefix
            assert n > 3
        dec.verify_row(0, 4, temp, 5)


def test_base_cache_matches_committed_tokens():
    Wd, sd, Wb, sb = tiny_pair(13, std=0.3)
    dec = spec.SpecDecoder(Wd, sd, Wb, sb, k=2, max_len=64)
    dec.generate([[1, 2, 3]], 12, 3, 1.0, seed=9)
    r = dec.rows[0]
    n = len(r.tokens)
    fresh = M.KVCache(sb, 64)
    for pos, t in enumerate(r.tokens[: n - 1]):
        M.forward_exact(Wb, sb, t, pos, fresh)
    assert np.array_equal(r.base.K[:, : n - 1], fresh.K[:, : n - 1])


def test_vocab_mismatch_rejected():
    Wd, sd, Wb, sb = tiny_pair(14)
    with pytest.raises(ValueError):
        spec.SpecDecoder(Wd, sd._replace(vocab=65) if hasattr(sd, "_replace")
                         else M.Shape(**{**sd.__dict__, "vocab": 65}), Wb, sb)


# ------------------------------------------------ distribution (chi-square)

_G = {}


def _init_worker(args):
    _G["args"] = args


def _run_chunk(seeds):
    Wd, sd, Wb, sb, groups, mode, prompt, gamma = _G["args"]
    dec = spec.SpecDecoder(Wd, sd, Wb, sb, groups=groups, mode=mode, max_len=16)
    V = sb.vocab
    counts = np.zeros(V ** 3, np.int64)
    for s in seeds:
        out = dec.generate([prompt], 3, gamma, 1.0, seed=int(s))[0]
        counts[(out[0] * V + out[1]) * V + out[2]] += 1
    return counts


N_DRAWS = int(os.environ.get("ES_CHISQ_DRAWS", "100000"))


@pytest.mark.slow
@pytest.mark.parametrize("mode", [M.FULL_LAYER, M.ATTN_ONLY])
def test_sampled_output_follows_base_distribution(mode):
    """Joint law of the first three emitted tokens over N_DRAWS seeded runs
    vs the brute-force base distribution (V = 8, so 512 cells).  With
    gamma = 2 the three tokens cover the accepted, resampled and bonus
    (all-accepted) outcomes of the first phase."""
    Wd, sd, Wb, sb = tiny_pair(20, V=8, d=8, Ld=3, Lb=2, H=2, Hkv=1, F=8, std=0.5)
    prompt, gamma = [1, 2, 3], 2
    p1 = spec.exact_next_dist(Wb, sb, prompt, 1.0)
    joint = []
    for a in range(8):
        p2 = spec.exact_next_dist(Wb, sb, prompt + [a], 1.0)
        for b in range(8):
            p3 = spec.exact_next_dist(Wb, sb, prompt + [a, b], 1.0)
            joint.append(p1[a] * p2[b] * p3)
    joint = np.concatenate(joint)
    args = (Wd, sd, Wb, sb, [[0], [1, 2]], mode, prompt, gamma)
    nproc = max(1, min(os.cpu_count() or 1, 16))
    chunks = np.array_split(np.arange(N_DRAWS), nproc * 4)
    with mp.get_context("spawn").Pool(nproc, initializer=_init_worker, initargs=(args,)) as pool:
        counts = sum(pool.map(_run_chunk, chunks))
    exp = joint * N_DRAWS
    keep = exp >= 5
    obs = np.append(counts[keep], counts[~keep].sum())
    ex = np.append(exp[keep], exp[~keep].sum())
    chi = stats.chisquare(obs, ex * obs.sum() / ex.sum())
    assert chi.pvalue > 1e-3, (chi, counts, exp)


# ------------------------------------------------ calibration ablation
# Without calibration the accepted drafts keep the entries their layer-parallel
# forwards wrote (the pages' ablation: the fuzzy errors then accumulate). The
# rule itself fixes three checkable facts.

@pytest.mark.parametrize("k,mode", [(2, M.FULL_LAYER), (3, M.ATTN_ONLY)])
def test_no_calibration_greedy_still_lossless(k, mode):
    # losslessness does not depend on the draft's cache
    Wd, sd, Wb, sb = tiny_pair(10, std=0.3, Ld=5)
    prompts = [[5, 6, 7, 8], [60, 1, 2]]
    want = [spec.seq_decode(Wb, sb, p, 20, 64) for p in prompts]
    dec = spec.SpecDecoder(Wd, sd, Wb, sb, k=k, mode=mode, max_len=64, calibrate=False)
    assert dec.generate(prompts, 20, 4, 0.0) == want


@pytest.mark.parametrize("temp", [0.0, 1.0])
def test_no_calibration_with_exact_drafts_changes_nothing(temp):
    # with one-layer sets every draft forward is exact, so the kept entries
    # are the calibrated ones: tokens and draft logits must be identical.
    # A self-draft pair makes every draft accepted often, which exercises the
    # d_gamma row (no entry of its own) of the narrowed calibration window.
    _, _, Wb, sb = tiny_pair(11, std=0.3)
    Wd = _perturbed(Wb, 0.02, 1)
    runs = {}
    for cal in (True, False):
        dec = spec.SpecDecoder(Wd, sb, Wb, sb, k=1, max_len=96, calibrate=cal)
        dec.prefill([[3, 1, 4, 1, 5]])
        zq, acc = [], []
        for _ in range(8):
            dec.draft_row(0, 4, temp, 7)
            zq.append(dec.rows[0].zq.copy())
            acc.append(dec.verify_row(0, 4, temp, 7)[0])
        runs[cal] = (dec.rows[0].tokens, zq, acc)
    assert 4 in runs[True][2]
    assert runs[True][0] == runs[False][0]
    assert all(np.array_equal(a, b) for a, b in zip(runs[True][1], runs[False][1]))


@pytest.mark.parametrize("mode", [M.FULL_LAYER, M.ATTN_ONLY])
def test_no_calibration_cache_keeps_accepted_fuzzy_entries(mode):
    # Replay the committed tokens position by position, taking the layer-
    # parallel forward exactly at the positions whose drafts were accepted and
    # had been draft inputs (d_1..d_min(a, gamma-1) of each phase), the exact
    # one elsewhere. Each forward reads only earlier positions, so the replay
    # must reproduce the draft cache bit for bit.
    _, _, Wb, sb = tiny_pair(15, std=0.3, Lb=6)
    Wd = _perturbed(Wb, 0.02, 2)
    gamma = 4
    dec = spec.SpecDecoder(Wd, sb, Wb, sb, k=2, mode=mode, max_len=96, calibrate=False)
    assert any(len(g) > 1 for g in dec.groups)
    dec.prefill([[2, 7, 1, 8]])
    r = dec.rows[0]
    fuzzy_pos, accepted = set(), []
    for _ in range(8):
        n = len(r.tokens)
        dec.draft_row(0, gamma, 0.0, 3)
        a, _ = dec.verify_row(0, gamma, 0.0, 3)
        accepted.append(a)
        fuzzy_pos.update(range(n, n + min(a, gamma - 1)))
    dec.draft_row(0, gamma, 0.0, 3)   # the narrowed calibration of the last commits
    n = r.draft_len
    assert n == len(r.tokens) and len(fuzzy_pos) >= 3, accepted
    replay = M.KVCache(sb, 96)
    for pos, t in enumerate(r.tokens[:n]):
        if pos in fuzzy_pos:
            M.forward_fuzzy(Wd, sb, t, pos, replay, dec.groups, mode)
        else:
            M.forward_exact(Wd, sb, t, pos, replay)
    assert np.array_equal(r.draft.K[:, :n], replay.K[:, :n])
    assert np.array_equal(r.draft.V[:, :n], replay.V[:, :n])
    # and the kept entries are not the exact ones
    exact = M.KVCache(sb, 96)
    for pos, t in enumerate(r.tokens[:n]):
        M.forward_exact(Wd, sb, t, pos, exact)
    p = min(fuzzy_pos)
    assert not np.allclose(r.draft.K[:, p], exact.K[:, p])


@pytest.mark.parametrize("temp", [0.0, 1.0])
def test_block_forwards_leave_the_loop_unchanged(temp):
    """The loop with its exact multi-token forwards run as block forwards
    (prefill, calibration, verify) emits the same tokens and the same logits
    to rounding as the token-by-token loop, and its calibrated draft cache
    still equals a fresh sequential prefill."""
    Wd, sd, Wb, sb = tiny_pair(12, std=0.3, Ld=5)
    prompts = [[5, 6, 7, 8, 9, 10, 11], [60, 1, 2]]
    a = spec.SpecDecoder(Wd, sd, Wb, sb, k=2, mode=M.FULL_LAYER, max_len=64)
    b = spec.SpecDecoder(Wd, sd, Wb, sb, k=2, mode=M.FULL_LAYER, max_len=64, block=True)
    a.prefill(prompts)
    b.prefill(prompts)
    for ph in range(5):
        for r in range(2):
            da = a.draft_row(r, 4, temp, 3)
            db = b.draft_row(r, 4, temp, 3)
            assert da == db
            assert np.max(np.abs(a.rows[r].zq - b.rows[r].zq)) < 1e-10
            assert a.verify_row(r, 4, temp, 3) == b.verify_row(r, 4, temp, 3)
            assert np.max(np.abs(a.rows[r].zp - b.rows[r].zp)) < 1e-10
    r = b.rows[0]
    b.calibrate_row(r)
    fresh = M.KVCache(sd, 64)
    for pos, t in enumerate(r.tokens):
        M.forward_exact(Wd, sd, t, pos, fresh)
    n = len(r.tokens)
    assert np.max(np.abs(r.draft.K[:, :n] - fresh.K[:, :n])) < 1e-11
