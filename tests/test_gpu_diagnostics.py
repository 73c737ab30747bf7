"""The fuzzy-drafting error diagnostic on a small bf16 self-draft pair.

Draft sets for 6 layers and k = 2 are {0}, {1}, {2, 3}, {4}, {5}. Layers 0
to 2 see exact inputs in the fuzzy forward, so their fuzzy K/V entries equal
the calibrated ones up to rounding. Layer 3 reads its set's input instead of
layer 2's output. Layers 4 and 5 read the set's summed output, so they carry
the error too.

The calibration ablation must change nothing, up to float32 rounding, when
every draft set has one layer (k = 1: the draft forwards are exact, so a kept
entry is the one calibration would write), and it must report every phase it
ran.
"""
import pytest

from gpu_util import Pair
from layer_drafting_draft_b300 import synth
from layer_drafting_draft_b300.diagnostics import calibration_ablation, fuzzy_kv_error
from layer_drafting_draft_b300.easyspec import ES_FULL_LAYER

pytestmark = pytest.mark.gpu


def test_only_the_fuzzy_layer_departs_from_exact():
    s = synth.shape(6, 256, 4, 2, 688, 1000, 1e4)
    pair = Pair(s, s, "bf16", 31, sigma=0.02)
    prompt = synth.make_prompts(1, 24, 1000, 32).numpy()
    g = pair.gpu(max_seq=256, mode=ES_FULL_LAYER)
    res = fuzzy_kv_error(g, s, prompt, k=2, gamma=4, phases=12, temperature=0.0)
    g.close()
    assert res[0]["n"] > 0, res
    exact = [0, 1, 2]
    for l in exact:
        assert res[l]["cos_k"] > 0.999 and res[l]["rel_k"] < 0.05, (l, res[l])
    floor = max(res[l]["rel_k"] for l in exact)
    for l in (3, 4, 5):
        assert res[l]["rel_k"] > 3 * floor + 1e-3, (l, res)


def test_ablation_with_exact_drafts_is_a_no_op():
    s = synth.shape(6, 256, 4, 2, 688, 1000, 1e4)
    pair = Pair(s, s, "f32", 33, sigma=0.05)
    prompts = synth.make_prompts(3, 16, 1000, 34).numpy()
    g = pair.gpu(max_seq=128, mode=ES_FULL_LAYER)
    res = calibration_ablation(g, prompts, k=1, gamma=4, max_new=40, temperature=0.0)
    g.close()
    # equal up to float32 rounding of near-tied argmaxes (a wrongly kept or
    # missing entry would cost far more than this at this acceptance)
    assert abs(res["on"]["accepted_per_phase"] - res["off"]["accepted_per_phase"]) <= 0.1, res
    assert res["on"]["phases"] == sum(b["phases"] for b in res["on"]["bins"]) > 0
    assert res["on"]["accepted_per_phase"] > 0.5, res


def test_fuzzy_kv_error_matches_the_oracle():
    """The diagnostic's per-layer figures against the same figures computed
    from the oracle's caches (OpenReview discussion page, reply on Table 3:
    fuzzy against exact states, layer by layer).

    The oracle replays the GPU run: the GPU's draft tokens and accept
    decisions are forced on it, so both sides write fuzzy entries for the
    same tokens at the same positions and then recompute them exactly in
    the next calibration.  The cosine and relative error of fuzzy against
    exact K and V, per layer, must agree within bf16 rounding."""
    import numpy as np

    s = synth.shape(6, 256, 4, 2, 688, 1000, 1e4)
    pair = Pair(s, s, "bf16", 35, sigma=0.02)
    prompt = synth.make_prompts(1, 24, 1000, 36).numpy()
    gamma, phases, k = 4, 12, 2
    g = pair.gpu(max_seq=256, mode=ES_FULL_LAYER)
    trace = []
    res = fuzzy_kv_error(g, s, prompt, k=k, gamma=gamma, phases=phases, temperature=0.0, trace=trace)
    g.close()
    assert len(trace) == phases

    o = pair.oracle(k=k, mode=ES_FULL_LAYER, max_len=256)
    o.prefill(prompt.tolist())
    r = o.rows[0]
    L = s["n_layers"]
    sums = np.zeros((L, 4))
    count = 0
    pending = None
    for ph in range(phases + 1):
        n = len(r.tokens)
        o.draft_row(0, gamma, 0.0, ph, force_d=trace[ph][0] if ph < phases else None)
        if pending is not None:            # calibration just rewrote the kept positions
            pos, kf, vf = pending
            for l in range(L):
                for i, p in enumerate(pos):
                    for j, (f, e) in enumerate(((kf[l][i], r.draft.K[l, p]), (vf[l][i], r.draft.V[l, p]))):
                        f, e = f.ravel(), e.ravel()
                        sums[l, j] += f @ e / (np.linalg.norm(f) * np.linalg.norm(e))
                        sums[l, 2 + j] += np.linalg.norm(f - e) / np.linalg.norm(e)
            count += len(pos)
            pending = None
        if ph == phases:
            break
        d, a, toks = trace[ph]
        kept = list(range(n, n + min(a, gamma - 1)))
        if kept:
            pending = (kept, [r.draft.K[l, kept].copy() for l in range(L)],
                       [r.draft.V[l, kept].copy() for l in range(L)])
        o.verify_row(0, gamma, 0.0, ph, force=(a, toks))
    assert count == res[0]["n"] and count > 0
    mean = sums / count
    for l in range(L):
        want = dict(zip(("cos_k", "cos_v", "rel_k", "rel_v"), mean[l]))
        for key, w in want.items():
            got = res[l][key]
            tol = 0.01 + (0.05 * w if key.startswith("rel") else 0.0)
            assert abs(got - w) <= tol, (l, key, got, w)
    print("per-layer (GPU, oracle) rel_k:", [(round(res[l]["rel_k"], 4), round(mean[l, 2], 4)) for l in range(L)])
