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
