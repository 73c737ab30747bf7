"""The fuzzy-drafting error diagnostic on a small bf16 self-draft pair.

Draft sets for 6 layers and k = 2 are {0}, {1}, {2, 3}, {4}, {5}. Layers 0
to 2 see exact inputs in the fuzzy forward, so their fuzzy K/V entries equal
the calibrated ones up to rounding. Layer 3 reads its set's input instead of
layer 2's output. Layers 4 and 5 read the set's summed output, so they carry
the error too.
"""
import pytest

from gpu_util import Pair
from layer_drafting_draft_b300 import synth
from layer_drafting_draft_b300.diagnostics import fuzzy_kv_error
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
