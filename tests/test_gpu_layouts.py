"""Layouts the default rule never produces, on the CUDA path, against the
oracle with the same sets (float32: emitted tokens bit-exact).

The first and last layers inside sets, non-uniform sizes, the other reading
of the rule (OpenReview discussion page, reply on Table 4 / Appendix B.1: the
authors expect other combinations to need only a configuration change).
The search runs end to end on a small pair.
"""
import pytest

from gpu_util import Pair
from layer_drafting_draft_b300 import layouts as LY
from layer_drafting_draft_b300 import synth
from layer_drafting_draft_b300.easyspec import ES_ATTN_ONLY, ES_FULL_LAYER

pytestmark = pytest.mark.gpu

BASE = synth.WORKLOADS["tiny_f32"]["base"]   # 8 layers


@pytest.fixture(scope="module")
def selfdraft():
    return Pair(BASE, BASE, "f32", 5, sigma=0.1)


LAYOUTS = [LY.with_ends(8, 4), LY.by_sizes([3, 1, 4]), LY.from_one(8, 3), LY.tapered(8, 4),
           LY.by_sizes([8])]


@pytest.mark.parametrize("sets", LAYOUTS, ids=[LY.name(s) for s in LAYOUTS])
@pytest.mark.parametrize("mode", [ES_FULL_LAYER, ES_ATTN_ONLY])
def test_layout_bit_exact(selfdraft, sets, mode):
    prompt = synth.make_prompts(1, 24, 512, 8).numpy()
    g = selfdraft.gpu(mode=mode, groups=sets)
    out, st = g.generate(prompt, 48, 5, 0, 1.0, 321)
    o = selfdraft.oracle(groups=sets, mode=mode)
    want = o.generate(prompt.tolist(), 48, 5, 1.0, seed=321)
    assert out[0].tolist() == want[0]
    assert st["accepted"] > 0
    g.close()


def test_search_end_to_end(selfdraft):
    wl = {"draft": BASE, "base": BASE, "dtype": "f32"}
    prompts = synth.make_prompts(2, 16, 512, 9).numpy()
    cands = {k: v for k, v in LY.candidates(8, sizes=(2, 4)).items()
             if k in ("sequential", "aligned4", "with_ends4")}
    rows = LY.search(LY.gpu_measure(wl, selfdraft.wd, selfdraft.wb, prompts, ES_FULL_LAYER, 4, 32, 1.0),
                     cands)
    assert [r["layout"] for r in rows] and len(rows) == 3
    assert all(r["tok_s"] > 0 and 1.0 <= r["tokens_per_phase"] <= 5.0 for r in rows)
