"""Edge cases of the CUDA path against the oracle (float32: tokens bit-exact).

* Prompts of one and two tokens: nothing is prefilled before the first phase,
  and the first calibration window (gamma + 1 rows) is mostly inactive rows.
* gamma = 1: no layer-parallel forward at all; verify over two rows.
* gamma = 8, the largest the context is built for: calibration and verify
  have 9 rows, past the 8-row weight pass, so they take the many-row path.
* A draft set size larger than the model (k = 8 on 4 draft layers).
* Capacity: a generation that ends exactly at max_seq runs; one token more is
  refused on the host with ES_ERR_CAPACITY, and the context stays usable.
"""
import pytest

from gpu_util import Pair
from layer_drafting_draft_b300 import synth
from layer_drafting_draft_b300.easyspec import ES_ATTN_ONLY, ES_FULL_LAYER, EasySpecError

pytestmark = pytest.mark.gpu

TINY = synth.WORKLOADS["tiny_f32"]


@pytest.fixture(scope="module")
def tiny():
    return Pair(TINY["draft"], TINY["base"], "f32", TINY["seed"])


def _same_as_oracle(pair, prompt, max_new, gamma, k, T, seed, mode=ES_FULL_LAYER, max_gamma=8, max_seq=256):
    g = pair.gpu(mode=mode, max_gamma=max_gamma, max_seq=max_seq)
    out, st = g.generate(prompt, max_new, gamma, k, T, seed)
    o = pair.oracle(k=k, mode=mode)
    want = o.generate(prompt.tolist(), max_new, gamma, T, seed=seed)
    g.close()
    assert out[0].tolist() == want[0]
    return st


@pytest.mark.parametrize("P", [1, 2])
@pytest.mark.parametrize("T", [0.0, 1.0])
def test_short_prompts(tiny, P, T):
    prompt = synth.make_prompts(1, P, 512, 40 + P).numpy()
    _same_as_oracle(tiny, prompt, 24, 4, 2, T, 7)


@pytest.mark.parametrize("mode", [ES_FULL_LAYER, ES_ATTN_ONLY])
def test_gamma_one(tiny, mode):
    prompt = synth.make_prompts(1, 9, 512, 43).numpy()
    st = _same_as_oracle(tiny, prompt, 20, 1, 2, 1.0, 8, mode=mode)
    assert st["phases"] >= 10


def test_gamma_at_the_maximum(tiny):
    prompt = synth.make_prompts(1, 11, 512, 44).numpy()
    _same_as_oracle(tiny, prompt, 30, 8, 2, 1.0, 9)


def test_set_size_beyond_the_model(tiny):
    prompt = synth.make_prompts(1, 10, 512, 45).numpy()
    _same_as_oracle(tiny, prompt, 20, 4, 8, 1.0, 10)


def test_capacity_boundary(tiny):
    P, max_new, gamma = 10, 20, 4
    limit = P + max_new + 2 * gamma + 2      # what generate() needs
    prompt = synth.make_prompts(1, P, 512, 46).numpy()
    g = tiny.gpu(max_seq=limit)
    out, _ = g.generate(prompt, max_new, gamma, 2, 1.0, 11)
    want = tiny.oracle(k=2).generate(prompt.tolist(), max_new, gamma, 1.0, seed=11)
    assert out[0].tolist() == want[0]
    with pytest.raises(EasySpecError, match="ES_ERR_CAPACITY"):
        g.generate(prompt, max_new + 1, gamma, 2, 1.0, 11)
    out2, _ = g.generate(prompt, max_new, gamma, 2, 1.0, 11)   # still usable
    assert out2.tolist() == out.tolist()
    g.close()
