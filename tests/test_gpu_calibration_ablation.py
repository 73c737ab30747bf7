"""The calibration ablation (es_set_calibration(0)) against the oracle.

Without calibration the accepted drafts keep the K/V entries their layer-
parallel forwards wrote, and the exact forward that starts the next phase
covers only the positions that hold no entry (the bonus token, and d_gamma
when every draft was accepted). The pages' ablation (OpenReview discussion
page, first reply) says the fuzzy errors then accumulate. float32 pairs:
tokens bit-exact with the oracle run under the same switch, per-phase logits
to float32 rounding, and the draft cache, kept fuzzy entries included, equal
to the oracle's.
"""
import numpy as np
import pytest

from gpu_util import Pair
from layer_drafting_draft_b300 import synth
from layer_drafting_draft_b300.easyspec import ES_ATTN_ONLY, ES_FULL_LAYER
from oracle import spec

pytestmark = pytest.mark.gpu

TINY = synth.WORKLOADS["tiny_f32"]
F32_LOGIT_ATOL = 2e-4
KV_ATOL = 1e-4


@pytest.fixture(scope="module")
def tiny():
    return Pair(TINY["draft"], TINY["base"], "f32", TINY["seed"])


@pytest.fixture(scope="module")
def selfdraft():
    # draft = base + small noise: drafts are often accepted, so fuzzy entries
    # are kept and d_gamma rows occur
    return Pair(TINY["base"], TINY["base"], "f32", 3, sigma=0.1)


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_no_calibration_generate_bit_exact(tiny, T):
    groups = TINY["groups"]
    prompt = synth.make_prompts(1, TINY["prompt"], 512, 3).numpy()
    g = tiny.gpu(groups=groups)
    g.es_set_calibration(False)
    out, _ = g.generate(prompt, TINY["max_new"], TINY["gamma"], 0, T, 1234)
    o = tiny.oracle(groups=groups, calibrate=False)
    want = o.generate(prompt.tolist(), TINY["max_new"], TINY["gamma"], T, seed=1234)
    assert out[0].tolist() == want[0]
    if T == 0.0:
        assert want[0] == spec.seq_decode(tiny.Wb, tiny.shape_b, prompt[0].tolist(), TINY["max_new"])
    g.close()


@pytest.mark.parametrize("mode,k", [(ES_FULL_LAYER, 2), (ES_ATTN_ONLY, 3)])
def test_no_calibration_phases_and_cache(selfdraft, mode, k):
    sd = selfdraft.shape_d
    prompt = synth.make_prompts(1, 20, 512, 4).numpy()
    g = selfdraft.gpu(mode=mode)
    g.es_set_calibration(False)
    o = selfdraft.oracle(k=k, mode=mode, calibrate=False)
    g.easyspec_prefill(prompt)
    o.prefill(prompt.tolist())
    gamma, T, seed = 4, 1.0, 55
    accepted = []
    for ph in range(10):
        d_gpu = g.draft_step(k, gamma, T, seed)
        d_or = o.draft_row(0, gamma, T, seed)
        zq = g.es_read_dist(2, gamma)[0]
        assert np.max(np.abs(zq - o.rows[0].zq)) <= F32_LOGIT_ATOL, ph
        assert list(d_gpu[0]) == list(d_or), ph
        n, toks = g.verify_step(T, seed, gamma)
        a, new = o.verify_row(0, gamma, T, seed)
        assert int(n[0]) == a and list(toks[0, : a + 1]) == new, ph
        accepted.append(a)
    g.calibrate_kv(gamma, T, seed)     # the narrowed window of the last commits
    o.calibrate_row(o.rows[0])
    r = o.rows[0]
    n = len(r.tokens)
    assert r.draft_len == n and max(accepted) >= 2, accepted
    for layer in range(sd.n_layers):
        kk, vv = g.es_read_kv(0, layer, 0, n, sd.n_kv_heads, sd.head_dim)
        assert np.max(np.abs(kk - r.draft.K[layer, :n])) < KV_ATOL, layer
        assert np.max(np.abs(vv - r.draft.V[layer, :n])) < KV_ATOL, layer
    g.close()


def test_switch_rejected_mid_phase(tiny):
    prompt = synth.make_prompts(1, 12, 512, 6).numpy()
    g = tiny.gpu()
    g.easyspec_prefill(prompt)
    g.draft_step(2, 4, 0.0, 1)
    with pytest.raises(RuntimeError):
        g.es_set_calibration(False)
    g.verify_step(0.0, 1, 4)
    g.es_set_calibration(False)
    g.es_set_calibration(True)
    g.close()


def test_bf16_no_calibration_grouped_row_attention():
    """bf16 self-draft pair with 8 kv heads and 8 KV pages of capacity: the
    calibration and verify attention run on the grouped-row tensor-core
    kernel (at least 64 group x kv head x page items), where the narrowed
    calibration window has inactive rows (positions with a kept fuzzy entry)
    inside a group. Teacher-forced on the GPU's tokens, the draft and base
    logits meet the bf16 tolerance against the oracle under the same switch,
    and the draft cache, kept fuzzy entries included, equals the oracle's to
    the cache's bf16 rounding."""
    s = synth.shape(4, 512, 8, 8, 1376, 1000, 1e4)
    pair = Pair(s, s, "bf16", 37, sigma=0.1)
    gamma, T, seed, k = 4, 1.0, 91, 2
    prompt = synth.make_prompts(1, 300, 1000, 38).numpy()
    g = pair.gpu(max_seq=512, max_gamma=gamma, mode=ES_FULL_LAYER)
    g.es_set_calibration(False)
    o = pair.oracle(k=k, mode=ES_FULL_LAYER, max_len=512, calibrate=False)
    o.block = True
    g.easyspec_prefill(prompt)
    o.prefill(prompt.tolist())
    worst, kept = 0.0, 0
    for ph in range(10):
        d_gpu = g.draft_step(k, gamma, T, seed)
        o.draft_row(0, gamma, T, seed, force_d=d_gpu[0])
        worst = max(worst, float(np.max(np.abs(g.es_read_dist(2, gamma)[0] - o.rows[0].zq))))
        n, toks = g.verify_step(T, seed, gamma)
        a = int(n[0])
        o.verify_row(0, gamma, T, seed, force=(a, toks[0, : a + 1]))
        worst = max(worst, float(np.max(np.abs(g.es_read_dist(3, gamma)[0] - o.rows[0].zp))))
        kept += min(a, gamma - 1)
    assert worst <= 3e-2, worst
    assert kept >= 2, kept        # some fuzzy entries were kept (inactive calibration rows)
    g.es_profile(1)               # the grouped kernel's chunk merge runs: the path is the one meant
    g.calibrate_kv(gamma, T, seed)
    assert "attention_merge" in g.es_profile_read()
    g.es_profile(0)
    o.calibrate_row(o.rows[0])
    r = o.rows[0]
    n = len(r.tokens)
    for layer in range(s["n_layers"]):
        kk, vv = g.es_read_kv(0, layer, 0, n, s["n_kv_heads"], s["head_dim"])
        scale = max(1.0, float(np.max(np.abs(r.draft.K[layer, :n]))))
        assert np.max(np.abs(kk - r.draft.K[layer, :n])) <= 2e-2 * scale, layer
        assert np.max(np.abs(vv - r.draft.V[layer, :n])) <= 2e-2 * max(1.0, float(np.max(np.abs(r.draft.V[layer, :n])))), layer
    g.close()
