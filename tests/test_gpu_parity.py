"""End-to-end parity of the CUDA path with the oracle.

float32 pairs: emitted tokens are bit-exact (greedy and seeded sampling), and
per-phase logits / probabilities agree to float32 rounding.  bf16 pairs: the
oracle is fed the same bf16-rounded weights in float64; logits must satisfy
max-abs <= 3e-2 and relative L2 <= 1e-2, and the acceptance-rate difference
is reported.  Calibration must leave the draft cache equal to a fresh
sequential prefill of the committed tokens (OpenReview discussion page,
reply on Figure 2: calibrated entries replace the fuzzy ones).
"""
import numpy as np
import pytest

from gpu_util import Pair, rel_l2
from layer_drafting_draft_b300 import synth
from layer_drafting_draft_b300.easyspec import ES_ATTN_ONLY, ES_FULL_LAYER
from oracle import model as M

pytestmark = pytest.mark.gpu

TINY = synth.WORKLOADS["tiny_f32"]
F32_LOGIT_ATOL = 2e-4      # float32 path vs float64 oracle, |logits| ~ 1
F32_PROB_ATOL = 2e-6
BF16_MAXABS, BF16_RELL2 = 3e-2, 1e-2


@pytest.fixture(scope="module")
def tiny():
    return Pair(TINY["draft"], TINY["base"], "f32", TINY["seed"])


def _prompt(V, P, seed):
    return synth.make_prompts(1, P, V, seed).numpy()


def _phase_compare(g, o, k, gamma, T, seed, n_phases, logit_atol, prob_atol, bf16=False):
    """Run phases on both sides; compare distributions and tokens each phase."""
    stats = {"maxabs_q": 0.0, "maxabs_p": 0.0, "rell2": 0.0, "acc_gpu": 0, "acc_or": 0}
    for ph in range(n_phases):
        d_gpu = g.draft_step(k, gamma, T, seed)
        # bf16: teacher-force the oracle onto the GPU's draft tokens
        d_or = o.draft_row(0, gamma, T, seed, force_d=d_gpu[0] if bf16 else None)
        zq = g.es_read_dist(2, gamma)[0]
        zq_or = np.asarray(o.rows[0].zq, np.float64)
        stats["maxabs_q"] = max(stats["maxabs_q"], float(np.max(np.abs(zq - zq_or))))
        stats["rell2"] = max(stats["rell2"], rel_l2(zq, zq_or))
        if not bf16:
            assert np.max(np.abs(zq - zq_or)) <= logit_atol, (ph, np.max(np.abs(zq - zq_or)))
            if T > 0:
                q = g.es_read_dist(0, gamma)[0]
                assert np.max(np.abs(q - o.rows[0].q)) <= prob_atol
        if not bf16:
            assert list(d_gpu[0]) == list(d_or), (ph, d_gpu[0], d_or, _margin(zq_or))
        else:
            stats["draft_agree"] = stats.get("draft_agree", 0) + int(list(d_gpu[0]) == o.rows[0].d_own)
        n, toks = g.verify_step(T, seed, gamma)
        if bf16:
            a_g = int(n[0])
            a, new = o.verify_row(0, gamma, T, seed, force=(a_g, toks[0, : a_g + 1]))
            stats["acc_gpu"] += a_g
            stats["acc_or"] += o.rows[0].own[0]
        else:
            a, new = o.verify_row(0, gamma, T, seed)
        zp = g.es_read_dist(3, gamma)[0]
        zp_or = np.asarray(o.rows[0].zp, np.float64)
        stats["maxabs_p"] = max(stats["maxabs_p"], float(np.max(np.abs(zp - zp_or))))
        stats["rell2"] = max(stats["rell2"], rel_l2(zp, zp_or))
        if not bf16:
            assert np.max(np.abs(zp - zp_or)) <= logit_atol, (ph, np.max(np.abs(zp - zp_or)))
        if not bf16:
            assert n[0] == a and list(toks[0, : a + 1]) == new, (ph, n[0], toks[0], a, new)
            stats["acc_gpu"] += int(n[0])
            stats["acc_or"] += a
    return stats


def _margin(z):
    s = np.sort(np.asarray(z, np.float64), axis=-1)
    return s[..., -1] - s[..., -2]


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_tiny_f32_generate_bit_exact(tiny, T):
    """Configured sets {0,1},{2,3}, gamma = 4, 64 new tokens, 32-token prompt."""
    groups = TINY["groups"]
    prompt = _prompt(512, TINY["prompt"], 3)
    g = tiny.gpu(groups=groups)
    out, st = g.generate(prompt, TINY["max_new"], TINY["gamma"], 0, T, 1234)
    o = tiny.oracle(groups=groups)
    want = o.generate(prompt.tolist(), TINY["max_new"], TINY["gamma"], T, seed=1234)
    assert out[0].tolist() == want[0]
    if T == 0.0:
        from oracle import spec
        assert want[0] == spec.seq_decode(tiny.Wb, tiny.shape_b, prompt[0].tolist(), TINY["max_new"])
    assert st["emitted"] >= TINY["max_new"] and st["phases"] >= 1
    # the run's counters: host wall-clock times of both parts, launches of
    # this library while decoding, drafts proposed to unfinished sequences
    assert st["prefill_ms"] > 0 and st["decode_ms"] > 0
    assert st["kernel_launches"] >= st["phases"] > 0
    assert st["drafted"] == TINY["gamma"] * st["phases"] and 0 <= st["accepted"] <= st["drafted"]
    g.close()


@pytest.mark.parametrize("mode", [ES_FULL_LAYER, ES_ATTN_ONLY])
@pytest.mark.parametrize("k", [1, 2, 3])
def test_tiny_f32_phases(tiny, mode, k):
    prompt = _prompt(512, 20, 4)
    g = tiny.gpu(mode=mode)
    o = tiny.oracle(k=k, mode=mode)
    g.easyspec_prefill(prompt)
    o.prefill(prompt.tolist())
    _phase_compare(g, o, k, 4, 1.0, 77 + k, 8, F32_LOGIT_ATOL, F32_PROB_ATOL)
    g.close()


def test_tiny_f32_calibrated_kv_equals_prefill(tiny):
    prompt = _prompt(512, 17, 5)
    g = tiny.gpu(mode=ES_FULL_LAYER)
    g.easyspec_prefill(prompt)
    gamma = 4
    for _ in range(5):
        g.draft_step(2, gamma, 1.0, 9)
        g.verify_step(1.0, 9, gamma)
    g.calibrate_kv(gamma, 1.0, 9)
    toks = g.es_read_tokens(0)
    n = len(toks)
    o = tiny.oracle()
    fresh = M.KVCache(tiny.shape_d, 256)
    for pos, t in enumerate(toks):
        M.forward_exact(tiny.Wd, tiny.shape_d, int(t), pos, fresh)
    for layer in range(tiny.shape_d.n_layers):
        k, v = g.es_read_kv(0, layer, 0, n, tiny.shape_d.n_kv_heads, tiny.shape_d.head_dim)
        assert np.max(np.abs(k - fresh.K[layer, :n])) < 1e-4
        assert np.max(np.abs(v - fresh.V[layer, :n])) < 1e-4
    # the base cache holds every committed token but the pending last one
    fresh_b = M.KVCache(tiny.shape_b, 256)
    for pos, t in enumerate(toks[:-1]):
        M.forward_exact(tiny.Wb, tiny.shape_b, int(t), pos, fresh_b)
    for layer in (0, tiny.shape_b.n_layers - 1):
        k, v = g.es_read_kv(1, layer, 0, n - 1, tiny.shape_b.n_kv_heads, tiny.shape_b.head_dim)
        assert np.max(np.abs(k - fresh_b.K[layer, : n - 1])) < 1e-4
    g.close()


def test_tiny_f32_batch_rows_independent(tiny):
    """Three sequences decoded together equal three single-sequence runs."""
    prompts = synth.make_prompts(3, 12, 512, 6).numpy()
    g = tiny.gpu(max_batch=3)
    out, _ = g.generate(prompts, 24, 3, 2, 1.0, 55)
    o = tiny.oracle(k=2)
    want = o.generate(prompts.tolist(), 24, 3, 1.0, seed=55)
    assert out.tolist() == want
    g.close()


# ------------------------------------------------------------------ bf16
def _bf16_pair(seed=7, V=1000, ragged=True):
    sd = synth.shape(6, 256, 4, 2, 688 if ragged else 512, V, 1e4)
    sb = synth.shape(4, 384, 6, 2, 1032 if ragged else 1024, V, 1e4, head_dim=64)
    return Pair(sd, sb, "bf16", seed)


@pytest.mark.parametrize("mode,k", [(ES_FULL_LAYER, 2), (ES_ATTN_ONLY, 4), (ES_FULL_LAYER, 1)])
def test_bf16_logits_within_tolerance(mode, k):
    pair = _bf16_pair()
    prompt = _prompt(pair.sd["vocab"], 70, 8)
    g = pair.gpu(mode=mode)
    o = pair.oracle(k=k, mode=mode)
    g.easyspec_prefill(prompt)
    o.prefill(prompt.tolist())
    st = _phase_compare(g, o, k, 4, 0.0, 3, 6, None, None, bf16=True)
    print(f"bf16 mode={mode} k={k}: {st}")
    assert st["maxabs_q"] <= BF16_MAXABS and st["maxabs_p"] <= BF16_MAXABS
    assert st["rell2"] <= BF16_RELL2
    g.close()

