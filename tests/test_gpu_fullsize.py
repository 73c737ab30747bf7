"""Checks at the full widths of the Qwen2.5-shaped pair (0.5B-shaped draft,
7B-shaped base), in the launch configuration the benchmark times.

* Lossless decoding (speculative-sampling rule, [SD]): at temperature 0 the
  output is the base model's greedy continuation whatever the draft does, so
  layer-parallel drafts with sets of 4 (both modes) and exact drafts (k = 1)
  must emit the same tokens.  This holds at any size; it exercises the full
  7B-shaped verify path, whose per-row results do not depend on where a row
  sits in the verify window.
* Full-width parity with the oracle: the 24-layer 0.5B-shaped draft and a
  2-layer base of the 7B widths (d 3584, ffn 18944, 28/4 heads of 128), with
  the vocabulary cut to 32000 so the float64 oracle fits in host memory.
  Per-phase draft and base logits must meet the bf16 tolerance.
"""
import numpy as np
import pytest
import torch

from gpu_util import Pair, rel_l2
from layer_drafting_draft_b300 import synth
from layer_drafting_draft_b300.easyspec import ES_ATTN_ONLY, ES_FULL_LAYER, EasySpec

pytestmark = pytest.mark.gpu

QWEN = synth.WORKLOADS["qwen2.5_0.5b_7b_bf16"]
BF16_MAXABS, BF16_RELL2 = 3e-2, 1e-2


def test_qwen_greedy_tokens_identical_across_draft_configs():
    wd, wb, prompts = synth.make_pair("qwen2.5_0.5b_7b_bf16", device="cuda")
    prompt = prompts[:1, :64].numpy()
    outs = {}
    for mode in (ES_FULL_LAYER, ES_ATTN_ONLY):
        g = EasySpec(wd, QWEN["draft"], wb, QWEN["base"], "bf16", 1, 256, 4, mode, None)
        for k in ((4, 1) if mode == ES_FULL_LAYER else (4,)):
            out, st = g.generate(prompt, 40, 4, k, 0.0, 5)
            outs[(mode, k)] = out[0].tolist()
            assert st["emitted"] >= 40
        g.close()
    ref = outs[(ES_FULL_LAYER, 1)]
    for key, toks in outs.items():
        assert toks == ref, (key, toks, ref)
    del wd, wb
    torch.cuda.empty_cache()


def test_fullwidth_logits_within_tolerance():
    d = dict(QWEN["draft"], vocab=32000)
    b = dict(QWEN["base"], n_layers=2, vocab=32000)
    pair = Pair(d, b, "bf16", 21)
    prompt = synth.make_prompts(1, 24, 32000, 22).numpy()
    g = pair.gpu(max_seq=128, mode=ES_FULL_LAYER)
    o = pair.oracle(k=4, mode=ES_FULL_LAYER, max_len=128)
    g.easyspec_prefill(prompt)
    o.prefill(prompt.tolist())
    worst = {"q": 0.0, "p": 0.0, "rel": 0.0}
    for ph in range(2):
        d_gpu = g.draft_step(4, 4, 0.0, 31)
        o.draft_row(0, 4, 0.0, 31, force_d=d_gpu[0])
        zq = g.es_read_dist(2, 4)[0]
        zq_or = np.asarray(o.rows[0].zq, np.float64)
        n, toks = g.verify_step(0.0, 31, 4)
        a = int(n[0])
        o.verify_row(0, 4, 0.0, 31, force=(a, toks[0, : a + 1]))
        zp = g.es_read_dist(3, 4)[0]
        zp_or = np.asarray(o.rows[0].zp, np.float64)
        worst["q"] = max(worst["q"], float(np.max(np.abs(zq - zq_or))))
        worst["p"] = max(worst["p"], float(np.max(np.abs(zp - zp_or))))
        worst["rel"] = max(worst["rel"], rel_l2(zq, zq_or), rel_l2(zp, zp_or))
    print("full-width bf16:", worst)
    assert worst["q"] <= BF16_MAXABS and worst["p"] <= BF16_MAXABS
    assert worst["rel"] <= BF16_RELL2
    g.close()


def test_wide_window_variant_within_tolerance():
    """A base of d 4096 and ffn 20480 verified over gamma+1 = 8 rows.

    The gate/up pass's activation window (8 rows x 4096 columns as hi/lo
    planes) does not fit the 8-warp budget. The planner therefore takes the
    16-warp variant for it, one 512-thread CTA per SM, as it does at the
    Llama-3-70B widths. Logits must meet the bf16 tolerance against the
    oracle.
    """
    d = synth.shape(4, 256, 4, 2, 688, 1000, 1e4)
    b = synth.shape(2, 4096, 32, 8, 20480, 1000, 5e5)
    pair = Pair(d, b, "bf16", 23)
    gamma = 7
    prompt = synth.make_prompts(1, 20, 1000, 24).numpy()
    g = pair.gpu(max_seq=128, max_gamma=8, mode=ES_FULL_LAYER)
    o = pair.oracle(k=2, mode=ES_FULL_LAYER, max_len=128)
    g.easyspec_prefill(prompt)
    o.prefill(prompt.tolist())
    worst, rel = 0.0, 0.0
    for ph in range(2):
        d_gpu = g.draft_step(2, gamma, 0.0, 41 + ph)
        o.draft_row(0, gamma, 0.0, 41 + ph, force_d=d_gpu[0])
        n, toks = g.verify_step(0.0, 41 + ph, gamma)
        a = int(n[0])
        o.verify_row(0, gamma, 0.0, 41 + ph, force=(a, toks[0, : a + 1]))
        zp = g.es_read_dist(3, gamma)[0]
        zp_or = np.asarray(o.rows[0].zp, np.float64)
        worst = max(worst, float(np.max(np.abs(zp - zp_or))))
        rel = max(rel, rel_l2(zp, zp_or))
    print("wide-window bf16:", worst, rel)
    assert worst <= BF16_MAXABS and rel <= BF16_RELL2
    g.close()


def test_tensor_core_decode_passes_at_70b_widths():
    """At the Llama-3-70B widths (d 8192, ffn 28672, 64/8 heads) the base's
    SwiGLU gate/up pair (940 MB) and an output head of at least 1.5 GB run
    on the tcgen05 tensor-core kernel even at 5 rows, with the normalised
    hi/lo planes written by the kernel before them.  One base layer and a
    96000-token vocabulary (a 1.57 GB head) keep the float64 oracle within
    host memory; verify logits must meet the bf16 tolerance."""
    d = synth.shape(2, 512, 8, 2, 1376, 96000, 5e5)
    b = synth.shape(1, 8192, 64, 8, 28672, 96000, 5e5)
    pair = Pair(d, b, "bf16", 25)
    gamma = 4
    prompt = synth.make_prompts(1, 20, 96000, 26).numpy()
    g = pair.gpu(max_seq=128, max_gamma=gamma, mode=ES_FULL_LAYER)
    o = pair.oracle(k=1, mode=ES_FULL_LAYER, max_len=128)
    o.block = True
    g.easyspec_prefill(prompt)
    o.prefill(prompt.tolist())
    worst, rel = 0.0, 0.0
    for ph in range(2):
        d_gpu = g.draft_step(1, gamma, 0.0, 51 + ph)
        o.draft_row(0, gamma, 0.0, 51 + ph, force_d=d_gpu[0])
        n, toks = g.verify_step(0.0, 51 + ph, gamma)
        a = int(n[0])
        o.verify_row(0, gamma, 0.0, 51 + ph, force=(a, toks[0, : a + 1]))
        zp = g.es_read_dist(3, gamma)[0]
        zp_or = np.asarray(o.rows[0].zp, np.float64)
        worst = max(worst, float(np.max(np.abs(zp - zp_or))))
        rel = max(rel, rel_l2(zp, zp_or))
    g.es_profile(1)
    g.draft_step(1, gamma, 0.0, 60)
    g.verify_step(0.0, 60, gamma)
    kernels = g.es_profile_read()
    g.es_profile(0)
    print("70B-width tensor-core decode passes, bf16:", worst, rel, sorted(kernels))
    assert "base.tc_gateup" in kernels and "base.tc_lm_head" in kernels
    assert worst <= BF16_MAXABS and rel <= BF16_RELL2
    g.close()
