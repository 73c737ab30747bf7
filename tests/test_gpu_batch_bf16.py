"""bf16 batches on the many-row path.

Three sequences decoded together make 15 verify rows and 15 calibration
rows. Those pass through the many-row weight path: bf16 tensor-core GEMMs on
hi/lo activation planes. The 3-row fuzzy drafts stay on the fused
tensor-core GEMV. Every row's draft and base logits must meet the bf16
tolerance against the oracle, which is teacher-forced onto the GPU's tokens.
This covers the prompt prefill too: 40 positions per sequence.
"""
import numpy as np
import pytest

from gpu_util import Pair, rel_l2
from layer_drafting_draft_b300 import synth
from layer_drafting_draft_b300.easyspec import ES_FULL_LAYER

pytestmark = pytest.mark.gpu

BF16_MAXABS, BF16_RELL2 = 3e-2, 1e-2


def test_bf16_batch_of_three_within_tolerance():
    sd = synth.shape(6, 256, 4, 2, 688, 1000, 1e4)
    sb = synth.shape(4, 384, 6, 2, 1032, 1000, 1e4, head_dim=64)
    pair = Pair(sd, sb, "bf16", 9)
    B, gamma, k = 3, 4, 2
    prompts = synth.make_prompts(B, 40, 1000, 10).numpy()
    g = pair.gpu(max_batch=B, mode=ES_FULL_LAYER)
    o = pair.oracle(k=k, mode=ES_FULL_LAYER)
    g.easyspec_prefill(prompts)
    o.prefill(prompts.tolist())
    worst = 0.0
    worst_rel = 0.0
    for ph in range(3):
        seed = 70 + ph
        d_gpu = g.draft_step(k, gamma, 0.0, seed)
        zq = g.es_read_dist(2, gamma)
        for b in range(B):
            o.draft_row(b, gamma, 0.0, seed, force_d=d_gpu[b])
            ref = np.asarray(o.rows[b].zq, np.float64)
            worst = max(worst, float(np.max(np.abs(zq[b] - ref))))
            worst_rel = max(worst_rel, rel_l2(zq[b], ref))
        n, toks = g.verify_step(0.0, seed, gamma)
        zp = g.es_read_dist(3, gamma)
        for b in range(B):
            a = int(n[b])
            o.verify_row(b, gamma, 0.0, seed, force=(a, toks[b, : a + 1]))
            ref = np.asarray(o.rows[b].zp, np.float64)
            worst = max(worst, float(np.max(np.abs(zp[b] - ref))))
            worst_rel = max(worst_rel, rel_l2(zp[b], ref))
    print(f"bf16 batch of {B}: max-abs {worst:.3g}, rel-L2 {worst_rel:.3g}")
    assert worst <= BF16_MAXABS and worst_rel <= BF16_RELL2
    g.close()
