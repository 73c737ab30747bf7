"""Run speculative phases of a synthetic workload for profiling.

    python -m layer_drafting_draft_b300.profile --workload qwen2.5_0.5b_7b_bf16 \
        --k 4 --phases 4 --warmup-phases 2 [--table] [--base-layers N] [--batch B]

After the prompt prefill and `--warmup-phases` untimed phases, `--phases`
phases (draft_step + verify_step) run inside the NVTX range "measure", so an
`ncu --nvtx --nvtx-include measure/` capture sees exactly their launches;
each draft_step / verify_step sits in a nested range "draft" / "verify"
(`--nvtx-include measure/verify/` selects the base model's launches).
With --table the same phases run a second time with per-launch CUDA-event
timing and a per-kernel table (time, launches, algorithmic bytes, GB/s) is
printed.  --base-layers / --draft-layers truncate the models (same widths)
and --vocab cuts the vocabulary of both, to keep a capture's device
footprint small.
"""
from __future__ import annotations

import argparse
import json

import torch

from . import build, synth
from .easyspec import ES_ATTN_ONLY, ES_FULL_LAYER, EasySpec


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="qwen2.5_0.5b_7b_bf16")
    ap.add_argument("--k", type=int, default=4)
    ap.add_argument("--mode", default="full", choices=["full", "attn"])
    ap.add_argument("--gamma", type=int, default=None)
    ap.add_argument("--temperature", type=float, default=1.0)
    ap.add_argument("--phases", type=int, default=4)
    ap.add_argument("--warmup-phases", type=int, default=2)
    ap.add_argument("--base-layers", type=int, default=None)
    ap.add_argument("--draft-layers", type=int, default=None)
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--vocab", type=int, default=None)
    ap.add_argument("--table", action="store_true")
    a = ap.parse_args(argv)

    build.build()
    wl = synth.WORKLOADS[a.workload]
    sd, sb = dict(wl["draft"]), dict(wl["base"])
    if a.draft_layers:
        sd["n_layers"] = a.draft_layers
    if a.base_layers:
        sb["n_layers"] = a.base_layers
    if a.vocab:
        sd["vocab"] = sb["vocab"] = a.vocab
    seed = 1000 * wl["seed"]
    wb = synth.make_weights(sb, seed + 2, wl["dtype"], "cuda")
    wd = synth.make_weights(sd, seed + 1, wl["dtype"], "cuda")
    prompt = synth.make_prompts(a.batch, wl["prompt"], sb["vocab"], seed + 3).numpy()
    gamma = a.gamma or wl["gamma"]
    k = a.k if sd["n_layers"] > 2 else 1
    n_ph = a.warmup_phases + a.phases
    max_seq = (wl["prompt"] + 2 * (n_ph + 1) * (gamma + 1) + 63) // 64 * 64
    stream = torch.cuda.Stream()
    g = EasySpec(wd, sd, wb, sb, wl["dtype"], a.batch, max_seq, gamma,
                 ES_FULL_LAYER if a.mode == "full" else ES_ATTN_ONLY, None, stream)

    def phases(n, s0):
        for i in range(n):
            torch.cuda.nvtx.range_push("draft")
            g.draft_step(k, gamma, a.temperature, s0 + i)
            torch.cuda.nvtx.range_pop()
            torch.cuda.nvtx.range_push("verify")
            g.verify_step(a.temperature, s0 + i, gamma)
            torch.cuda.nvtx.range_pop()

    g.easyspec_prefill(prompt)
    phases(a.warmup_phases, 100)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("measure")
    phases(a.phases, 200)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    if a.table:
        g.easyspec_prefill(prompt)
        phases(a.warmup_phases, 100)
        g.es_profile(True)
        phases(a.phases, 200)
        prof = g.es_profile_read()
        g.es_profile(False)
        total = sum(v[0] for v in prof.values())
        rows = sorted(prof.items(), key=lambda kv: -kv[1][0])
        print(f"{'kernel':24s} {'ms':>9s} {'share':>6s} {'launches':>8s} {'us/launch':>9s} {'GB/s':>8s}")
        for name, (ms, n, by) in rows:
            gbs = by / (ms * 1e-3) / 1e9 if by else 0.0
            print(f"{name:24s} {ms:9.3f} {ms / total:6.3f} {n:8d} {1e3 * ms / n:9.2f} {gbs:8.1f}")
        print(json.dumps({"workload": a.workload, "k": k, "gamma": gamma, "phases": a.phases,
                          "total_ms": total}))
    g.close()


if __name__ == "__main__":
    main()
