"""Fuzzy-drafting error per layer, and the calibration ablation, measured on
the CUDA path.

    python -m layer_drafting_draft_b300.diagnostics [--workload W] [--sigma S]
        [--k 4] [--mode full|attn] [--gamma G] [--phases 16] [--temperature 0]
    python -m layer_drafting_draft_b300.diagnostics --ablation [--workload W]
        [--sigma S] [--k 4] [--mode full|attn] [--gamma G] [--max-new 128]
        [--prompts 8] [--temperature 0]

Inside a phase, the draft's layer-parallel forwards write "fuzzy" K/V
entries for d_1..d_{gamma-1}. Every layer of a set reads the set's input
instead of its predecessor's output (OpenReview discussion page, reply on
Fig. 2). The next phase's calibration forward recomputes the committed
positions exactly and overwrites those entries. This tool reads each
draft layer's cache twice: after a draft step (fuzzy entries) and after the
next draft step's calibration (exact entries). For the accepted positions
that carried a fuzzy entry, it reports per layer the mean cosine similarity
and the relative L2 error of K and V between the two. The pages' Table 3
compares normalised hidden states of fuzzy and exact layers in the same
spirit; K and V are projections of those states.

Only the layers up to the first layer of the first multi-layer set see
exact inputs in the fuzzy forward, so only they show similarity 1 up to
rounding. Every later layer reads an input that carries the error of the
earlier sets: inside a set because it reads the set's input instead of its
predecessor's output, after a set because that set's summed deltas differ
from the sequential result.

The ablation runs the same prompts with calibration on and off
(es_set_calibration). Without it the accepted drafts keep their fuzzy
entries, which later drafts read; the pages' ablation (OpenReview discussion
page, first reply) says the errors then accumulate and acceptance suffers.
It reports the mean number of accepted drafts per phase in 32-token bins of
the output, per arm.
"""
from __future__ import annotations

import argparse
import json

import numpy as np
import torch

from . import build, synth
from .easyspec import ES_ATTN_ONLY, ES_FULL_LAYER, EasySpec


def fuzzy_kv_error(g: EasySpec, sd: dict, prompt: np.ndarray, k: int, gamma: int, phases: int,
                   temperature: float = 0.0, seed: int = 0, trace: list | None = None) -> dict:
    """Per-layer {cos_k, cos_v, rel_k, rel_v, n} over `phases` phases of one
    sequence (prompt [1, P]); g must hold that single sequence's context.
    When `trace` is a list, each phase appends (draft tokens, accepted
    count, committed tokens), so the run can be replayed elsewhere."""
    L, Hkv, hd = sd["n_layers"], sd["n_kv_heads"], sd["head_dim"]
    g.easyspec_prefill(prompt)
    n = prompt.shape[1]          # committed tokens
    sums = {l: np.zeros(4) for l in range(L)}
    count = 0
    pending = None               # (positions with fuzzy entries, their K/V per layer)
    for ph in range(phases + 1):
        drafts = g.draft_step(k, gamma, temperature, seed + ph)   # calibration of the previous phase's commits
        if pending is not None:
            pos, fuzzy = pending
            for l in range(L):
                ke, ve = g.es_read_kv(0, l, 0, max(pos) + 1, Hkv, hd)
                kf, vf = fuzzy[l]
                for i, p in enumerate(pos):
                    a, b = kf[i].ravel(), ke[p].ravel()
                    c, d = vf[i].ravel(), ve[p].ravel()
                    sums[l] += [np.dot(a, b) / (np.linalg.norm(a) * np.linalg.norm(b) + 1e-30),
                                np.dot(c, d) / (np.linalg.norm(c) * np.linalg.norm(d) + 1e-30),
                                np.linalg.norm(a - b) / (np.linalg.norm(b) + 1e-30),
                                np.linalg.norm(c - d) / (np.linalg.norm(d) + 1e-30)]
            count += len(pos)
            pending = None
        if ph == phases:
            break
        # fuzzy entries of d_1..d_{gamma-1}: positions n .. n + gamma - 2
        fuzzy_pos = list(range(n, n + gamma - 1))
        snap = {}
        for l in range(L):
            kk, vv = g.es_read_kv(0, l, 0, n + gamma - 1, Hkv, hd)
            snap[l] = (kk[n:], vv[n:])
        acc, toks = g.verify_step(temperature, seed + ph, gamma)
        a = int(acc[0])
        if trace is not None:
            trace.append((drafts[0].tolist(), a, toks[0, : a + 1].tolist()))
        kept = fuzzy_pos[: min(a, gamma - 1)]      # accepted drafts that carried a fuzzy entry
        if kept:
            pending = (kept, {l: (snap[l][0][: len(kept)], snap[l][1][: len(kept)]) for l in range(L)})
        n += a + 1
    out = {}
    for l in range(L):
        s = sums[l] / max(count, 1)
        out[l] = {"cos_k": float(s[0]), "cos_v": float(s[1]), "rel_k": float(s[2]), "rel_v": float(s[3]),
                  "n": count}
    return out


def calibration_ablation(g: EasySpec, prompts: np.ndarray, k: int, gamma: int, max_new: int,
                         temperature: float = 0.0, seed: int = 0, bin_tokens: int = 32) -> dict:
    """Per arm ("on", "off"): accepted drafts per phase, averaged over the
    prompts ([N, P], run one at a time) in bins of `bin_tokens` output tokens
    (a phase falls in the bin of its first output token), plus the overall
    mean and committed tokens per phase."""
    res = {}
    nbins = (max_new + bin_tokens - 1) // bin_tokens
    for arm in ("on", "off"):
        acc = np.zeros(nbins)
        cnt = np.zeros(nbins)
        phases = 0
        for i in range(prompts.shape[0]):
            g.es_set_calibration(arm == "on")
            g.easyspec_prefill(prompts[i:i + 1])
            out = 0
            ph = 0
            while out < max_new:
                g.draft_step(k, gamma, temperature, seed + i)
                n, _ = g.verify_step(temperature, seed + i, gamma)
                a = int(n[0])
                b = min(out // bin_tokens, nbins - 1)
                acc[b] += a
                cnt[b] += 1
                out += a + 1
                ph += 1
            phases += ph
        tot = float(acc.sum() / max(cnt.sum(), 1))
        res[arm] = {"accepted_per_phase": tot,
                    "tokens_per_phase": tot + 1.0,
                    "phases": phases,
                    "bins": [{"first_token": j * bin_tokens,
                              "accepted_per_phase": float(acc[j] / cnt[j]) if cnt[j] else None,
                              "phases": int(cnt[j])} for j in range(nbins)]}
    g.es_set_calibration(True)
    return res


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="llama3.2_1b_selfdraft_bf16")
    ap.add_argument("--sigma", type=float, default=0.05)
    ap.add_argument("--k", type=int, default=4)
    ap.add_argument("--mode", default="full", choices=["full", "attn"])
    ap.add_argument("--gamma", type=int, default=None)
    ap.add_argument("--phases", type=int, default=16)
    ap.add_argument("--temperature", type=float, default=0.0)
    ap.add_argument("--ablation", action="store_true", help="calibration on vs off")
    ap.add_argument("--max-new", type=int, default=128)
    ap.add_argument("--prompts", type=int, default=8)
    a = ap.parse_args(argv)
    build.build()
    wl = synth.WORKLOADS[a.workload]
    gamma = a.gamma or wl["gamma"]
    sigma = a.sigma if "sigmas" in wl else None
    wd, wb, prompts = synth.make_pair(a.workload, device="cuda", sigma=sigma)
    mode = ES_FULL_LAYER if a.mode == "full" else ES_ATTN_ONLY
    if a.ablation:
        P = prompts.shape[1]
        ps = synth.make_prompts(a.prompts, P, wl["draft"]["vocab"], 77).numpy()
        max_seq = (P + a.max_new + 2 * gamma + 2 + 63) // 64 * 64
        g = EasySpec(wd, wl["draft"], wb, wl["base"], wl["dtype"], 1, max_seq, gamma, mode, None)
        res = calibration_ablation(g, ps, a.k, gamma, a.max_new, a.temperature)
        g.close()
        torch.cuda.synchronize()
        print(json.dumps({"workload": a.workload, "sigma": sigma, "k": a.k, "mode": a.mode, "gamma": gamma,
                          "max_new": a.max_new, "prompts": a.prompts, "temperature": a.temperature,
                          "ablation": res}))
        return
    prompt = prompts[:1].numpy()
    max_seq = (prompt.shape[1] + (a.phases + 2) * (gamma + 1) + 2 * gamma + 2 + 63) // 64 * 64
    g = EasySpec(wd, wl["draft"], wb, wl["base"], wl["dtype"], 1, max_seq, gamma, mode, None)
    res = fuzzy_kv_error(g, wl["draft"], prompt, a.k, gamma, a.phases, a.temperature)
    g.close()
    torch.cuda.synchronize()
    print(json.dumps({"workload": a.workload, "sigma": sigma, "k": a.k, "mode": a.mode, "gamma": gamma,
                      "layers": res}))


if __name__ == "__main__":
    main()
