"""Layer-set layouts of the layer-parallel draft, and a measured search.

    python -m layer_drafting_draft_b300.layouts [--workload W] [--sigma S]
        [--mode full|attn] [--gamma G] [--prompts 8] [--max-new 128]
        [--temperature 1.0] [--layouts name,name,...]

A layout lists the draft's layer sets in order; every layer lies in exactly
one set, and a set runs layer-parallel on its input (one layer: exact).

The default rule (OpenReview discussion page, reply on Table 4 / Appendix
B.1): layer 0 and the last layer stay alone, because the first and last
layers are the most sensitive to the approximation, and the layers between
fall in blocks aligned to multiples of the set size N. This is the only
reading of the garbled rule that gives the page's own 32-layer, N = 4
example, where layers 28 to 30 form a 3-set because layer 31 is the last.
The same reply says the authors are not sure this rule is the best and that
other combinations cost only a configuration change. The variants here:

  aligned(L, N)    the default rule above
  from_one(L, N)   consecutive N-sets from layer 1, then a shorter set, then
                   the last layer alone (the other reading of the rule)
  with_ends(L, N)  consecutive N-sets from layer 0, the first and last layers
                   included in sets
  tapered(L, N)    singletons at both ends, 2-sets next to them, N-sets in the
                   middle (non-uniform sizes)
  by_sizes(sizes)  any sequence of set sizes

search() measures each candidate on the CUDA path: committed tokens per
phase (acceptance), milliseconds per phase (draft + verify) and their
ratio, decode tokens per second. It ranks the candidates by that ratio, the
quantity the layout is chosen for.
"""
from __future__ import annotations

import argparse
import json
from typing import Callable

MAX_SET = 8  # layers per set the fused kernels take


def by_sizes(sizes) -> list[list[int]]:
    out, l = [], 0
    for s in sizes:
        if s < 1:
            raise ValueError("set sizes must be >= 1")
        out.append(list(range(l, l + s)))
        l += s
    return out


def aligned(L: int, N: int) -> list[list[int]]:
    if N < 1 or L < 1:
        raise ValueError("need L >= 1 and N >= 1")
    if N == 1 or L <= 2:
        return [[l] for l in range(L)]
    sets = [[0]]
    for b0 in range(0, L, N):
        block = [l for l in range(max(b0, 1), min(b0 + N, L - 1))]
        if block:
            sets.append(block)
    sets.append([L - 1])
    return sets


def from_one(L: int, N: int) -> list[list[int]]:
    if N < 1 or L < 1:
        raise ValueError("need L >= 1 and N >= 1")
    if L <= 2:
        return [[l] for l in range(L)]
    sets = [[0]]
    for b0 in range(1, L - 1, N):
        sets.append(list(range(b0, min(b0 + N, L - 1))))
    sets.append([L - 1])
    return sets


def with_ends(L: int, N: int) -> list[list[int]]:
    if N < 1 or L < 1:
        raise ValueError("need L >= 1 and N >= 1")
    return [list(range(b0, min(b0 + N, L))) for b0 in range(0, L, N)]


def tapered(L: int, N: int) -> list[list[int]]:
    if L < 6 or N < 2:
        return aligned(L, N)
    mid = L - 6
    sizes = [1, 2] + [N] * (mid // N) + ([mid % N] if mid % N else []) + [2, 1]
    return by_sizes(sizes)


def check(sets, L: int, max_set: int = MAX_SET) -> None:
    """Raise ValueError unless the sets cover 0..L-1 once, in order, each
    with 1..max_set layers."""
    flat = [l for s in sets for l in s]
    if flat != list(range(L)):
        raise ValueError("layer sets must cover 0..L-1 once, in order")
    if any(not 1 <= len(s) <= max_set for s in sets):
        raise ValueError(f"every set needs 1..{max_set} layers")


def starts(sets) -> list[int]:
    """The first layer of every set (the library's group_starts)."""
    return [s[0] for s in sets]


def name(sets) -> str:
    return "|".join(f"{s[0]}-{s[-1]}" if len(s) > 1 else str(s[0]) for s in sets)


def candidates(L: int, sizes=(2, 3, 4, 8), max_set: int = MAX_SET) -> dict[str, list[list[int]]]:
    """Named layouts to try: sequential (N = 1) and every generator above for
    each set size, valid and distinct ones only (first name wins)."""
    gens = {"aligned": aligned, "from_one": from_one, "with_ends": with_ends, "tapered": tapered}
    out, seen = {"sequential": aligned(L, 1)}, {name(aligned(L, 1))}
    for N in sizes:
        for gname, f in gens.items():
            s = f(L, N)
            try:
                check(s, L, max_set)
            except ValueError:
                continue
            if name(s) in seen:
                continue
            seen.add(name(s))
            out[f"{gname}{N}"] = s
    return out


def search(measure: Callable[[list[list[int]]], dict], cands: dict[str, list[list[int]]]) -> list[dict]:
    """measure(sets) -> {"tokens": committed tokens, "phases": phases,
    "ms": decode milliseconds, optionally "useful": the tokens asked for}
    over the same prompts for every candidate. The rate counts the useful
    tokens (the last phase may commit past the end). Returns one record per
    candidate, best decode rate first."""
    rows = []
    for nm, sets in cands.items():
        m = measure(sets)
        ph = max(m["phases"], 1)
        rows.append({"layout": nm, "sets": name(sets),
                     "tokens_per_phase": m["tokens"] / ph,
                     "ms_per_phase": m["ms"] / ph,
                     "tok_s": m.get("useful", m["tokens"]) / (m["ms"] / 1e3) if m["ms"] > 0 else 0.0})
    rows.sort(key=lambda r: -r["tok_s"])
    return rows


def gpu_measure(wl: dict, draft_w, base_w, prompts, mode: int, gamma: int, max_new: int,
                temperature: float, seed: int = 0, warmup: int = 1):
    """A measure() for search(): decodes every prompt (one at a time) through
    es_decode under the given layout and times it with CUDA events."""
    import torch

    from .easyspec import EasySpec
    P = prompts.shape[1]
    max_seq = ((P + max_new + 2 * gamma + 2) + 63) // 64 * 64
    stream = torch.cuda.Stream()

    def measure(sets):
        g = EasySpec(draft_w, wl["draft"], base_w, wl["base"], wl["dtype"], 1, max_seq, gamma, mode,
                     starts(sets), stream)
        tot = {"tokens": 0, "phases": 0, "ms": 0.0, "useful": 0}
        try:
            for w in range(warmup):
                g.easyspec_prefill(prompts[:1])
                g.es_decode(max_new, gamma, 0, temperature, 10_000 + w)
            for i in range(prompts.shape[0]):
                g.easyspec_prefill(prompts[i:i + 1])
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                st = g.es_decode(max_new, gamma, 0, temperature, seed + i)
                e1.record(stream)
                e1.synchronize()
                tot["ms"] += e0.elapsed_time(e1)
                tot["tokens"] += st["emitted"]
                tot["phases"] += st["phases"]
                tot["useful"] += max_new
        finally:
            g.close()
        return tot

    return measure


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="llama3.2_1b_selfdraft_bf16")
    ap.add_argument("--sigma", type=float, default=0.05)
    ap.add_argument("--mode", default="full", choices=["full", "attn"])
    ap.add_argument("--gamma", type=int, default=None)
    ap.add_argument("--prompts", type=int, default=8)
    ap.add_argument("--max-new", type=int, default=128)
    ap.add_argument("--temperature", type=float, default=1.0)
    ap.add_argument("--layouts", default=None, help="comma-separated candidate names (default: all)")
    a = ap.parse_args(argv)
    import torch

    from . import build, synth
    from .easyspec import ES_ATTN_ONLY, ES_FULL_LAYER
    build.build()
    wl = synth.WORKLOADS[a.workload]
    gamma = a.gamma or wl["gamma"]
    sigma = a.sigma if "sigmas" in wl else None
    wd, wb, prompts = synth.make_pair(a.workload, device="cuda", sigma=sigma)
    ps = synth.make_prompts(a.prompts, prompts.shape[1], wl["draft"]["vocab"], 91).numpy()
    cands = candidates(wl["draft"]["n_layers"])
    if a.layouts:
        bad = [k for k in a.layouts.split(",") if k not in cands]
        if bad:
            raise SystemExit(f"--layouts: unknown {', '.join(bad)}; known: {', '.join(cands)}")
        cands = {k: cands[k] for k in a.layouts.split(",")}
    mode = ES_FULL_LAYER if a.mode == "full" else ES_ATTN_ONLY
    rows = search(gpu_measure(wl, wd, wb, ps, mode, gamma, a.max_new, a.temperature), cands)
    torch.cuda.synchronize()
    print(json.dumps({"workload": a.workload, "sigma": sigma, "mode": a.mode, "gamma": gamma,
                      "prompts": a.prompts, "max_new": a.max_new, "temperature": a.temperature,
                      "ranking": rows}))


if __name__ == "__main__":
    main()
