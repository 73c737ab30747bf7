#!/usr/bin/env python
"""Benchmark: EasySpec layer-parallel speculative decoding on one B300.

One step = one speculative generation of `max_new` tokens at batch 1 for the
workload (default: the largest single-GPU pair, a Llama-3-shaped bf16 pair
with an 8B-shaped draft and a 70B-shaped base, about 157 GB of weights,
512-token prompt, gamma 4, 128 new tokens, layer-set size k = 4,
temperature 1.0), random-initialised weights and uniform prompt ids.

  value      decode tokens/s with the prompt already prefilled in HBM: CUDA
             events on the library's stream around es_decode (all phases:
             calibration + fuzzy drafts + verification + accept/resample)
  e2e        the same generation through the C-ABI call generate() with host
             buffers: prompt upload, both prefills, decoding and the token
             read-back inside the timed region (host wall clock); prefill_ms
             is the prompt prefill part of it (both models)
  draft/verify  per-phase breakdown of one more generation (the library's
             part timing: CUDA events around each phase part's graph
             launch): calibration, the gamma-1 fuzzy drafts ("fuzzy": the
             layer-parallel draft forwards alone) and verify+accept, each
             with its fraction of the HBM weight-stream roofline: bytes =
             weights streamed + KV read/written
  roofline   the dominant kernel (most device time in a per-launch event
             pass over one generation): algorithmic bytes / event time vs the
             measured HBM copy bandwidth
  cpu_baseline  the CPU oracle (float64 numpy) on a bounded sample

With --impl reference the oracle arm runs instead (CPU only).
Multi-GPU (torchrun): independent replicas, one per GPU; no collective on
the data path.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "llama3_8b_70b_bf16"
METRIC = "draft & end-to-end tok/s, bs=1, 1xB300; % of HBM weight-stream roofline"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--k", type=int, default=4)
    ap.add_argument("--mode", default="full", choices=["full", "attn"])
    ap.add_argument("--temperature", type=float, default=1.0)
    ap.add_argument("--gamma", type=int, default=None)
    ap.add_argument("--batch", type=int, default=1,
                    help="sequences decoded together (the batched long-context workload: 1, 4 or 16)")
    ap.add_argument("--sigma", type=float, default=None,
                    help="self-draft workloads: draft = base + N(0, (sigma*0.02)^2)")
    ap.add_argument("--layout", default=None,
                    help="named draft layer-set layout (layouts.candidates); replaces --k")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


# ------------------------------------------------------------------ bytes model
def weight_bytes(s: dict, esz: int) -> dict:
    d, hd, F, V = s["d"], s["head_dim"], s["ffn"], s["vocab"]
    qd, kvd = s["n_heads"] * hd, s["n_kv_heads"] * hd
    layer = (qd * d + 2 * kvd * d + d * qd + 3 * F * d + 2 * d) * esz
    return {"layers": s["n_layers"] * layer, "head": (V * d + d) * esz, "embed_row": d * esz}


def kv_bytes(s: dict, esz: int, ctx: int, rows: int) -> float:
    """K/V read by `rows` queries at context ~ctx plus the rows' K/V writes."""
    per_pos = 2 * s["n_kv_heads"] * s["head_dim"] * esz * s["n_layers"]
    return per_pos * (ctx * rows + rows)


def shape_str(s: dict) -> str:
    return (f"{s['n_layers']}L d{s['d']} {s['n_heads']}H/{s['n_kv_heads']}KV hd{s['head_dim']} "
            f"ffn{s['ffn']} V{s['vocab']}")


def phase_bytes(wl: dict, gamma: int, ctx: int, B: int = 1) -> dict:
    """Bytes one phase must move for B sequences: the weights once, the KV
    and embedding rows per sequence."""
    esz = 2 if wl["dtype"] == "bf16" else 4
    wd, wb = weight_bytes(wl["draft"], esz), weight_bytes(wl["base"], esz)
    draft_fwd = wd["layers"] + wd["head"] + B * wd["embed_row"]
    draft = gamma * draft_fwd + B * kv_bytes(wl["draft"], esz, ctx, 2 * gamma)
    # the gamma - 1 fuzzy forwards alone (one row per sequence each)
    fuzzy = (gamma - 1) * draft_fwd + B * kv_bytes(wl["draft"], esz, ctx, gamma - 1)
    verify = (wb["layers"] + wb["head"] + B * (gamma + 1) * wb["embed_row"]
              + B * kv_bytes(wl["base"], esz, ctx, gamma + 1))
    return {"draft_fwd": draft_fwd, "draft": draft, "fuzzy": fuzzy, "verify": verify}


def measured_traffic(kernel: str, workload: str, rows: int):
    """DRAM bytes per launch of `kernel` from the committed ncu summary
    (profiles/traffic.json), or None when there is none for this workload and
    number of activation rows, or the kernel source has changed since the
    counters were taken (sha256 of its files)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        t = json.load(f)
    for e in t.get(kernel, []):
        if e.get("workload") != workload or e.get("rows") != rows:
            continue
        h = hashlib.sha256()
        for rel in e["sources"]:
            with open(os.path.join(ROOT, rel), "rb") as f:
                h.update(f.read())
        return e["dram_bytes_per_launch"] if h.hexdigest() == e["sources_sha256"] else None
    return None


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return 6400.0, "fallback"


# ------------------------------------------------------------------ clocks
class Clocks:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--id={gpu_id}", f"--query-gpu={self.FIELDS}",
                                       "--format=csv,noheader,nounits", "-lms", "200"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.p = None

    def stop(self) -> dict:
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        self.p.wait()
        self.f.seek(0)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.f.read().splitlines():
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.f.name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ CPU oracle
# Committed tokens per phase and sequence that the CPU sample converts its
# per-forward times with.  Both arms (the GPU line's cpu_baseline and
# --impl reference) use the same figure, so they report the same quantity;
# it is the acceptance this benchmark measures on the GPU path for the
# workload at its default gamma and temperature 1.
SAMPLE_TOKENS_PER_PHASE = {
    "tiny_f32": 2.0, "qwen2.5_0.5b_7b_bf16": 1.92, "llama3_8b_70b_bf16": 1.28,
    "llama3.2_1b_selfdraft_bf16": 2.92, "qwen2.5_longctx_bf16": 2.0,
}
SAMPLE_REPS = 16       # tokens timed per layer and per head in one sample
SAMPLE_HEAD_SLICE = 8  # the output head is timed on 1/8 of its rows, then scaled


class OracleSample:
    """The CPU oracle timed on a bounded sample of the workload.

    For each model: one exact decoder layer at full width (float64 numpy, as
    the oracle runs it) over SAMPLE_REPS tokens at context prompt + 64 (the
    cache filled with random K/V), and the output head over a slice of
    ceil(V / 8) rows, each token one at a time.  The per-token cost is
    scaled to the full depth and the full vocabulary and to one speculative
    phase: calibration of the committed tokens + gamma-1 fuzzy forwards on
    the draft, gamma+1 verified tokens on the base.  Weights are drawn on the
    host (the sample needs no GPU) and built once; run() is one sample."""

    def __init__(self, wl: dict, gamma: int, tokens_per_phase: float, seed: int = 0):
        from layer_drafting_draft_b300 import synth
        from oracle import model as M
        self.M, self.wl, self.gamma, self.tpp = M, wl, gamma, tokens_per_phase
        self.ctx = wl["prompt"] + 64
        self.parts = {}
        for which in ("draft", "base"):
            full = wl[which]
            vs = -(-full["vocab"] // SAMPLE_HEAD_SLICE)
            s = dict(full, n_layers=1, vocab=vs)
            W = M.as_f64_weights(synth.make_weights(s, 7 + seed, wl["dtype"], "cpu"))
            W["embed"] = W["embed"][:4].copy()   # only a few rows are read
            shape = M.Shape(**s)
            cache = M.KVCache(shape, self.ctx + 64)
            r = np.random.default_rng(1)
            cache.K[:, :self.ctx] = r.normal(size=cache.K[:, :self.ctx].shape)
            cache.V[:, :self.ctx] = r.normal(size=cache.V[:, :self.ctx].shape)
            self.parts[which] = (W, shape, cache, full["n_layers"], full["vocab"] / vs)

    def run(self, reps: int = SAMPLE_REPS) -> dict:
        M = self.M
        per = {}
        for which, (W, shape, cache, L, vscale) in self.parts.items():
            h = W["embed"][3].copy()
            t0 = time.perf_counter()
            for i in range(reps):
                h = M.layer_exact(W, shape, 0, h, self.ctx + (i % 32), cache)
            t_layer = (time.perf_counter() - t0) / reps
            t0 = time.perf_counter()
            for i in range(reps):
                M.head_logits(W, shape, h)
            t_head = (time.perf_counter() - t0) / reps * vscale
            per[which] = L * t_layer + t_head
        gamma, tpp, wl = self.gamma, self.tpp, self.wl
        phase_s = (tpp + gamma - 1) * per["draft"] + (gamma + 1) * per["base"]
        try:
            from threadpoolctl import threadpool_info
            cores = max((i.get("num_threads", 1) for i in threadpool_info()), default=1)
        except Exception:
            cores = os.cpu_count()
        return {"value": tpp / phase_s, "unit": "tok/s", "cores": cores, "kind": "oracle",
                "sample": (f"float64 numpy oracle: one exact layer of each model at full width and "
                           f"1/{SAMPLE_HEAD_SLICE} of its output head, {reps} tokens each, context "
                           f"{self.ctx}; per-token cost scaled to {wl['draft']['n_layers']}+"
                           f"{wl['base']['n_layers']} layers and the full vocabulary, and to one phase "
                           f"of {tpp:.2f} committed tokens (gamma {gamma})"),
                "draft_forward_s": per["draft"], "base_token_s": per["base"],
                "tokens_per_phase": tpp}


def config_of(args, wl: dict, gamma: int, world: int) -> dict:
    """The workload description both arms print."""
    pb = phase_bytes(wl, gamma, wl["prompt"] + wl["max_new"] // 2, args.batch)
    return {"workload": args.workload, "draft": shape_str(wl["draft"]), "base": shape_str(wl["base"]),
            "batch": args.batch, "prompt": wl["prompt"], "max_new": wl["max_new"], "gamma": gamma,
            "k": 0 if args.layout else args.k, "mode": args.mode,
            **({"layout": args.layout} if args.layout else {}),
            "temperature": args.temperature, "sigma": args.sigma, "parallelism": f"replicas x{world}",
            "l2": f"inputs larger than L2 (weights {(pb['draft'] + pb['verify']) / 1e9:.1f} GB "
                  f"streamed per phase)"}


# ------------------------------------------------------------------ GPU arm
def run_ours(args, rank: int, world: int):
    import torch

    from layer_drafting_draft_b300 import build, synth
    from layer_drafting_draft_b300.easyspec import ES_ATTN_ONLY, ES_FULL_LAYER, EasySpec
    build.build()
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    wl = synth.WORKLOADS[args.workload]
    gamma = args.gamma or wl["gamma"]
    P, max_new, T, k = wl["prompt"], wl["max_new"], args.temperature, args.k
    draft_w, base_w, prompts = synth.make_pair(args.workload, device="cuda", sigma=args.sigma)
    B = args.batch
    if B > prompts.shape[0]:
        raise SystemExit(f"--batch {B}: the workload has {prompts.shape[0]} prompts")
    prompts = prompts[:B].numpy()
    stream = torch.cuda.Stream()
    mode = ES_FULL_LAYER if args.mode == "full" else ES_ATTN_ONLY
    max_seq = ((P + max_new + 2 * gamma + 2) + 63) // 64 * 64
    gs = None
    if args.layout:
        from layer_drafting_draft_b300 import layouts
        cands = layouts.candidates(wl["draft"]["n_layers"])
        if args.layout not in cands:
            raise SystemExit(f"--layout {args.layout}: not one of {', '.join(cands)}")
        sets = cands[args.layout]
        gs, k = layouts.starts(sets), 0
    g = EasySpec(draft_w, wl["draft"], base_w, wl["base"], wl["dtype"], B, max_seq, gamma, mode,
                 gs, stream)
    seed0 = 1000 * rank

    def one_decode(step):
        g.easyspec_prefill(prompts)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        st = g.es_decode(max_new, gamma, k, T, seed0 + step)
        ev1.record(stream)
        ev1.synchronize()
        return ev0.elapsed_time(ev1), st

    for w in range(args.warmup):
        one_decode(10_000 + w)
    barrier(world)
    torch.cuda.synchronize()
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    uuid = getattr(props, "uuid", None)
    clocks = Clocks(f"GPU-{uuid}" if uuid is not None else str(torch.cuda.current_device()))
    dec_ms, stats = [], []
    t_wall = time.perf_counter()
    for s in range(args.steps):
        ms, st = one_decode(s)
        dec_ms.append(ms)
        stats.append(st)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t_wall
    clk = clocks.stop()
    barrier(world)
    total_ms = max_over_ranks(sum(dec_ms), world)
    value = world * args.steps * B * max_new / (total_ms / 1e3)
    emitted = sum(s["emitted"] for s in stats)
    phases = sum(s["phases"] for s in stats)
    accepted = sum(s["accepted"] for s in stats)
    drafted = sum(s["drafted"] for s in stats)
    launches = sum(s["kernel_launches"] for s in stats)
    tok_per_phase = emitted / max(phases * B, 1)  # per sequence

    # ---- per-phase breakdown: one more generation with the library's part
    # timing (CUDA events around each phase part's graph launch, calibration
    # and fuzzy drafts as two graphs)
    g.easyspec_prefill(prompts)
    g.es_profile(2)
    st_parts = g.es_decode(max_new, gamma, k, T, seed0 + 777)
    parts = g.es_profile_read()
    g.es_profile(0)
    nph = max(st_parts["phases"], 1)
    calib_ms = parts["phase.calibrate"][0] / nph
    fuzzy_ms = parts["phase.fuzzy"][0] / nph
    verify_ms = parts["phase.verify"][0] / nph
    draft_ms = calib_ms + fuzzy_ms
    peak, peak_src = peaks()
    pb = phase_bytes(wl, gamma, P + max_new // 2, B)
    draft_gbs = pb["draft"] / (draft_ms * 1e-3) / 1e9
    fuzzy_gbs = pb["fuzzy"] / (fuzzy_ms * 1e-3) / 1e9
    verify_gbs = pb["verify"] / (verify_ms * 1e-3) / 1e9
    phase_roof_s = (pb["draft"] + pb["verify"]) / (peak * 1e9)
    roof_tok_s = B * tok_per_phase / phase_roof_s

    # ---- e2e through generate() with host buffers
    e2e_ms, prefill_ms = [], []
    out_host = None
    for s in range(max(2, min(args.steps, 5))):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        out_host, gst = g.generate(prompts, max_new, gamma, k, T, seed0 + 500 + s)
        e2e_ms.append((time.perf_counter() - t0) * 1e3)
        prefill_ms.append(gst["prefill_ms"])
    e2e_value = world * B * max_new / (max_over_ranks(statistics.mean(e2e_ms), world) / 1e3)

    # ---- dominant kernel: per-launch event pass over one generation
    g.easyspec_prefill(prompts)
    g.es_profile(True)
    g.es_decode(max_new, gamma, k, T, seed0 + 999)
    prof = g.es_profile_read()
    g.es_profile(False)
    top = max((kv for kv in prof.items() if kv[1][2] > 0), key=lambda kv: kv[1][0])
    name, (pms, pn, pbytes) = top
    achieved = pbytes / (pms * 1e-3) / 1e9
    total_prof_ms = sum(v[0] for v in prof.values())
    g.close()

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "tok/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": wl["dtype"], "data": "synthetic",
        "config": config_of(args, wl, gamma, world),
        "e2e": {"value": round(e2e_value, 2), "unit": "tok/s",
                "h2d_bytes_per_step": int(prompts.size * 4 + 16 + 8),
                "d2h_bytes_per_step": int(B * max_new * 4),
                "prefill_ms": round(statistics.mean(prefill_ms), 2)},
        "draft": {"tok_s": round(B * gamma / (draft_ms * 1e-3), 1), "ms_per_phase": round(draft_ms, 4),
                  "achieved_gbs": round(draft_gbs, 1), "roofline_frac": round(draft_gbs / peak, 4),
                  "bytes_per_phase": int(pb["draft"]),
                  "calibrate_ms_per_phase": round(calib_ms, 4),
                  "fuzzy": {"tok_s": round(B * (gamma - 1) / (fuzzy_ms * 1e-3), 1),
                            "ms_per_phase": round(fuzzy_ms, 4), "achieved_gbs": round(fuzzy_gbs, 1),
                            "roofline_frac": round(fuzzy_gbs / peak, 4),
                            "bytes_per_phase": int(pb["fuzzy"])}},
        "verify": {"ms_per_phase": round(verify_ms, 4), "achieved_gbs": round(verify_gbs, 1),
                   "roofline_frac": round(verify_gbs / peak, 4), "bytes_per_phase": int(pb["verify"])},
        "weight_stream_roofline": {"tok_s": round(roof_tok_s, 1), "e2e_frac": round(value / world / roof_tok_s, 4),
                                   "peak_gbs": peak, "peak_source": peak_src},
        "acceptance": {"tokens_per_phase": round(tok_per_phase, 3),
                       "rate": round(accepted / max(drafted, 1), 4)},
        "roofline": {"bound": "hbm", "kernel": name, "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": measured_traffic(name, args.workload, B * (gamma + 1)),
                     "launches": pn, "share_of_device_time": round(pms / total_prof_ms, 4),
                     "peak_source": peak_src},
        "clocks": clk, "gpu_launches": int(launches),
        "timed_wall_s": round(wall, 3),
    }
    # the CPU oracle's figure belongs to the single-GPU line only
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = OracleSample(wl, gamma, SAMPLE_TOKENS_PER_PHASE[args.workload]).run()
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_reference(args, rank: int, world: int):
    """The oracle arm: the CPU oracle timed on this host's cores, each step
    one sample exactly as the GPU line's cpu_baseline takes it."""
    if rank != 0:
        return
    from layer_drafting_draft_b300 import synth
    wl = synth.WORKLOADS[args.workload]
    gamma = args.gamma or wl["gamma"]
    sample = OracleSample(wl, gamma, SAMPLE_TOKENS_PER_PHASE[args.workload])
    for w in range(args.warmup):
        sample.run()
    vals = []
    t0 = time.perf_counter()
    for s in range(args.steps):
        vals.append(sample.run())
    wall = time.perf_counter() - t0
    v = statistics.mean(x["value"] for x in vals)
    cb = dict(vals[-1])
    cb["value"] = v
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tok/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": wall / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_of(args, wl, gamma, world),
            "cpu_baseline": cb, "e2e": {"value": v, "unit": "tok/s", "h2d_bytes_per_step": 0,
                                        "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ distributed
def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1"))


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def main():
    args = parse()
    rank, world = dist_env()
    if world > 1:
        import torch
        import torch.distributed as dist
        dist.init_process_group("nccl" if (torch.cuda.is_available() and args.impl == "ours") else "gloo")
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_ours(args, rank, world)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
