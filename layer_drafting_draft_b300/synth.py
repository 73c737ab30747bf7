"""Seeded synthetic inputs: model shapes, random-init weights and prompts.

This module holds no arithmetic of the decoding method; it only draws the
inputs that both the CUDA path and its checker consume.  Weights are i.i.d.
N(0, std^2) (std 0.02), RMSNorm gains are 1, prompts are i.i.d. uniform token
ids -- the recipe of the synthetic workloads (no checkpoints or datasets are
used anywhere).

Draw order (fixed, so a seed names one model): embed; for each layer
attn_norm (ones), wq, wk, wv, wo, mlp_norm (ones), wgate, wup, wdown;
final_norm (ones); lm_head.  Layouts are row-major [out_features,
in_features]: wq [H*hd, d], wk/wv [Hkv*hd, d], wo [d, H*hd], wgate/wup
[F, d], wdown [d, F], embed/lm_head [V, d].
"""
from __future__ import annotations

import torch

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


def shape(n_layers, d, n_heads, n_kv_heads, ffn, vocab, rope_theta, head_dim=None, eps=1e-6):
    return dict(n_layers=n_layers, d=d, n_heads=n_heads, n_kv_heads=n_kv_heads,
                head_dim=head_dim if head_dim is not None else d // n_heads,
                ffn=ffn, vocab=vocab, rope_theta=float(rope_theta), eps=float(eps))


# Workloads: draft/base pairs shaped like the same-series pairs the method is
# evaluated on (LLaMA-3 and Qwen families), random-initialised.
WORKLOADS = {
    "tiny_f32": dict(
        draft=shape(4, 128, 4, 2, 344, 512, 1e4),
        base=shape(8, 256, 8, 4, 688, 512, 1e4),
        dtype="f32", seed=0, groups=[[0, 1], [2, 3]], batch=1, prompt=32,
        gamma=4, max_new=64),
    "qwen2.5_0.5b_7b_bf16": dict(
        draft=shape(24, 896, 14, 2, 4864, 151936, 1e6),
        base=shape(28, 3584, 28, 4, 18944, 151936, 1e6),
        dtype="bf16", seed=1, groups=None, batch=1, prompt=256, gamma=4,
        max_new=128, ks=(1, 2, 4)),
    "llama3_8b_70b_bf16": dict(
        draft=shape(32, 4096, 32, 8, 14336, 128256, 5e5),
        base=shape(80, 8192, 64, 8, 28672, 128256, 5e5),
        dtype="bf16", seed=2, groups=None, batch=1, prompt=512, gamma=4,
        max_new=128, ks=(2, 4, 8)),
    "llama3.2_1b_selfdraft_bf16": dict(
        draft=shape(16, 2048, 32, 8, 8192, 128256, 5e5),
        base=shape(16, 2048, 32, 8, 8192, 128256, 5e5),
        dtype="bf16", seed=3, groups=None, batch=1, prompt=128, gamma=6,
        max_new=128, ks=(1, 2, 4), sigmas=(0.05, 0.2)),
    "qwen2.5_longctx_bf16": dict(
        draft=shape(24, 896, 14, 2, 4864, 151936, 1e6),
        base=shape(28, 3584, 28, 4, 18944, 151936, 1e6),
        dtype="bf16", seed=4, groups=None, batch=16, prompt=4096, gamma=4,
        max_new=128, ks=(4,)),
}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def make_weights(s: dict, seed: int, dtype: str = "f32", device="cpu", std: float = 0.02):
    """Random-init weights of shape dict ``s`` (see module docstring)."""
    dev = torch.device(device)
    g = _gen(seed, dev)
    tdt = DTYPES[dtype]
    d, hd = s["d"], s["head_dim"]
    qd, kvd, F, V = s["n_heads"] * hd, s["n_kv_heads"] * hd, s["ffn"], s["vocab"]

    def rnd(*shp):
        t = torch.randn(*shp, generator=g, device=dev, dtype=torch.float32)
        return (t * std).to(tdt)

    def ones(n):
        return torch.ones(n, device=dev, dtype=tdt)

    w = {"embed": rnd(V, d), "layers": []}
    for _ in range(s["n_layers"]):
        w["layers"].append({
            "attn_norm": ones(d), "wq": rnd(qd, d), "wk": rnd(kvd, d), "wv": rnd(kvd, d),
            "wo": rnd(d, qd), "mlp_norm": ones(d), "wgate": rnd(F, d), "wup": rnd(F, d),
            "wdown": rnd(d, F)})
    w["final_norm"] = ones(d)
    w["lm_head"] = rnd(V, d)
    return w


def perturbed_copy(w: dict, sigma: float, seed: int, std: float = 0.02):
    """w + N(0, (sigma*std)^2) on every matrix (gains untouched): a draft that
    agrees with its base to a controlled degree."""
    ref = w["embed"]
    g = _gen(seed, ref.device)

    def pert(t):
        if t.dim() < 2:
            return t.clone()
        n = torch.randn(t.shape, generator=g, device=t.device, dtype=torch.float32)
        return (t.float() + n * (sigma * std)).to(t.dtype)

    out = {k: pert(w[k]) for k in ("embed", "final_norm", "lm_head")}
    out["layers"] = [{k: pert(v) for k, v in lw.items()} for lw in w["layers"]]
    return out


def make_prompts(batch: int, length: int, vocab: int, seed: int) -> torch.Tensor:
    """[batch, length] int32 token ids, i.i.d. uniform over the vocabulary."""
    g = _gen(seed, torch.device("cpu"))
    return torch.randint(0, vocab, (batch, length), generator=g, dtype=torch.int64).to(torch.int32)


def make_pair(name: str, device="cpu", sigma: float | None = None):
    """(draft weights, base weights, prompts) for a named workload.

    Sub-seeds: draft 1000*seed+1, base 1000*seed+2, prompts 1000*seed+3,
    perturbation (self-draft pairs) 1000*seed+4.
    """
    wl = WORKLOADS[name]
    sd = 1000 * wl["seed"]
    base = make_weights(wl["base"], sd + 2, wl["dtype"], device)
    if sigma is not None:
        draft = perturbed_copy(base, sigma, sd + 4)
    else:
        draft = make_weights(wl["draft"], sd + 1, wl["dtype"], device)
    prompts = make_prompts(wl["batch"], wl["prompt"], wl["base"]["vocab"], sd + 3)
    return draft, base, prompts
