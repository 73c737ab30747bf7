"""Llama-style decoder, exact and layer-parallel ("fuzzy"), in float64 numpy.

TEST INFRASTRUCTURE ONLY -- see the package docstring.

Model (the configs' "Llama-style" pairs; the pages use LLaMA-3 and Qwen2
families and fix no further detail):
  h = E[token]
  per layer l:
    x = RMSNorm(h; g_attn_l)          RMSNorm(x; g) = x / sqrt(mean(x^2) + eps) * g
    q, k, v = Wq x, Wk x, Wv x        (no biases)
    RoPE on q and k at the token's position ("rotate half" pairing of
      element i with i + hd/2, frequency theta**(-2i/hd))
    K/V cache[l][pos] = k, v
    a = softmax(q K^T / sqrt(hd)) V   grouped-query: query head h reads
                                      kv head h // (H / Hkv), causal
    h = h + Wo a
    h = h + Wdown(silu(Wgate y) * Wup y),  y = RMSNorm(h; g_mlp_l)
  logits = Wlm RMSNorm(h; g_final)    (untied from E)

Layer-parallel ("fuzzy") speculation, EasySpec (arXiv abstract page; OpenReview
discussion page, replies on Figure 1(b) / Table 4 and on Table 3): the layers of
one layer set all read the set's input hidden state instead of their
predecessor's output, so they can run at the same time.  Two readings are
built, selected by ``mode``:

  ATTN_ONLY  (the discussion page: only the attention sublayers of a set run in
             parallel, the MLPs stay sequential -- reply on Figure 1(b)/Table 4)
             A_j = Wo_j Attn_j(RMSNorm(h; g_attn_j)) for every j in the set,
             then x = h; for j in set order: x += A_j; x += MLP_j(RMSNorm(x)).
  FULL_LAYER (attention and MLP of every layer of the set read the set input
             and their residual deltas are summed onto it)
             out = h + sum_j [ A_j + MLP_j(RMSNorm(h; g_mlp_j)) ].

A set of a single layer is not parallelised: it runs the exact layer above in
both modes (the discussion page describes layer sets of size one, the first
and the last layer, as left un-parallelised; with set size 1 the model is the
original sequential one -- "no modifications to the original model
architecture", reply on Table 4 / Appendix B.1).

K/V written by a set's layers during a fuzzy forward are computed from the set
input, i.e. they are the "fuzzy" cache entries (reply on Figure 2).

Layer-set rule (reply on Table 4 / Appendix B.1; the sentence is garbled on
the page, the reading below is the only one that reproduces its own 32-layer,
N=4 example "0, 1~4, 4~7, ..., 28~30" with 28, 29, 30 forming a 3-set because
31 is the last layer): layer 0 and layer L-1 are singletons; layers 1..L-2 are
cut into the aligned blocks [mN, mN+N-1], the first and last blocks clipped.

``forward_block`` is the exact forward of a run of consecutive tokens in one
go (matrix products over the run), for long prompts; it computes what
``forward_exact`` computes token by token.

Parity: pinned by tests/test_oracle_model.py (closed forms for zeroed weights,
RoPE identity at position 0 and relative-position invariance, single-position
attention, an independent full-sequence causal forward, cosine invariance of
gain-free RMSNorm (reply on Table 3), set size 1 == sequential, brute-force
delta sums for FULL_LAYER, the grouping example, the block forward equal to
the token-by-token one).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

ATTN_ONLY = 0
FULL_LAYER = 1


@dataclass(frozen=True)
class Shape:
    n_layers: int
    d: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    rope_theta: float
    eps: float = 1e-6

    @property
    def q_dim(self) -> int:
        return self.n_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim


def as_f64_weights(w: dict) -> dict:
    """Copy a weight dict (numpy / torch tensors of any float dtype) to float64."""
    def cvt(t):
        if hasattr(t, "detach"):
            t = t.detach().to("cpu").float().numpy()
        return np.asarray(t, dtype=np.float64)
    out = {k: cvt(w[k]) for k in ("embed", "lm_head", "final_norm")}
    out["layers"] = [{k: cvt(v) for k, v in lw.items()} for lw in w["layers"]]
    return out


# ----------------------------------------------------------------- primitives

def rms_norm(x, g, eps):
    return x / np.sqrt(np.mean(x * x) + eps) * g


def silu(x):
    return x / (1.0 + np.exp(-x))


def rope(xh, pos: int, theta: float):
    """Rotate each head vector of ``xh`` [n, hd] to position ``pos``."""
    hd = xh.shape[-1]
    half = hd // 2
    i = np.arange(half, dtype=np.float64)
    ang = pos * theta ** (-2.0 * i / hd)
    c, s = np.cos(ang), np.sin(ang)
    a, b = xh[..., :half], xh[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def attend(q, K, V, n_heads: int, n_kv: int):
    """One query position over cached keys/values.

    q : [H, hd]; K, V : [T, Hkv, hd] (positions 0..T-1, all visible).
    Returns the concatenated head outputs [H*hd].
    """
    hd = q.shape[-1]
    group = n_heads // n_kv
    out = np.empty((n_heads, hd))
    for h in range(n_heads):
        kvh = h // group
        s = K[:, kvh, :] @ q[h] / np.sqrt(hd)
        s = np.exp(s - s.max())
        out[h] = (s / s.sum()) @ V[:, kvh, :]
    return out.reshape(-1)


def round_bf16(x):
    """Values of x (float64) as stored in bfloat16: rounded to float32, then
    to the nearest bfloat16 (8 significant bits), ties to even, returned as
    float64.  A bfloat16 is the upper half of a float32's bit pattern."""
    b = np.ascontiguousarray(np.asarray(x, dtype=np.float32)).view(np.uint32).astype(np.uint64)
    keep = b >> 16
    rest = b & 0xFFFF
    up = (rest > 0x8000) | ((rest == 0x8000) & ((keep & 1) == 1))
    keep = keep + up.astype(np.uint64)
    return ((keep << 16).astype(np.uint32)).view(np.float32).astype(np.float64)


class KVCache:
    """Per-model cache: K, V of shape [L, max_len, Hkv, hd] (float64).

    ``dtype`` is the storage precision of the entries: "f64" keeps them as
    computed; "bf16" stores round_bf16 of every entry (a bf16 model's cache),
    and every later read, the writing position's own included, sees the
    stored value."""

    def __init__(self, shape: Shape, max_len: int, dtype: str = "f64"):
        if dtype not in ("f64", "bf16"):
            raise ValueError("cache dtype must be 'f64' or 'bf16'")
        self.K = np.zeros((shape.n_layers, max_len, shape.n_kv_heads, shape.head_dim))
        self.V = np.zeros_like(self.K)
        self.store = round_bf16 if dtype == "bf16" else (lambda x: x)


# ---------------------------------------------------------------- sublayers

def attn_delta(lw, shape: Shape, x_normed, pos: int, cache: KVCache, l: int):
    """Wo * Attn(x) for layer l at ``pos``; writes K/V[l][pos]."""
    hd = shape.head_dim
    q = (lw["wq"] @ x_normed).reshape(shape.n_heads, hd)
    k = (lw["wk"] @ x_normed).reshape(shape.n_kv_heads, hd)
    v = (lw["wv"] @ x_normed).reshape(shape.n_kv_heads, hd)
    q = rope(q, pos, shape.rope_theta)
    k = rope(k, pos, shape.rope_theta)
    cache.K[l, pos] = cache.store(k)
    cache.V[l, pos] = cache.store(v)
    a = attend(q, cache.K[l, : pos + 1], cache.V[l, : pos + 1],
               shape.n_heads, shape.n_kv_heads)
    return lw["wo"] @ a


def mlp_delta(lw, x_normed):
    return lw["wdown"] @ (silu(lw["wgate"] @ x_normed) * (lw["wup"] @ x_normed))


def layer_exact(W, shape: Shape, l: int, h, pos: int, cache: KVCache):
    lw = W["layers"][l]
    h = h + attn_delta(lw, shape, rms_norm(h, lw["attn_norm"], shape.eps), pos, cache, l)
    return h + mlp_delta(lw, rms_norm(h, lw["mlp_norm"], shape.eps))


def group_fuzzy(W, shape: Shape, group, h, pos: int, cache: KVCache, mode: int):
    """One layer set (>= 2 layers) run layer-parallel on the set input ``h``."""
    A = [attn_delta(W["layers"][l], shape,
                    rms_norm(h, W["layers"][l]["attn_norm"], shape.eps),
                    pos, cache, l) for l in group]
    if mode == ATTN_ONLY:
        x = h
        for j, l in enumerate(group):
            lw = W["layers"][l]
            x = x + A[j]
            x = x + mlp_delta(lw, rms_norm(x, lw["mlp_norm"], shape.eps))
        return x
    if mode == FULL_LAYER:
        x = h
        for j, l in enumerate(group):
            lw = W["layers"][l]
            x = x + A[j]
            x = x + mlp_delta(lw, rms_norm(h, lw["mlp_norm"], shape.eps))
        return x
    raise ValueError(f"unknown mode {mode}")


# ---------------------------------------------------------------- grouping

def default_groups(n_layers: int, k: int):
    """Layer sets for set size ``k`` (reply on Table 4 / Appendix B.1)."""
    if k < 1:
        raise ValueError("set size must be >= 1")
    if k == 1 or n_layers <= 2:
        return [[l] for l in range(n_layers)]
    groups = [[0]]
    inner = list(range(1, n_layers - 1))
    start = 0
    while start < n_layers:
        block = [l for l in range(start, start + k) if l in inner]
        if block:
            groups.append(block)
        start += k
    groups.append([n_layers - 1])
    return groups


def check_groups(groups, n_layers: int):
    flat = [l for g in groups for l in g]
    if flat != list(range(n_layers)) or any(len(g) == 0 for g in groups):
        raise ValueError("layer sets must cover 0..L-1 once, in order")


# ---------------------------------------------------------------- forwards

def embed(W, token: int):
    return W["embed"][token].copy()


def head_logits(W, shape: Shape, h):
    return W["lm_head"] @ rms_norm(h, W["final_norm"], shape.eps)


def forward_exact(W, shape: Shape, token: int, pos: int, cache: KVCache,
                  return_hidden: bool = False):
    """Exact sequential forward of one token; returns float64 logits."""
    h = embed(W, token)
    hidden = [h]
    for l in range(shape.n_layers):
        h = layer_exact(W, shape, l, h, pos, cache)
        hidden.append(h)
    z = head_logits(W, shape, h)
    return (z, hidden) if return_hidden else z


def forward_fuzzy(W, shape: Shape, token: int, pos: int, cache: KVCache,
                  groups, mode: int, return_hidden: bool = False):
    """Layer-parallel forward of one token over the layer sets ``groups``.

    ``hidden`` holds the input of every layer set followed by the final
    hidden state.
    """
    h = embed(W, token)
    hidden = [h]
    for g in groups:
        if len(g) == 1:
            h = layer_exact(W, shape, g[0], h, pos, cache)
        else:
            h = group_fuzzy(W, shape, g, h, pos, cache, mode)
        hidden.append(h)
    z = head_logits(W, shape, h)
    return (z, hidden) if return_hidden else z


# ------------------------------------------------------- block forward (long prompts)

def rms_norm_rows(X, g, eps):
    """rms_norm applied to every row of X [T, d]."""
    return X / np.sqrt(np.mean(X * X, axis=-1, keepdims=True) + eps) * g


def rope_rows(x, pos, theta: float):
    """rope() of every row: x [T, n, hd], row t rotated to position pos[t]."""
    hd = x.shape[-1]
    half = hd // 2
    i = np.arange(half, dtype=np.float64)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * theta ** (-2.0 * i / hd)
    c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def attend_rows(q, K, V, pos, n_heads: int, n_kv: int):
    """attend() for several query rows at once.

    q : [T, H, hd] (row t at position pos[t]); K, V : [P, Hkv, hd] with P >
    max(pos).  Row t sees positions 0..pos[t] (causal).  Returns [T, H*hd].
    """
    T, _, hd = q.shape
    group = n_heads // n_kv
    visible = np.arange(K.shape[0])[None, :] <= np.asarray(pos)[:, None]
    out = np.empty((T, n_heads, hd))
    for h in range(n_heads):
        kvh = h // group
        s = q[:, h, :] @ K[:, kvh, :].T / np.sqrt(hd)
        s = np.where(visible, s, -np.inf)
        s = np.exp(s - s.max(axis=-1, keepdims=True))
        out[:, h] = (s / s.sum(axis=-1, keepdims=True)) @ V[:, kvh, :]
    return out.reshape(T, -1)


def forward_block(W, shape: Shape, tokens, pos0: int, cache: KVCache, logit_rows=None):
    """Exact forward of consecutive tokens, token t at position pos0 + t.

    The result is that of calling forward_exact on each token in order (the
    same exact model, written with matrix products over the block): every
    row writes its K/V at its position and attends to positions 0..its own,
    which for rows of the block include the block's earlier rows.  Returns
    the float64 logits of the rows listed in ``logit_rows`` (all rows when
    None), [len(rows), V].
    """
    T = len(tokens)
    pos = pos0 + np.arange(T)
    hd = shape.head_dim
    H = W["embed"][np.asarray(tokens, dtype=np.int64)].astype(np.float64)
    for l in range(shape.n_layers):
        lw = W["layers"][l]
        X = rms_norm_rows(H, lw["attn_norm"], shape.eps)
        q = rope_rows((X @ lw["wq"].T).reshape(T, shape.n_heads, hd), pos, shape.rope_theta)
        k = rope_rows((X @ lw["wk"].T).reshape(T, shape.n_kv_heads, hd), pos, shape.rope_theta)
        v = (X @ lw["wv"].T).reshape(T, shape.n_kv_heads, hd)
        cache.K[l, pos0:pos0 + T] = cache.store(k)
        cache.V[l, pos0:pos0 + T] = cache.store(v)
        a = attend_rows(q, cache.K[l, :pos0 + T], cache.V[l, :pos0 + T], pos,
                        shape.n_heads, shape.n_kv_heads)
        H = H + a @ lw["wo"].T
        Y = rms_norm_rows(H, lw["mlp_norm"], shape.eps)
        H = H + (silu(Y @ lw["wgate"].T) * (Y @ lw["wup"].T)) @ lw["wdown"].T
    rows = np.arange(T) if logit_rows is None else np.asarray(logit_rows, dtype=np.int64)
    if len(rows) == 0:
        return np.zeros((0, shape.vocab))
    return rms_norm_rows(H[rows], W["final_norm"], shape.eps) @ W["lm_head"].T
