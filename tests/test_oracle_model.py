"""Pins for the oracle's decoder: closed forms, invariants, an independent
full-sequence formulation, and the layer-set rule printed on the pages."""
import copy

import numpy as np
import pytest
from scipy.special import expit

from conftest import golden_lines
from oracle import model as M
from oracle_util import tiny_pair, zero_layer


# ------------------------------------------------------------ layer sets

def test_grouping_rule_reproduces_page_example():
    want = [[int(x) for x in ln.split()] for ln in golden_lines("grouping_L32_N4.txt")]
    assert M.default_groups(32, 4) == want


def test_grouping_rule_small_cases():
    assert M.default_groups(24, 1) == [[l] for l in range(24)]
    g = M.default_groups(24, 4)
    assert g[0] == [0] and g[1] == [1, 2, 3] and g[-2] == [20, 21, 22] and g[-1] == [23]
    assert M.default_groups(24, 2)[:3] == [[0], [1], [2, 3]]
    for L in range(1, 40):
        for k in range(1, 9):
            M.check_groups(M.default_groups(L, k), L)
    with pytest.raises(ValueError):
        M.check_groups([[0, 2], [1]], 3)


# ------------------------------------------------------------ primitives

def test_rope_identity_at_zero_and_norm_preserving():
    r = np.random.default_rng(0)
    x = r.normal(size=(3, 16))
    assert np.array_equal(M.rope(x, 0, 1e4), x)
    y = M.rope(x, 37, 1e4)
    assert np.allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)


def test_rope_relative_position_invariance():
    r = np.random.default_rng(1)
    q, k = r.normal(size=(1, 32)), r.normal(size=(1, 32))
    a = (M.rope(q, 10, 1e4) * M.rope(k, 3, 1e4)).sum()
    b = (M.rope(q, 107, 1e4) * M.rope(k, 100, 1e4)).sum()
    assert abs(a - b) < 1e-10


def test_rope_pairs_i_with_i_plus_half():
    # a unit vector on element 1 rotates into element 1 + hd/2 only
    hd = 8
    x = np.zeros((1, hd)); x[0, 1] = 1.0
    y = M.rope(x, 5, 100.0)
    ang = 5 * 100.0 ** (-2.0 * 1 / hd)
    want = np.zeros(hd); want[1] = np.cos(ang); want[1 + hd // 2] = np.sin(ang)
    assert np.allclose(y[0], want, atol=1e-15)


def test_single_position_attention_returns_v_of_mapped_kv_head():
    r = np.random.default_rng(2)
    H, Hkv, hd = 6, 2, 4
    q = r.normal(size=(H, hd))
    K = r.normal(size=(1, Hkv, hd))
    V = r.normal(size=(1, Hkv, hd))
    out = M.attend(q, K, V, H, Hkv).reshape(H, hd)
    for h in range(H):
        assert np.allclose(out[h], V[0, h // (H // Hkv)])


def test_attention_uniform_when_keys_equal():
    r = np.random.default_rng(3)
    K = np.repeat(r.normal(size=(1, 1, 4)), 5, axis=0)
    V = r.normal(size=(5, 1, 4))
    out = M.attend(r.normal(size=(1, 4)), K, V, 1, 1)
    assert np.allclose(out, V[:, 0].mean(axis=0))


def test_rmsnorm_gain_free_preserves_cosine():
    # reply on Table 3: with a normalisation at the module entry,
    # cos(h1, h2) == cos(h1', h2')
    r = np.random.default_rng(4)
    h1, h2 = r.normal(size=64) * 3, r.normal(size=64) * 0.1
    n1, n2 = M.rms_norm(h1, 1.0, 0.0), M.rms_norm(h2, 1.0, 0.0)
    cos = lambda a, b: a @ b / np.linalg.norm(a) / np.linalg.norm(b)
    assert abs(cos(h1, h2) - cos(n1, n2)) < 1e-14
    assert abs(np.sqrt(np.mean(n1 * n1)) - 1.0) < 1e-14


# ------------------------------------------------------------ forwards

def test_zeroed_layers_give_head_of_embedding():
    Wd, sd, _, _ = tiny_pair(0)
    W = copy.deepcopy(Wd)
    W["layers"] = [zero_layer(lw) for lw in W["layers"]]
    cache = M.KVCache(sd, 8)
    for pos, t in enumerate([5, 9, 1]):
        z = M.forward_exact(W, sd, t, pos, cache)
        e = W["embed"][t]
        want = W["lm_head"] @ (e / np.sqrt(np.mean(e * e) + sd.eps))
        assert np.allclose(z, want, rtol=1e-13, atol=1e-15)


def _textbook_logits(W, s: M.Shape, tokens):
    """Full-sequence causal forward written independently: complex-number
    rotary embedding, a masked score matrix, repeated KV heads."""
    T, hd, H, Hkv = len(tokens), s.head_dim, s.n_heads, s.n_kv_heads
    half = hd // 2
    freq = 1.0 / s.rope_theta ** (np.arange(half) * 2.0 / hd)
    rot = np.exp(1j * np.outer(np.arange(T), freq))           # [T, half]

    def rotate(x):                                              # x [T, n, hd]
        c = (x[..., :half] + 1j * x[..., half:]) * rot[:, None, :]
        return np.concatenate([c.real, c.imag], axis=-1)

    def norm(x, g):
        return x * (np.mean(x ** 2, axis=-1, keepdims=True) + s.eps) ** -0.5 * g

    mask = np.triu(np.full((T, T), -np.inf), 1)
    x = W["embed"][np.asarray(tokens)]
    for lw in W["layers"]:
        y = norm(x, lw["attn_norm"])
        q = rotate((y @ lw["wq"].T).reshape(T, H, hd))
        k = rotate((y @ lw["wk"].T).reshape(T, Hkv, hd))
        v = (y @ lw["wv"].T).reshape(T, Hkv, hd)
        k = np.repeat(k, H // Hkv, axis=1)
        v = np.repeat(v, H // Hkv, axis=1)
        sc = np.einsum("thd,shd->hts", q, k) / np.sqrt(hd) + mask
        pr = np.exp(sc - sc.max(-1, keepdims=True))
        pr /= pr.sum(-1, keepdims=True)
        a = np.einsum("hts,shd->thd", pr, v).reshape(T, H * hd)
        x = x + a @ lw["wo"].T
        y = norm(x, lw["mlp_norm"])
        g = y @ lw["wgate"].T
        x = x + (g * expit(g) * (y @ lw["wup"].T)) @ lw["wdown"].T
    return norm(x, W["final_norm"]) @ W["lm_head"].T


@pytest.mark.parametrize("which", ["draft", "base"])
def test_incremental_forward_matches_full_sequence_textbook(which):
    Wd, sd, Wb, sb = tiny_pair(1, std=0.2)
    W, s = (Wd, sd) if which == "draft" else (Wb, sb)
    toks = [3, 17, 17, 40, 2, 63, 0, 11]
    cache = M.KVCache(s, 16)
    inc = np.array([M.forward_exact(W, s, t, p, cache) for p, t in enumerate(toks)])
    ref = _textbook_logits(W, s, toks)
    assert np.max(np.abs(inc - ref)) < 1e-11 * max(1.0, np.max(np.abs(ref)))


@pytest.mark.parametrize("which", ["draft", "base"])
def test_block_forward_matches_textbook_and_token_by_token(which):
    """The block forward over a whole sequence equals the independent
    textbook forward; a block that starts after a token-by-token prefix
    leaves the same cache and logits as continuing token by token."""
    Wd, sd, Wb, sb = tiny_pair(3, std=0.2)
    W, s = (Wd, sd) if which == "draft" else (Wb, sb)
    toks = [3, 17, 17, 40, 2, 63, 0, 11, 9, 9, 30]
    ref = _textbook_logits(W, s, toks)
    cb = M.KVCache(s, 16)
    blk = M.forward_block(W, s, toks, 0, cb)
    assert np.max(np.abs(blk - ref)) < 1e-11 * max(1.0, np.max(np.abs(ref)))
    # prefix of 4 tokens one at a time, then the remaining 7 as one block
    ci, cm = M.KVCache(s, 16), M.KVCache(s, 16)
    inc = [M.forward_exact(W, s, t, p, ci) for p, t in enumerate(toks)]
    for p, t in enumerate(toks[:4]):
        M.forward_exact(W, s, t, p, cm)
    tail = M.forward_block(W, s, toks[4:], 4, cm, logit_rows=[0, 6])
    assert np.max(np.abs(tail - np.array([inc[4], inc[10]]))) < 1e-11 * max(1.0, np.max(np.abs(ref)))
    n = len(toks)
    assert np.max(np.abs(cm.K[:, :n] - ci.K[:, :n])) < 1e-12
    assert np.max(np.abs(cm.V[:, :n] - ci.V[:, :n])) < 1e-12
    assert np.max(np.abs(cb.K[:, :n] - ci.K[:, :n])) < 1e-12


def _prefill(W, s, toks, cache):
    for p, t in enumerate(toks):
        M.forward_exact(W, s, t, p, cache)


@pytest.mark.parametrize("mode", [M.ATTN_ONLY, M.FULL_LAYER])
def test_set_size_one_is_sequential_bitwise(mode):
    Wd, sd, _, _ = tiny_pair(2, std=0.2)
    c1, c2 = M.KVCache(sd, 8), M.KVCache(sd, 8)
    _prefill(Wd, sd, [1, 2, 3], c1)
    _prefill(Wd, sd, [1, 2, 3], c2)
    z1 = M.forward_exact(Wd, sd, 7, 3, c1)
    z2 = M.forward_fuzzy(Wd, sd, 7, 3, c2, M.default_groups(sd.n_layers, 1), mode)
    assert np.array_equal(z1, z2) and np.array_equal(c1.K, c2.K) and np.array_equal(c1.V, c2.V)


def test_attn_only_with_zero_wo_is_sequential():
    Wd, sd, _, _ = tiny_pair(3, std=0.2)
    for lw in Wd["layers"]:
        lw["wo"][:] = 0.0
    c1, c2 = M.KVCache(sd, 8), M.KVCache(sd, 8)
    _prefill(Wd, sd, [4, 5], c1)
    _prefill(Wd, sd, [4, 5], c2)
    z1 = M.forward_exact(Wd, sd, 9, 2, c1)
    z2 = M.forward_fuzzy(Wd, sd, 9, 2, c2, [[0, 1, 2, 3]], M.ATTN_ONLY)
    assert np.array_equal(z1, z2)


def _set_output(W, s, group, h, mode, toks, Wprefix=None):
    cache = M.KVCache(s, 8)
    _prefill(W if Wprefix is None else Wprefix, s, toks, cache)
    return M.group_fuzzy(W, s, group, h, len(toks), cache, mode)


@pytest.mark.parametrize("mode", [M.ATTN_ONLY, M.FULL_LAYER])
def test_set_deltas_add_up(mode):
    """FULL_LAYER: a set's delta is the sum of its layers' deltas, each taken
    from the set input.  ATTN_ONLY: the same holds for the attention deltas
    when the MLPs are zero.  Checked by zeroing all but one layer of the set."""
    Wd, sd, _, _ = tiny_pair(4, std=0.2)
    if mode == M.ATTN_ONLY:
        for lw in Wd["layers"]:
            lw["wdown"][:] = 0.0
    h = np.random.default_rng(5).normal(size=sd.d)
    toks = [8, 1, 30]
    group = [1, 2]
    full = _set_output(Wd, sd, group, h, mode, toks)
    parts = []
    for keep in group:
        W = copy.deepcopy(Wd)
        for other in group:
            if other != keep:
                W["layers"][other] = zero_layer(W["layers"][other])
        parts.append(_set_output(W, sd, group, h, mode, toks, Wprefix=Wd) - h)
    assert np.allclose(full - h, parts[0] + parts[1], rtol=1e-12, atol=1e-14)


def test_full_layer_set_differs_from_sequential_and_attn_only():
    Wd, sd, _, _ = tiny_pair(6, std=0.2)
    h = np.random.default_rng(7).normal(size=sd.d)
    a = _set_output(Wd, sd, [1, 2], h, M.FULL_LAYER, [1, 2])
    b = _set_output(Wd, sd, [1, 2], h, M.ATTN_ONLY, [1, 2])
    assert not np.allclose(a, b)


def test_fuzzy_forward_writes_only_its_position():
    Wd, sd, _, _ = tiny_pair(8, std=0.2)
    c = M.KVCache(sd, 8)
    _prefill(Wd, sd, [1, 2, 3], c)
    K0, V0 = c.K.copy(), c.V.copy()
    M.forward_fuzzy(Wd, sd, 5, 3, c, [[0], [1, 2], [3]], M.FULL_LAYER)
    assert np.array_equal(c.K[:, :3], K0[:, :3]) and np.array_equal(c.K[:, 4:], K0[:, 4:])
    assert np.array_equal(c.V[:, :3], V0[:, :3])
    # layer 0 is a singleton whose input is the exact embedding: exact entry
    ce = M.KVCache(sd, 8)
    _prefill(Wd, sd, [1, 2, 3, 5], ce)
    assert np.array_equal(c.K[0, 3], ce.K[0, 3])
    assert not np.allclose(c.K[2, 3], ce.K[2, 3])


def _exact_on(W, s, l, h, pos, cache):
    return M.layer_exact(W, s, l, h, pos, cache)


def _variant(W, l, key):
    V = copy.deepcopy(W)
    V["layers"][l][key] = np.zeros_like(V["layers"][l][key])
    return V


@pytest.mark.parametrize("mode", [M.ATTN_ONLY, M.FULL_LAYER])
def test_set_layers_match_exact_layers_on_set_input(mode):
    """Each layer of a set is its own exact layer fed the set input: its K/V
    entry equals the exact layer's on that input, and the set output is
    rebuilt from exact single-layer evaluations (a separate code path):
      attention delta A_j(h) = exact_j[Wdown = 0](h) - h
      MLP delta on input y   = exact_j[Wo = 0](y) - y
    FULL_LAYER: out = h + sum_j (A_j(h) + MLPdelta_j(h))
    ATTN_ONLY : x = h; for j: x = exact_j[Wo=0](x + A_j(h))."""
    Wd, sd, _, _ = tiny_pair(9, std=0.2)
    toks, group = [8, 1, 30], [1, 2]
    pos = len(toks)
    h = np.random.default_rng(10).normal(size=sd.d)
    base = M.KVCache(sd, 8)
    _prefill(Wd, sd, toks, base)

    cf = copy.deepcopy(base)
    out = M.group_fuzzy(Wd, sd, group, h, pos, cf, mode)

    A, mlp_on_h = {}, {}
    for l in group:
        c = copy.deepcopy(base)
        A[l] = _exact_on(_variant(Wd, l, "wdown"), sd, l, h, pos, c) - h
        assert np.array_equal(cf.K[l, pos], c.K[l, pos]) and np.array_equal(cf.V[l, pos], c.V[l, pos])
        mlp_on_h[l] = _exact_on(_variant(Wd, l, "wo"), sd, l, h, pos, copy.deepcopy(base)) - h
    if mode == M.FULL_LAYER:
        want = h + sum(A[l] + mlp_on_h[l] for l in group)
    else:
        x = h
        for l in group:
            x = _exact_on(_variant(Wd, l, "wo"), sd, l, x + A[l], pos, copy.deepcopy(base))
        want = x
    assert np.allclose(out, want, rtol=1e-12, atol=1e-14)


def test_round_bf16_matches_the_library_conversion_and_ties_to_even():
    """round_bf16 is float32 rounding followed by round-to-nearest-even to
    8 significant bits: equal to torch's bfloat16 conversion of the float32
    value, with the halfway cases going to the even neighbour."""
    import torch
    r = np.random.default_rng(5)
    x = np.concatenate([r.normal(size=4000) * 10.0 ** r.integers(-6, 6, size=4000),
                        [0.0, -0.0, 1.0, -3.5, 65504.0, 1e-40]])
    want = torch.tensor(x.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(M.round_bf16(x), want)
    ulp = 2.0 ** -7
    assert M.round_bf16(1 + ulp / 2) == 1.0                 # tie, 1.0 is even
    assert M.round_bf16(1 + 3 * ulp / 2) == 1 + 2 * ulp     # tie, 1 + 2 ulp is even
    assert M.round_bf16(-(1 + 3 * ulp / 2)) == -(1 + 2 * ulp)
    assert M.round_bf16(1 + ulp / 2 + 1e-6) == 1 + ulp      # above the tie


def test_bf16_cache_stores_rounded_entries_that_the_forward_reads():
    Wd, sd, _, _ = tiny_pair(6, std=0.2)
    toks = [4, 8, 15, 16, 23, 42]
    c64, c16 = M.KVCache(sd, 8), M.KVCache(sd, 8, "bf16")
    z64 = [M.forward_exact(Wd, sd, t, p, c64) for p, t in enumerate(toks)]
    z16 = [M.forward_exact(Wd, sd, t, p, c16) for p, t in enumerate(toks)]
    n = len(toks)
    assert np.array_equal(M.round_bf16(c16.K[:, :n]), c16.K[:, :n])
    assert np.array_equal(M.round_bf16(c16.V[:, :n]), c16.V[:, :n])
    # layer 0 at the first position sees only the embedding: its entries are
    # the rounded float64 ones
    assert np.array_equal(c16.K[0, 0], M.round_bf16(c64.K[0, 0]))
    assert np.array_equal(c16.V[0, 0], M.round_bf16(c64.V[0, 0]))
    # later logits move by about the bf16 rounding of K/V, no more
    d = np.max(np.abs(np.array(z16) - np.array(z64)))
    assert 0 < d < 2e-2 * np.max(np.abs(z64))
    # the block forward stores the same rounded entries
    cb = M.KVCache(sd, 8, "bf16")
    zb = M.forward_block(Wd, sd, toks, 0, cb)
    assert np.max(np.abs(zb - np.array(z16))) < 1e-9
    assert np.max(np.abs(cb.K[:, :n] - c16.K[:, :n])) <= 2.0 ** -8 * np.max(np.abs(c16.K[:, :n]))
