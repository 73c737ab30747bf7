"""EasySpec speculative decoding loop (oracle side), one sequence at a time.

TEST INFRASTRUCTURE ONLY -- see the package docstring.

Stage order per drafting-and-verification iteration follows the method's
description (arXiv abstract page; OpenReview discussion page, reply on
Figure 2): fuzzy drafting of N (= gamma) tokens, verification by the base
model in one forward, then calibration of the draft model's KV cache in a
single forward pass, which replaces the fuzzy entries so their effect never
outlives one drafting phase.

State of one sequence (``Row``):
  tokens      committed tokens x_0..x_{n-1} (prompt + output so far)
  base cache  exact K/V for positions 0..n-2; x_{n-1} is pending for the base
  draft cache exact K/V for positions 0..draft_len-1; tokens from draft_len on
              are pending calibration (their cached K/V, if any, are fuzzy)

Readings (the pages leave these steps open; see also the design notes):
  * Calibration is merged with the next phase's first draft forward: the
    exact draft forward over the pending tokens [accepted drafts..., bonus]
    rewrites their K/V and its last row gives q_1, from which d_1 is drawn.
    A phase therefore runs gamma draft forwards: one exact multi-token
    calibration forward and gamma-1 fuzzy single-token forwards.
  * The fuzzy positions of a phase are those of d_1..d_{gamma-1}; d_gamma is
    never a draft input within its phase.
  * The base verifies [x_{n-1}, d_1..d_gamma] at positions n-1..n+gamma-1 and
    yields p_1..p_{gamma+1}.
  * After acceptance of a tokens and the bonus/resampled y: tokens grow by
    a+1, the base keeps positions up to n+a-1 (y pending), the draft keeps
    exact positions up to n-1 and [d_1..d_a, y] become its pending tokens.
  * The prompt's base prefill covers x_0..x_{P-2}; the draft's prompt
    prefill is the first calibration.
  * Every phase drafts a full gamma; the output is cut to max_new at the end.
  * Calibration ablation (``calibrate=False``; the pages' ablation says that
    without calibration the fuzzy errors accumulate): after acceptance of a
    drafts the accepted drafts that carried a fuzzy entry (d_1..d_min(a,
    gamma-1)) keep it. Only the positions that have no entry, the bonus y
    and, when every draft was accepted, d_gamma, go through the exact draft
    forward that starts the next phase.
"""
from __future__ import annotations

import numpy as np

from . import model as M
from .rng import phase_draws
from .sampling import accept_resample, argmax_f32, draft_token, softmax_f32


def _dist(z64, temperature: float):
    """float32 logits (greedy) or float32 probabilities softmax(z/T)."""
    z = np.asarray(z64, dtype=np.float32)
    if temperature == 0.0:
        return z
    return softmax_f32(z, temperature)


class Row:
    def __init__(self, shape_d: M.Shape, shape_b: M.Shape, max_len: int, kv_dtype: str = "f64"):
        self.tokens: list[int] = []
        self.base = M.KVCache(shape_b, max_len, kv_dtype)
        self.draft = M.KVCache(shape_d, max_len, kv_dtype)
        self.draft_len = 0
        self.phase = 0
        # per-phase records (for parity checks against the CUDA path)
        self.q = None      # [gamma, V] float32 draft distributions (or logits)
        self.p = None      # [gamma+1, V] float32 base distributions (or logits)
        self.d = None      # [gamma] draft tokens
        self.zq = None     # [gamma, V] float64 draft logits
        self.zp = None     # [gamma+1, V] float64 base logits
        self.n_acc = None


class SpecDecoder:
    """EasySpec loop for a batch of independent rows (row index = RNG row)."""

    def __init__(self, Wd, shape_d: M.Shape, Wb, shape_b: M.Shape,
                 groups=None, k: int = 1, mode: int = M.FULL_LAYER,
                 max_len: int = 256, calibrate: bool = True, block: bool = False,
                 kv_dtype: str = "f64"):
        if shape_d.vocab != shape_b.vocab:
            raise ValueError("draft and base must share one vocabulary")
        self.Wd, self.sd, self.Wb, self.sb = Wd, shape_d, Wb, shape_b
        self.groups = groups if groups is not None else M.default_groups(shape_d.n_layers, k)
        M.check_groups(self.groups, shape_d.n_layers)
        self.mode = mode
        self.max_len = max_len
        self.calibrate = calibrate
        # exact multi-token forwards (prompt prefill, calibration, verify) run
        # as one block forward instead of token by token: the same model,
        # fast enough for prompts of thousands of tokens
        self.block = block
        # storage precision of both models' K/V caches ("f64" or "bf16")
        self.kv_dtype = kv_dtype
        self.rows: list[Row] = []

    # -------------------------------------------------------------- stages
    def prefill(self, prompts):
        self.rows = []
        for prompt in prompts:
            r = Row(self.sd, self.sb, self.max_len, self.kv_dtype)
            r.tokens = [int(t) for t in prompt]
            if self.block:
                M.forward_block(self.Wb, self.sb, r.tokens[:-1], 0, r.base, logit_rows=[])
            else:
                for pos in range(len(r.tokens) - 1):
                    M.forward_exact(self.Wb, self.sb, r.tokens[pos], pos, r.base)
            self.rows.append(r)

    def calibrate_row(self, r: Row):
        """Exact draft forward over pending tokens; returns last row's logits."""
        z = None
        if self.block and len(r.tokens) - r.draft_len > 1:
            z = M.forward_block(self.Wd, self.sd, r.tokens[r.draft_len:], r.draft_len, r.draft,
                                logit_rows=[len(r.tokens) - r.draft_len - 1])[0]
        else:
            for pos in range(r.draft_len, len(r.tokens)):
                z = M.forward_exact(self.Wd, self.sd, r.tokens[pos], pos, r.draft)
        r.draft_len = len(r.tokens)
        return z

    def draft_row(self, b: int, gamma: int, temperature: float, seed: int, force_d=None):
        """Calibration + gamma-1 fuzzy forwards.  ``force_d`` (checking aid)
        replaces the drawn tokens by given ones; the oracle's own draws are
        kept in ``row.d_own``."""
        r = self.rows[b]
        greedy = temperature == 0.0
        draws = None if greedy else phase_draws(seed, b, r.phase, gamma)
        n = len(r.tokens)
        z = self.calibrate_row(r)
        zq, q, d, own = [], [], [], []
        for i in range(gamma):
            if i > 0:
                z = M.forward_fuzzy(self.Wd, self.sd, d[-1], n + i - 1, r.draft,
                                    self.groups, self.mode)
            zq.append(z)
            q.append(_dist(z, temperature))
            own.append(draft_token(q[-1], None if greedy else draws[i], greedy))
            d.append(own[-1] if force_d is None else int(force_d[i]))
        r.zq, r.q, r.d, r.d_own = np.array(zq), np.array(q), d, own
        return d

    def verify_row(self, b: int, gamma: int, temperature: float, seed: int, force=None):
        """Verification + accept/resample + commit.  ``force`` = (a, tokens)
        (checking aid) commits given decisions; the oracle's own are kept in
        ``row.own``."""
        r = self.rows[b]
        greedy = temperature == 0.0
        draws = None if greedy else phase_draws(seed, b, r.phase, gamma)
        n = len(r.tokens)
        zp, p = [], []
        run = [r.tokens[-1]] + list(r.d)
        if self.block:
            zp = list(M.forward_block(self.Wb, self.sb, run, n - 1, r.base))
        else:
            zp = [M.forward_exact(self.Wb, self.sb, tok, n - 1 + j, r.base) for j, tok in enumerate(run)]
        p = [_dist(z, temperature) for z in zp]
        r.zp, r.p = np.array(zp), np.array(p)
        a, new = accept_resample(r.p, r.q, r.d,
                                 None if greedy else draws[gamma:2 * gamma],
                                 None if greedy else draws[2 * gamma], greedy)
        r.own = (a, new)
        if force is not None:
            a, new = int(force[0]), [int(t) for t in force[1]]
        r.n_acc = a
        r.tokens += new
        # calibration recomputes every committed position from n on; without
        # it the fuzzy entries of the accepted d_1..d_min(a, gamma-1) stay
        r.draft_len = n if self.calibrate else n + min(a, gamma - 1)
        r.phase += 1
        return a, new

    # -------------------------------------------------------------- driver
    def generate(self, prompts, max_new: int, gamma: int, temperature: float,
                 seed: int = 0):
        """Speculative generation; returns [B][max_new] new tokens."""
        self.prefill(prompts)
        P = [len(p) for p in prompts]
        for b, r in enumerate(self.rows):
            while len(r.tokens) - P[b] < max_new:
                if len(r.tokens) + gamma + 1 > self.max_len:
                    raise ValueError("sequence would exceed max_len")
                self.draft_row(b, gamma, temperature, seed)
                self.verify_row(b, gamma, temperature, seed)
        return [r.tokens[P[b]:P[b] + max_new] for b, r in enumerate(self.rows)]


def seq_decode(Wb, shape_b: M.Shape, prompt, max_new: int, max_len: int = 256):
    """Plain greedy decoding with the base model (the losslessness reference)."""
    cache = M.KVCache(shape_b, max_len)
    toks = [int(t) for t in prompt]
    z = None
    for pos, t in enumerate(toks):
        z = M.forward_exact(Wb, shape_b, t, pos, cache)
    out = []
    for _ in range(max_new):
        y = argmax_f32(np.asarray(z, dtype=np.float32))
        out.append(y)
        z = M.forward_exact(Wb, shape_b, y, len(toks), cache)
        toks.append(y)
    return out


def exact_next_dist(Wb, shape_b: M.Shape, history, temperature: float, max_len: int = 256):
    """float64 base distribution of the token following ``history`` (fresh cache)."""
    cache = M.KVCache(shape_b, max_len)
    z = None
    for pos, t in enumerate(history):
        z = M.forward_exact(Wb, shape_b, int(t), pos, cache)
    z = np.asarray(z, dtype=np.float64) / temperature
    e = np.exp(z - z.max())
    return e / e.sum()
