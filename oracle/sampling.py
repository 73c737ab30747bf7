"""Token decisions of speculative decoding (oracle side).

TEST INFRASTRUCTURE ONLY -- see the package docstring.

The EasySpec pages call the method lossless: the output follows the base
model's distribution ("preserving the original distributions of the base
LLMs", arXiv abstract page; "accuracy" means the acceptance rate, OpenReview
discussion page, first reply).  They do not restate the rule that makes it
so; it is the one defined by the two works they cite, "Fast Inference from
Transformers via Speculative Decoding" (Leviathan et al., Algorithm 1) and
"Accelerating Large Language Model Decoding with Speculative Sampling"
(Chen et al., Algorithm 2):

  draft token x ~ q is accepted with probability min(1, p(x)/q(x));
  at the first rejection the output is drawn from norm(max(0, p - q));
  if every draft token is accepted one more token is drawn from the base
  model's next distribution.

Readings where the pages and the cited works leave a step open (each is also
listed in the design notes):
  * accept iff float32(u * q(x)) < p(x), u = uniform24(draw): the test
    "u < p/q" multiplied through by q > 0, strict, in float32.
  * categorical draws use an integer-quantised inverse CDF: weights
    W_i = floor(w_i * 2**40) (w_i float32, unnormalised allowed),
    T = sum W_i, t = floor(u64 * T / 2**64), result = smallest i whose
    prefix sum exceeds t.  Integer sums are exact, so the index does not
    depend on summation order.  If every W_i is 0 (a residual that rounded
    to nothing) the draw falls back to the base distribution p.
  * greedy decoding (temperature 0) compares argmaxes of float32 logits,
    lowest index on ties, and consumes no draws.

Parity: pinned by tests/test_oracle_sampling.py -- the acceptance probability
equals sum_x min(p(x), q(x)) (Leviathan et al., the closed form for the
expected acceptance), the emitted token follows p (chi-square), and the
quantised sampler matches the exact inverse CDF on hand-made weights.
"""
from __future__ import annotations

import numpy as np

from .rng import uniform24

Q_SHIFT = 40


def argmax_f32(z) -> int:
    """Index of the largest float32 value, lowest index on ties."""
    z = np.asarray(z, dtype=np.float32)
    return int(np.argmax(z))  # numpy returns the first occurrence


def quantise(w) -> np.ndarray:
    """W_i = floor(w_i * 2**40) for float32 weights w_i >= 0, as uint64."""
    w = np.asarray(w, dtype=np.float32).astype(np.float64)
    if np.any(w < 0):
        raise ValueError("sampling weights must be non-negative")
    return np.floor(w * float(1 << Q_SHIFT)).astype(np.uint64)


def sample_quantised(w, u64: int) -> int:
    """Integer inverse-CDF draw from unnormalised float32 weights ``w``.

    Returns -1 when every quantised weight is zero.
    """
    W = quantise(w)
    prefix = np.cumsum(W, dtype=np.uint64)
    total = int(prefix[-1])
    if total == 0:
        return -1
    t = (int(u64) * total) >> 64
    return int(np.searchsorted(prefix, np.uint64(t), side="right"))


def softmax_f32(z, temperature: float) -> np.ndarray:
    """Float32 probabilities softmax(z / T) of float32 logits (computed in f64)."""
    z = np.asarray(z, dtype=np.float32).astype(np.float64) / float(temperature)
    z = z - z.max()
    e = np.exp(z)
    return (e / e.sum()).astype(np.float32)


def draft_token(q_or_logits, u64: int | None, greedy: bool) -> int:
    """d_i ~ q_i (sampled) or argmax of the draft logits (greedy)."""
    if greedy:
        return argmax_f32(q_or_logits)
    i = sample_quantised(q_or_logits, u64)
    if i < 0:
        raise ValueError("draft distribution quantised to zero mass")
    return i


def accept_resample(p, q, d, accept_draws, bonus_draw, greedy: bool):
    """Accept/resample over one row.

    p : [gamma+1, V] float32 base probabilities (greedy: base logits)
    q : [gamma, V]   float32 draft probabilities (greedy: draft logits)
    d : [gamma]      draft tokens
    accept_draws : gamma 64-bit draws for the accept tests
    bonus_draw   : one 64-bit draw for the residual / bonus sample
    Returns (n_accepted, tokens) with len(tokens) == n_accepted + 1.
    """
    p = np.asarray(p, dtype=np.float32)
    q = np.asarray(q, dtype=np.float32)
    gamma = len(d)
    out = []
    for i in range(gamma):
        x = int(d[i])
        if greedy:
            ok = argmax_f32(p[i]) == x
        else:
            u = uniform24(accept_draws[i])
            ok = np.float32(u * q[i, x]) < p[i, x]
        if ok:
            out.append(x)
            continue
        if greedy:
            y = argmax_f32(p[i])
        else:
            resid = np.maximum(np.float32(0), p[i] - q[i])  # float32 subtraction
            y = sample_quantised(resid, bonus_draw)
            if y < 0:
                y = sample_quantised(p[i], bonus_draw)
        out.append(y)
        return i, out
    if greedy:
        y = argmax_f32(p[gamma])
    else:
        y = sample_quantised(p[gamma], bonus_draw)
    out.append(y)
    return gamma, out
