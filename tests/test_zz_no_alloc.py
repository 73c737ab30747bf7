"""The accept/resample entry point that allocates no device memory.

es_accept_resample_noalloc serves callers that cannot allocate device memory
where they call it: a serving host whose device memory is reserved up front
for its own pool allocator, or a decode loop that cannot take cudaFree's
device-wide synchronisation between tokens.  It uses a fixed scratch array
inside the library instead of allocating, so two things are checked here:
its decisions equal those of es_accept_resample on the same inputs, and a
second call right after the first (the array still holding the first call's
contents) is as correct as the first.  Sizes beyond the array are refused.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

from layer_drafting_draft_b300.easyspec import (ES_ERR_ARG, EasySpecError, es_accept_resample,
                                                es_accept_resample_noalloc)

pytestmark = pytest.mark.gpu


def _case(seed, B, gamma, V, greedy):
    r = np.random.default_rng(seed)
    z = r.normal(size=(B, gamma + 1, V)).astype(np.float32) * 2
    zq = z[:, :gamma] + r.normal(size=(B, gamma, V)).astype(np.float32) * 0.5
    if greedy:
        p, q = z, zq
        d = np.argmax(zq, axis=-1).astype(np.int32)
        d[::2, 0] = np.argmax(z[::2, 0], axis=-1)  # some accepted drafts
        u = None
    else:
        e = np.exp(z - z.max(-1, keepdims=True))
        p = (e / e.sum(-1, keepdims=True)).astype(np.float32)
        eq = np.exp(zq - zq.max(-1, keepdims=True))
        q = (eq / eq.sum(-1, keepdims=True)).astype(np.float32)
        # drafts drawn from q by inverse CDF in float64
        cdf = np.cumsum(q.astype(np.float64), axis=-1)
        t = r.random(size=(B, gamma)) * cdf[..., -1]
        d = np.stack([[min(int(np.searchsorted(cdf[b, i], t[b, i], side="right")), V - 1)
                       for i in range(gamma)] for b in range(B)]).astype(np.int32)
        u = r.integers(0, 2 ** 63, size=(B, gamma + 1), dtype=np.int64)
    dev = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return dev(p), dev(q), dev(d), dev(u)


@pytest.mark.parametrize("greedy", [False, True])
@pytest.mark.parametrize("B,gamma,V", [(4, 4, 1000), (16, 6, 151936), (1, 16, 4099)])
def test_noalloc_matches_allocating_entry_point_twice(B, gamma, V, greedy):
    for call in range(2):  # the second call finds the first call's scratch contents
        p, q, d, u = _case(1000 * call + B + V, B, gamma, V, greedy)
        n_ref, t_ref = es_accept_resample(p, q, d, u, greedy)
        n_got, t_got = es_accept_resample_noalloc(p, q, d, u, greedy)
        assert torch.equal(n_got.cpu(), n_ref.cpu()), (call, n_got, n_ref)
        assert torch.equal(t_got.cpu(), t_ref.cpu()), (call, t_got, t_ref)


def test_noalloc_refuses_sizes_beyond_its_scratch():
    p, q, d, u = _case(7, 17, 2, 64, False)
    with pytest.raises(EasySpecError) as e:
        es_accept_resample_noalloc(p, q, d, u, False)
    assert e.value.status == ES_ERR_ARG
