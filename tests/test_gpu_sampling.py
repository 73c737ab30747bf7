"""GPU sampler and accept/resample: bit-exact against the oracle given the
same probabilities and draws (the rule of the works the EasySpec pages cite:
Leviathan et al.; Chen et al.)."""
import numpy as np
import pytest
import torch

from oracle.sampling import accept_resample, sample_quantised, softmax_f32

pytestmark = pytest.mark.gpu


def _u64(r, shape):
    return r.integers(0, 2 ** 63, size=shape, dtype=np.int64).astype(np.uint64) * np.uint64(2) + \
        r.integers(0, 2, size=shape, dtype=np.int64).astype(np.uint64)


@pytest.mark.parametrize("V", [1, 7, 1000, 1031, 151936])
def test_quantised_sampler_bit_exact(V):
    from layer_drafting_draft_b300.easyspec import es_sample
    r = np.random.default_rng(V)
    B = 64
    w = r.random((B, V)).astype(np.float32) ** 4  # skewed weights
    w[0] = 0.0            # all-zero row -> -1
    if V > 3:
        w[1, :-1] = 0.0   # single non-zero at the ragged tail
    u = _u64(r, B)
    got = es_sample(torch.from_numpy(w).cuda(), torch.from_numpy(u.view(np.int64)).cuda()).cpu().numpy()
    want = [sample_quantised(w[b], int(u[b])) for b in range(B)]
    assert list(got) == want


@pytest.mark.parametrize("gamma,V,greedy", [(1, 16, False), (4, 1000, False), (8, 4099, False),
                                           (4, 151936, False), (4, 1000, True), (6, 257, True)])
def test_accept_resample_bit_exact(gamma, V, greedy):
    from layer_drafting_draft_b300.easyspec import es_accept_resample
    r = np.random.default_rng(gamma * 1000 + V)
    B = 48
    # near-identical p and q so that acceptances, rejections and full
    # acceptance (bonus) all occur
    z = r.normal(size=(B, gamma + 1, V)).astype(np.float32) * 2
    zq = z[:, :gamma] + r.normal(size=(B, gamma, V)).astype(np.float32) * 0.5
    if greedy:
        p, q = z, zq
        d = np.argmax(zq, axis=-1).astype(np.int32)
        d[::3, 0] = np.argmax(z[::3, 0], axis=-1)   # force some accepts
        z[5, 1, :4] = 9.0                           # ties: lowest index wins
        p = z
        u = None
    else:
        p = np.stack([[softmax_f32(z[b, i], 1.0) for i in range(gamma + 1)] for b in range(B)])
        q = np.stack([[softmax_f32(zq[b, i], 1.0) for i in range(gamma)] for b in range(B)])
        ud = _u64(r, (B, gamma))
        d = np.array([[sample_quantised(q[b, i], int(ud[b, i])) for i in range(gamma)] for b in range(B)], np.int32)
        u = _u64(r, (B, gamma + 1))
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    n, tok = es_accept_resample(dev(p), dev(q), dev(d), None if u is None else dev(u.view(np.int64)), greedy)
    n, tok = n.cpu().numpy(), tok.cpu().numpy()
    seen = set()
    for b in range(B):
        a, out = accept_resample(p[b], q[b], d[b], None if greedy else [int(x) for x in u[b, :gamma]],
                                 None if greedy else int(u[b, gamma]), greedy)
        assert n[b] == a, (b, n[b], a)
        assert list(tok[b, : a + 1]) == out
        assert all(t == -1 for t in tok[b, a + 1:])
        seen.add(a == gamma)
        seen.add(a == 0)
    assert True in seen
