"""The binding refuses arguments that would make a kernel read past a device
buffer, or the library write past a host array, before it calls into the
library: accept/resample and the quantised sampler take dense device arrays
of the sizes the first argument's shape implies, and es_read_kv's host
buffers hold the model's own kv heads and head size."""
import pytest
import torch

from layer_drafting_draft_b300 import easyspec as E


def _accept_args(device="cpu", B=2, g=2, V=8):
    p = torch.zeros(B, g + 1, V, device=device)
    q = torch.zeros(B, g, V, device=device)
    d = torch.zeros(B, g, dtype=torch.int32, device=device)
    u = torch.zeros(B, g + 1, dtype=torch.int64, device=device)
    return p, q, d, u


def test_host_tensors_are_refused():
    for fn in (E.es_accept_resample, E.es_accept_resample_noalloc):
        with pytest.raises(ValueError, match="CUDA"):
            fn(*_accept_args(), False)
    with pytest.raises(ValueError, match="CUDA"):
        E.es_sample(torch.zeros(2, 8), torch.zeros(2, dtype=torch.int64))


def test_ranks_and_missing_draws_are_refused():
    p, q, d, _ = _accept_args()
    with pytest.raises(ValueError, match="p must be"):
        E.es_accept_resample(p[0], q, d, None, True)
    with pytest.raises(ValueError, match="draws"):
        E.es_accept_resample(p, q, d, None, False)
    with pytest.raises(ValueError, match="w must be"):
        E.es_sample(torch.zeros(8), torch.zeros(8, dtype=torch.int64))


def test_read_kv_buffers_must_match_the_model():
    g = object.__new__(E.EasySpec)   # no context: the check comes first
    g._shapes = ({"n_kv_heads": 2, "head_dim": 64}, {"n_kv_heads": 4, "head_dim": 128})
    with pytest.raises(ValueError, match="draft model has 2 kv heads of 64"):
        g.es_read_kv(0, 0, 0, 4, 4, 64)
    with pytest.raises(ValueError, match="base model has 4 kv heads of 128"):
        g.es_read_kv(1, 0, 0, 4, 4, 64)


@pytest.mark.gpu
def test_device_dtypes_shapes_and_layouts_are_checked():
    p, q, d, u = _accept_args("cuda")
    bad = [
        (p, q[:, :1], d, u),                                          # q one draft short
        (p, q, d.long(), u),                                          # int64 drafts
        (p, q, d, u[:, :2]),                                          # draws one short
        (p, q.transpose(0, 1).contiguous().transpose(0, 1), d, u),    # q not contiguous
        (p.double(), q, d, u),                                        # float64 p
    ]
    for args in bad:
        for fn in (E.es_accept_resample, E.es_accept_resample_noalloc):
            with pytest.raises(ValueError):
                fn(*args, False)
    w = torch.ones(2, 8, device="cuda")
    for ww, uu in ((w, torch.zeros(3, dtype=torch.int64, device="cuda")),
                   (w.double(), torch.zeros(2, dtype=torch.int64, device="cuda")),
                   (w, torch.zeros(2, dtype=torch.int32, device="cuda")),
                   (w.t().contiguous().t(), torch.zeros(2, dtype=torch.int64, device="cuda"))):
        with pytest.raises(ValueError):
            E.es_sample(ww, uu)
    idx = E.es_sample(w, torch.zeros(2, dtype=torch.int64, device="cuda")).cpu()
    assert idx.shape == (2,) and all(0 <= int(i) < 8 for i in idx)
