"""Error behaviour of the C ABI on the CPU (no GPU needed).

Every entry point returns a status and no exception crosses the boundary. A
null context gives ES_ERR_ARG. easyspec_init checks its configuration before
any CUDA call, so each invalid field gives ES_ERR_ARG with *out left NULL. On
a machine without a usable GPU a valid configuration fails with ES_ERR_CUDA,
again with *out NULL, and the failed context is torn down without a crash.
"""
import ctypes as C

import pytest
import torch

from layer_drafting_draft_b300 import easyspec as E


def _shape(L, d, H, Hkv, hd, F, V):
    return E.es_model_shape(L, d, H, Hkv, hd, F, V, 1e4, 1e-6, 1)


def _cfg(**kw):
    cfg = E.es_config()
    cfg.draft = _shape(4, 128, 4, 2, 32, 344, 512)
    cfg.base = _shape(8, 256, 8, 4, 32, 688, 512)
    cfg.max_batch, cfg.max_seq, cfg.max_gamma, cfg.parallel_mode = 1, 64, 4, E.ES_FULL_LAYER
    for k, v in kw.items():
        setattr(cfg, k, v)
    return cfg


def _init(cfg):
    L = E.lib()
    w = E.es_weights()
    out = C.c_void_p(1)
    st = L.easyspec_init(C.byref(cfg), C.byref(w), C.byref(w), C.byref(out))
    return st, out.value


def test_null_context_calls():
    L = E.lib()
    i32 = C.POINTER(C.c_int32)()
    assert L.easyspec_prefill(None, i32, 1, 1) == E.ES_ERR_ARG
    assert L.calibrate_kv(None, 4, 0.0, 0) == E.ES_ERR_ARG
    assert L.es_set_calibration(None, 0) == E.ES_ERR_ARG
    assert L.draft_step(None, 2, 4, 0.0, 0, i32) == E.ES_ERR_ARG
    assert L.verify_step(None, 0.0, 0, i32, i32) == E.ES_ERR_ARG
    assert L.es_decode(None, 8, 4, 2, 0.0, 0, None) == E.ES_ERR_ARG
    assert L.es_profile(None, 1) == E.ES_ERR_ARG
    n = C.c_int(0)
    assert L.es_read_tokens(None, 0, i32, 0, C.byref(n)) == E.ES_ERR_ARG
    assert L.easyspec_last_error(None) == b"null context"
    L.easyspec_destroy(None)


def test_init_without_out_or_config():
    L = E.lib()
    w = E.es_weights()
    assert L.easyspec_init(C.byref(_cfg()), C.byref(w), C.byref(w), None) == E.ES_ERR_ARG
    out = C.c_void_p(1)
    assert L.easyspec_init(None, C.byref(w), C.byref(w), C.byref(out)) == E.ES_ERR_ARG
    assert out.value is None


def _starts(vals):
    arr = (C.c_int * len(vals))(*vals)
    return C.cast(arr, C.POINTER(C.c_int)), arr


@pytest.mark.parametrize("field", ["vocab", "batch", "gamma", "seq", "mode", "first_set", "order", "big_set"])
def test_invalid_config_rejected_before_any_cuda_call(field):
    keep = None
    if field == "vocab":
        cfg = _cfg(base=_shape(8, 256, 8, 4, 32, 688, 513))
    elif field == "batch":
        cfg = _cfg(max_batch=0)
    elif field == "gamma":
        cfg = _cfg(max_gamma=17)
    elif field == "seq":
        cfg = _cfg(max_seq=4)
    elif field == "mode":
        cfg = _cfg(parallel_mode=7)
    else:
        vals = {"first_set": [1, 2], "order": [0, 2, 2], "big_set": [0]}[field]
        ptr, keep = _starts(vals)
        cfg = _cfg(draft=_shape(12 if field == "big_set" else 4, 128, 4, 2, 32, 344, 512),
                   group_starts=ptr, n_groups=len(vals))
    st, out = _init(cfg)
    assert st == E.ES_ERR_ARG and out is None
    del keep


@pytest.mark.skipif(torch.cuda.is_available(), reason="needs a machine without a usable GPU")
def test_init_without_gpu_fails_cleanly():
    st, out = _init(_cfg())
    assert st == E.ES_ERR_CUDA and out is None
