"""ctypes binding of libeasyspec.so (argument marshalling only).

Every step of the decoding path runs inside the CUDA library; this module only
converts Python/PyTorch arguments to the C ABI declared in
include/easyspec.h.  PyTorch is used for device memory and streams.  If the
library is missing the import of the binding fails loudly -- there is no CPU
or Python fallback.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libeasyspec.so")

ES_OK, ES_ERR_ARG, ES_ERR_OOM, ES_ERR_CUDA, ES_ERR_TIMEOUT, ES_ERR_STATE, ES_ERR_CAPACITY = 0, -1, -2, -3, -4, -5, -6
ES_DTYPE_F32, ES_DTYPE_BF16 = 0, 1
ES_ATTN_ONLY, ES_FULL_LAYER = 0, 1

STATUS_NAMES = {0: "ES_OK", -1: "ES_ERR_ARG", -2: "ES_ERR_OOM", -3: "ES_ERR_CUDA",
                -4: "ES_ERR_TIMEOUT", -5: "ES_ERR_STATE", -6: "ES_ERR_CAPACITY"}

EXPORTED = ["easyspec_init", "easyspec_prefill", "calibrate_kv", "es_set_calibration", "draft_step", "verify_step",
            "generate", "es_decode", "es_profile", "es_profile_read", "es_accept_resample",
            "es_accept_resample_noalloc",
            "es_sample", "es_wait_selftest", "es_read_kv", "es_read_dist", "es_read_tokens", "es_layer_sets", "easyspec_last_error",
            "easyspec_destroy"]


class es_model_shape(C.Structure):
    _fields_ = [("n_layers", C.c_int), ("d", C.c_int), ("n_heads", C.c_int),
                ("n_kv_heads", C.c_int), ("head_dim", C.c_int), ("ffn", C.c_int),
                ("vocab", C.c_int), ("rope_theta", C.c_float), ("eps", C.c_float),
                ("dtype", C.c_int)]


_PP = C.POINTER(C.c_void_p)


class es_weights(C.Structure):
    _fields_ = [("embed", C.c_void_p), ("lm_head", C.c_void_p), ("final_norm", C.c_void_p),
                ("attn_norm", _PP), ("wq", _PP), ("wk", _PP), ("wv", _PP), ("wo", _PP),
                ("mlp_norm", _PP), ("wgate", _PP), ("wup", _PP), ("wdown", _PP)]


class es_config(C.Structure):
    _fields_ = [("draft", es_model_shape), ("base", es_model_shape), ("max_batch", C.c_int),
                ("max_seq", C.c_int), ("max_gamma", C.c_int), ("parallel_mode", C.c_int),
                ("group_starts", C.POINTER(C.c_int)), ("n_groups", C.c_int),
                ("cuda_stream", C.c_void_p)]


class es_stats(C.Structure):
    _fields_ = [("phases", C.c_int64), ("drafted", C.c_int64), ("accepted", C.c_int64),
                ("emitted", C.c_int64), ("kernel_launches", C.c_int64), ("prefill_ms", C.c_double),
                ("decode_ms", C.c_double)]


_lib = None


def lib() -> C.CDLL:
    """Open libeasyspec.so (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m layer_drafting_draft_b300.build`")
        L = C.CDLL(LIB_PATH)
        i32p, f32p, u64p, vp = C.POINTER(C.c_int32), C.POINTER(C.c_float), C.POINTER(C.c_uint64), C.c_void_p
        ctxp = C.c_void_p
        sig = {
            "easyspec_init": ([C.POINTER(es_config), C.POINTER(es_weights), C.POINTER(es_weights), C.POINTER(C.c_void_p)], C.c_int),
            "easyspec_prefill": ([ctxp, i32p, C.c_int, C.c_int], C.c_int),
            "calibrate_kv": ([ctxp, C.c_int, C.c_float, C.c_uint64], C.c_int),
            "es_set_calibration": ([ctxp, C.c_int], C.c_int),
            "draft_step": ([ctxp, C.c_int, C.c_int, C.c_float, C.c_uint64, i32p], C.c_int),
            "verify_step": ([ctxp, C.c_float, C.c_uint64, i32p, i32p], C.c_int),
            "generate": ([ctxp, i32p, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, C.c_float, C.c_uint64, i32p, C.POINTER(es_stats)], C.c_int),
            "es_decode": ([ctxp, C.c_int, C.c_int, C.c_int, C.c_float, C.c_uint64, C.POINTER(es_stats)], C.c_int),
            "es_profile": ([ctxp, C.c_int], C.c_int),
            "es_profile_read": ([ctxp, C.c_int, C.c_char_p, C.c_int, C.POINTER(C.c_double), C.POINTER(C.c_int64), C.POINTER(C.c_double)], C.c_int),
            "es_accept_resample": ([vp, vp, vp, vp, C.c_int, C.c_int, C.c_int, C.c_int, vp, vp, vp], C.c_int),
            "es_accept_resample_noalloc": ([vp, vp, vp, vp, C.c_int, C.c_int, C.c_int, C.c_int, vp, vp, vp], C.c_int),
            "es_sample": ([vp, vp, C.c_int, C.c_int, vp, vp], C.c_int),
            "es_wait_selftest": ([C.c_int64, C.c_int64, vp], C.c_int),
            "es_read_kv": ([ctxp, C.c_int, C.c_int, C.c_int, C.c_int, f32p, f32p], C.c_int),
            "es_read_dist": ([ctxp, C.c_int, f32p], C.c_int),
            "es_read_tokens": ([ctxp, C.c_int, i32p, C.c_int, C.POINTER(C.c_int)], C.c_int),
            "es_layer_sets": ([C.c_int, C.c_int, i32p, C.c_int, C.POINTER(C.c_int)], C.c_int),
            "easyspec_last_error": ([ctxp], C.c_char_p),
            "easyspec_destroy": ([ctxp], None),
        }
        for name, (args, res) in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def layer_sets(n_layers: int, k: int) -> list[int]:
    """The library's default draft layer sets for set size k, as the first
    layer of each set (host only, no GPU)."""
    import numpy as np
    L = lib()
    n = C.c_int(0)
    out = np.zeros(max(n_layers, 1), dtype=np.int32)
    st = L.es_layer_sets(n_layers, k, out.ctypes.data_as(C.POINTER(C.c_int32)), len(out), C.byref(n))
    if st != ES_OK:
        raise EasySpecError(st, "es_layer_sets: invalid arguments")
    return out[: n.value].tolist()


class EasySpecError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


def _ptr(t: torch.Tensor) -> int:
    return t.data_ptr()


def _i32(a):
    return a.ctypes.data_as(C.POINTER(C.c_int32))


def _shape(s: dict, dtype: str) -> es_model_shape:
    return es_model_shape(s["n_layers"], s["d"], s["n_heads"], s["n_kv_heads"], s["head_dim"],
                          s["ffn"], s["vocab"], s["rope_theta"], s["eps"],
                          ES_DTYPE_BF16 if dtype == "bf16" else ES_DTYPE_F32)


class _WeightTable:
    """Keeps the per-layer pointer arrays alive for the context's lifetime."""

    def __init__(self, w: dict):
        L = len(w["layers"])
        self.arrays = {}
        for key in ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "wgate", "wup", "wdown"):
            arr = (C.c_void_p * L)(*[_ptr(lw[key]) for lw in w["layers"]])
            self.arrays[key] = arr
        self.struct = es_weights(_ptr(w["embed"]), _ptr(w["lm_head"]), _ptr(w["final_norm"]),
                                 *[C.cast(self.arrays[k], _PP) for k in
                                   ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "wgate", "wup", "wdown")])


class EasySpec:
    """A decoding context over a draft/base pair of device weight dicts."""

    def __init__(self, draft_w: dict, draft_shape: dict, base_w: dict, base_shape: dict,
                 dtype: str = "bf16", max_batch: int = 1, max_seq: int = 512, max_gamma: int = 8,
                 mode: int = ES_FULL_LAYER, group_starts=None, stream: torch.cuda.Stream | None = None):
        import numpy as np
        self._lib = lib()
        self._keep = [draft_w, base_w]
        self._wd, self._wb = _WeightTable(draft_w), _WeightTable(base_w)
        self.stream = stream if stream is not None else torch.cuda.current_stream()
        self.V = draft_shape["vocab"]
        self._shapes = (dict(draft_shape), dict(base_shape))
        self._gs = None
        cfg = es_config(_shape(draft_shape, dtype), _shape(base_shape, dtype), max_batch, max_seq,
                        max_gamma, mode, None, 0, C.c_void_p(self.stream.cuda_stream))
        if group_starts is not None:
            self._gs = np.ascontiguousarray(group_starts, dtype=np.int32)
            cfg.group_starts = _i32(self._gs)
            cfg.n_groups = len(self._gs)
        self._cfg = cfg
        h = C.c_void_p()
        st = self._lib.easyspec_init(C.byref(cfg), C.byref(self._wd.struct), C.byref(self._wb.struct), C.byref(h))
        if st != ES_OK:
            raise EasySpecError(st, "easyspec_init failed (see stderr)")
        self.ctx = h
        self.max_gamma = max_gamma

    # ------------------------------------------------------------ helpers
    def _check(self, st: int):
        if st != ES_OK:
            msg = self._lib.easyspec_last_error(self.ctx)
            raise EasySpecError(st, msg.decode() if msg else "")

    def close(self):
        if getattr(self, "ctx", None):
            self._lib.easyspec_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ------------------------------------------------------------ ABI calls
    def easyspec_prefill(self, prompts):
        import numpy as np
        p = np.ascontiguousarray(np.asarray(prompts, dtype=np.int32))
        self._check(self._lib.easyspec_prefill(self.ctx, _i32(p), p.shape[0], p.shape[1]))
        self.B = p.shape[0]

    def calibrate_kv(self, gamma: int, temperature: float, seed: int):
        self._check(self._lib.calibrate_kv(self.ctx, gamma, temperature, seed))

    def es_set_calibration(self, on: bool):
        """on=False: the calibration ablation (accepted drafts keep their
        layer-parallel KV entries)."""
        self._check(self._lib.es_set_calibration(self.ctx, 1 if on else 0))

    def draft_step(self, k: int, gamma: int, temperature: float, seed: int):
        import numpy as np
        out = np.zeros((self.B, gamma), np.int32)
        self._check(self._lib.draft_step(self.ctx, k, gamma, temperature, seed, _i32(out)))
        return out

    def verify_step(self, temperature: float, seed: int, gamma: int):
        import numpy as np
        n = np.zeros(self.B, np.int32)
        t = np.zeros((self.B, gamma + 1), np.int32)
        self._check(self._lib.verify_step(self.ctx, temperature, seed, _i32(n), _i32(t)))
        return n, t

    def generate(self, prompts, max_new: int, gamma: int, k: int, temperature: float, seed: int):
        import numpy as np
        p = np.ascontiguousarray(np.asarray(prompts, dtype=np.int32))
        out = np.zeros((p.shape[0], max_new), np.int32)
        st = es_stats()
        self._check(self._lib.generate(self.ctx, _i32(p), p.shape[0], p.shape[1], max_new, gamma, k,
                                       temperature, seed, _i32(out), C.byref(st)))
        self.B = p.shape[0]
        return out, {f: getattr(st, f) for f, _ in es_stats._fields_}

    def es_decode(self, max_new: int, gamma: int, k: int, temperature: float, seed: int):
        st = es_stats()
        self._check(self._lib.es_decode(self.ctx, max_new, gamma, k, temperature, seed, C.byref(st)))
        return {f: getattr(st, f) for f, _ in es_stats._fields_}

    def es_profile(self, on):
        """on: False/0 off, True/1 per kernel, 2 per phase part (graphs kept)."""
        self._check(self._lib.es_profile(self.ctx, int(on)))

    def es_profile_read(self):
        """{kernel name: (ms, launches, algorithmic bytes)} since es_profile()."""
        out, i = {}, 0
        buf = C.create_string_buffer(128)
        ms, n, by = C.c_double(), C.c_int64(), C.c_double()
        while self._lib.es_profile_read(self.ctx, i, buf, 128, C.byref(ms), C.byref(n), C.byref(by)) == ES_OK:
            out[buf.value.decode()] = (ms.value, n.value, by.value)
            i += 1
        return out

    def es_read_kv(self, which: int, layer: int, seq: int, n: int, kv_heads: int, head_dim: int):
        import numpy as np
        # the library writes n x (the model's kv heads) x (its head size)
        # floats per array: the host buffers must have exactly that size
        s = self._shapes[1 if which else 0]
        if (kv_heads, head_dim) != (s["n_kv_heads"], s["head_dim"]):
            raise ValueError(f"es_read_kv: the {'base' if which else 'draft'} model has "
                             f"{s['n_kv_heads']} kv heads of {s['head_dim']}, not {kv_heads} of {head_dim}")
        k = np.zeros((n, kv_heads, head_dim), np.float32)
        v = np.zeros_like(k)
        self._check(self._lib.es_read_kv(self.ctx, which, layer, seq, n,
                                         k.ctypes.data_as(C.POINTER(C.c_float)),
                                         v.ctypes.data_as(C.POINTER(C.c_float))))
        return k, v

    def es_read_dist(self, which: int, gamma: int):
        import numpy as np
        rows = gamma if which in (0, 2) else gamma + 1
        out = np.zeros((self.B, rows, self.V), np.float32)
        self._check(self._lib.es_read_dist(self.ctx, which, out.ctypes.data_as(C.POINTER(C.c_float))))
        return out

    def es_read_tokens(self, seq: int, cap: int = 1 << 16):
        import numpy as np
        out = np.zeros(cap, np.int32)
        n = C.c_int()
        self._check(self._lib.es_read_tokens(self.ctx, seq, _i32(out), cap, C.byref(n)))
        return out[: n.value]


def _check_accept_args(p, q, d, u, greedy: bool):
    """The kernels read p, q, d and u as dense device arrays of the sizes that
    p's shape implies: refuse anything else here rather than let a kernel
    read past a buffer."""
    if p.dim() != 3:
        raise ValueError("p must be [B, gamma+1, V]")
    B, g1, V = p.shape
    want = [("p", p, torch.float32, (B, g1, V)), ("q", q, torch.float32, (B, g1 - 1, V)),
            ("d", d, torch.int32, (B, g1 - 1))]
    if u is not None or not greedy:
        if u is None:
            raise ValueError("sampled accept/resample needs the draws u")
        want.append(("u", u, torch.int64, (B, g1)))
    for name, t, dt, shp in want:
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if t.dtype != dt or tuple(t.shape) != shp or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous {dt} tensor of shape {shp}, "
                             f"got {t.dtype} {tuple(t.shape)}")
        if t.device != p.device:
            raise ValueError(f"{name} is on {t.device}, p on {p.device}")
    return B, g1, V


def es_accept_resample(p: torch.Tensor, q: torch.Tensor, d: torch.Tensor, u: torch.Tensor | None,
                       greedy: bool):
    """Accept/resample on device tensors: p [B,g+1,V] f32, q [B,g,V] f32,
    d [B,g] int32, u [B,g+1] uint64 (as int64).  Returns (n_acc, tok)."""
    B, g1, V = _check_accept_args(p, q, d, u, greedy)
    n_acc = torch.empty(B, dtype=torch.int32, device=p.device)
    tok = torch.empty(B, g1, dtype=torch.int32, device=p.device)
    st = lib().es_accept_resample(_ptr(p), _ptr(q), _ptr(d), _ptr(u) if u is not None else None,
                                  B, g1 - 1, V, 1 if greedy else 0, _ptr(n_acc), _ptr(tok),
                                  torch.cuda.current_stream().cuda_stream)
    if st != ES_OK:
        raise EasySpecError(st, "es_accept_resample")
    return n_acc, tok


def es_accept_resample_noalloc(p: torch.Tensor, q: torch.Tensor, d: torch.Tensor, u: torch.Tensor | None,
                               greedy: bool):
    """es_accept_resample through the entry point that allocates no device
    memory (fixed scratch inside the library; B <= 16, gamma <= 16).
    Only the outputs are allocated here, by the caller's side."""
    B, g1, V = _check_accept_args(p, q, d, u, greedy)
    n_acc = torch.empty(B, dtype=torch.int32, device=p.device)
    tok = torch.empty(B, g1, dtype=torch.int32, device=p.device)
    st = lib().es_accept_resample_noalloc(_ptr(p), _ptr(q), _ptr(d), _ptr(u) if u is not None else None,
                                          B, g1 - 1, V, 1 if greedy else 0, _ptr(n_acc), _ptr(tok),
                                          torch.cuda.current_stream().cuda_stream)
    if st != ES_OK:
        raise EasySpecError(st, "es_accept_resample_noalloc")
    return n_acc, tok


def es_sample(w: torch.Tensor, u: torch.Tensor):
    """Quantised categorical draw per row of w [B,V] f32 with draws u [B]."""
    if not isinstance(w, torch.Tensor) or w.dim() != 2:
        raise ValueError("w must be a [B, V] tensor")
    B, V = w.shape
    # the kernel reads w and u as dense device arrays of these sizes
    for name, t, dt, shp in (("w", w, torch.float32, (B, V)), ("u", u, torch.int64, (B,))):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.device != w.device:
            raise ValueError(f"{name} must be a CUDA tensor on w's device")
        if t.dtype != dt or tuple(t.shape) != shp or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous {dt} tensor of shape {shp}, "
                             f"got {t.dtype} {tuple(t.shape)}")
    idx = torch.empty(B, dtype=torch.int32, device=w.device)
    st = lib().es_sample(_ptr(w), _ptr(u), B, V, _ptr(idx), torch.cuda.current_stream().cuda_stream)
    if st != ES_OK:
        raise EasySpecError(st, "es_sample")
    return idx


def es_wait_selftest(limit_ns: int, arrive_ns: int) -> int:
    """Run the tensor-core passes' bounded wait alone; returns the es_status
    (ES_ERR_TIMEOUT when the wait gave up)."""
    return lib().es_wait_selftest(int(limit_ns), int(arrive_ns), torch.cuda.current_stream().cuda_stream)
