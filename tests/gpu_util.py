"""Helpers for the GPU parity tests: a CUDA context plus the oracle twin."""
import numpy as np
import torch

from layer_drafting_draft_b300 import synth
from layer_drafting_draft_b300.easyspec import ES_ATTN_ONLY, ES_FULL_LAYER, EasySpec
from oracle import model as M
from oracle import spec

MODES = {ES_ATTN_ONLY: M.ATTN_ONLY, ES_FULL_LAYER: M.FULL_LAYER}


def starts_of(groups):
    return [g[0] for g in groups]


class Pair:
    """Weights generated once on the GPU; the oracle receives a float64 copy."""

    def __init__(self, sd: dict, sb: dict, dtype: str, seed: int, sigma=None):
        self.sd, self.sb, self.dtype = sd, sb, dtype
        self.wb = synth.make_weights(sb, 1000 * seed + 2, dtype, "cuda")
        if sigma is None:
            self.wd = synth.make_weights(sd, 1000 * seed + 1, dtype, "cuda")
        else:
            self.wd = synth.perturbed_copy(self.wb, sigma, 1000 * seed + 4)
        torch.cuda.synchronize()
        self.Wd = M.as_f64_weights(self.wd)
        self.Wb = M.as_f64_weights(self.wb)
        self.shape_d = M.Shape(**sd)
        self.shape_b = M.Shape(**sb)

    def gpu(self, max_batch=1, max_seq=256, max_gamma=8, mode=ES_FULL_LAYER, groups=None):
        return EasySpec(self.wd, self.sd, self.wb, self.sb, self.dtype, max_batch, max_seq,
                        max_gamma, mode, None if groups is None else starts_of(groups))

    def oracle(self, k=1, mode=ES_FULL_LAYER, groups=None, max_len=256, calibrate=True):
        # a bf16 pair keeps its K/V cache in bf16 on both sides
        return spec.SpecDecoder(self.Wd, self.shape_d, self.Wb, self.shape_b, groups=groups,
                                k=k, mode=MODES[mode], max_len=max_len, calibrate=calibrate,
                                kv_dtype="bf16" if self.dtype == "bf16" else "f64")


def rel_l2(a, b):
    a = np.asarray(a, np.float64); b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))
