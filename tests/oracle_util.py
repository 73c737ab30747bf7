"""Helpers shared by the oracle tests (tiny shapes, weight conversion)."""
import numpy as np

from layer_drafting_draft_b300 import synth
from oracle import model as M


def shape_of(s: dict) -> M.Shape:
    return M.Shape(**s)


def tiny_shapes(V=64, d=32, Ld=4, Lb=3, H=4, Hkv=2, F=48, theta=1e4):
    sd = synth.shape(Ld, d, H, Hkv, F, V, theta)
    sb = synth.shape(Lb, 2 * d, 2 * H, Hkv, 2 * F, V, theta)
    return sd, sb


def tiny_pair(seed=0, V=64, std=0.02, **kw):
    sd, sb = tiny_shapes(V=V, **kw)
    Wd = M.as_f64_weights(synth.make_weights(sd, 100 + seed, "f32", "cpu", std))
    Wb = M.as_f64_weights(synth.make_weights(sb, 200 + seed, "f32", "cpu", std))
    return Wd, shape_of(sd), Wb, shape_of(sb)


def zero_layer(lw):
    return {k: (np.ones_like(v) if k.endswith("norm") else np.zeros_like(v)) for k, v in lw.items()}
