"""Counter-based random stream used by the speculative loop (oracle side).

TEST INFRASTRUCTURE ONLY -- see the package docstring.

The pages never say how random numbers are drawn; lossless speculative
sampling only needs independent uniforms.  Both the oracle and the CUDA
library therefore implement the same published generator, SplitMix64
(G. L. Steele Jr., D. Lea, C. H. Flood, "Fast Splittable Pseudorandom Number
Generators", OOPSLA 2014), each side from that definition, so that a seeded
run draws identical numbers on the CPU and on the GPU.

  splitmix64(x)   the first output of a SplitMix64 generator whose state is x:
                  the state is advanced by the golden gamma 0x9E3779B97F4A7C15
                  and passed through the 64-bit finaliser (xor-shift 30,
                  multiply, xor-shift 27, multiply, xor-shift 31).
  draw(seed, row, phase, slot, gamma)
                  splitmix64(seed XOR splitmix64(row * 2**32
                                                 + phase * (2*gamma + 1) + slot))
                  Slots 0..gamma-1: the draft samples d_1..d_gamma; slots
                  gamma..2*gamma-1: the accept tests of d_1..d_gamma; slot
                  2*gamma: the residual / bonus draw.
  uniform24(u)    (u >> 40) * 2**-24, an exact float32 in [0, 1).

Parity: pinned by tests/test_oracle_rng.py against the generator's published
output sequence for state 0 (tests/golden/splitmix64_seed0.txt).
"""
from __future__ import annotations

import numpy as np

MASK64 = (1 << 64) - 1
GOLDEN_GAMMA = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB


def _finalise(z: int) -> int:
    z = ((z ^ (z >> 30)) * _M1) & MASK64
    z = ((z ^ (z >> 27)) * _M2) & MASK64
    return z ^ (z >> 31)


def splitmix64(x: int) -> int:
    """First output of SplitMix64 started from state ``x``."""
    return _finalise((x + GOLDEN_GAMMA) & MASK64)


def splitmix64_sequence(state: int, n: int) -> list[int]:
    """The generator run as a stream: n successive outputs from ``state``."""
    out = []
    for _ in range(n):
        state = (state + GOLDEN_GAMMA) & MASK64
        out.append(_finalise(state))
    return out


def draw(seed: int, row: int, phase: int, slot: int, gamma: int) -> int:
    """64-bit draw for (sequence row, speculation phase, slot)."""
    counter = ((row << 32) + phase * (2 * gamma + 1) + slot) & MASK64
    return splitmix64((seed & MASK64) ^ splitmix64(counter))


def uniform24(u: int) -> np.float32:
    """Top 24 bits of a draw as an exact float32 uniform in [0, 1)."""
    return np.float32((u >> 40) * (2.0 ** -24))


def phase_draws(seed: int, row: int, phase: int, gamma: int) -> list[int]:
    """All 2*gamma+1 draws of one phase, in slot order."""
    return [draw(seed, row, phase, s, gamma) for s in range(2 * gamma + 1)]
