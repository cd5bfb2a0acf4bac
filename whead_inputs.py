"""Seeded synthetic inputs for the serial draft-head walk.

This module is shared by the tests, the benchmark and the smoke check. It only draws random numbers
and stores them in the walk's input formats: it holds none of the walk's arithmetic, so both the CPU
oracle and the CUDA library receive identical bytes without sharing any computation.

Distributions follow the workloads of "Weights That Stay: On-Chip Megakernels for Serial Heads in
Speculative Decoding" (Qwen3 vocabularies of 151,936 and 248,064 rows, rank 256): W ~ N(0, 1/r),
E ~ N(0, 1), initial state ~ N(0, 1), base logits ~ N(0, 2), recurrent A ~ N(0, 1/r), c = 0, where
N(0, s) means mean 0 and variance s. Each tensor has its own stream: numpy's Philox bit generator
keyed on (seed, tensor id) with ids W=1, E=2, u0=3, base=4, A=5, h0=6.
"""
from __future__ import annotations

import math

import numpy as np

TENSOR_ID = {"W": 1, "E": 2, "u0": 3, "base": 4, "A": 5, "h0": 6}

MARKOV = 0
RECURRENT = 1

# Named workloads: kind, V, r, B, gamma, T. The sweep workload is expanded by the tests.
WORKLOADS = {
    "markov_v4096_r64_b1_g4": dict(kind=MARKOV, V=4096, r=64, B=1, gamma=4, T=0.0),
    "markov_v151936_r256_b1_g16": dict(kind=MARKOV, V=151936, r=256, B=1, gamma=16, T=0.0),
    "markov_v248064_r256_b1_g16": dict(kind=MARKOV, V=248064, r=256, B=1, gamma=16, T=0.0),
    "markov_v248064_r256_b4_g16": dict(kind=MARKOV, V=248064, r=256, B=4, gamma=16, T=0.0),
    "recurrent_v151936_r256_b1_g15": dict(kind=RECURRENT, V=151936, r=256, B=1, gamma=15, T=0.0),
    # the same tensors with W in E4M3 (one scale per row) and the state split into two E4M3 vectors
    "markov_v151936_r256_b1_g16_e4m3": dict(kind=MARKOV, V=151936, r=256, B=1, gamma=16, T=0.0, w="e4m3"),
    "markov_v248064_r256_b1_g16_e4m3": dict(kind=MARKOV, V=248064, r=256, B=1, gamma=16, T=0.0, w="e4m3"),
    "markov_v248064_r256_b4_g16_e4m3": dict(kind=MARKOV, V=248064, r=256, B=4, gamma=16, T=0.0, w="e4m3"),
}
SWEEP = dict(kind=MARKOV, V=151936, r=256, gammas=(1, 7, 16), Bs=(1, 2, 4, 8, 16), Ts=(0.0, 1.0))


def _gen(seed: int, name: str) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(key=[int(seed) & (2**64 - 1), TENSOR_ID[name]]))


def normal_f32(seed: int, name: str, shape, variance: float) -> np.ndarray:
    g = _gen(seed, name)
    x = g.standard_normal(size=shape, dtype=np.float32)
    return (x * np.float32(math.sqrt(variance))).astype(np.float32)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Store float32 values in bf16 (round to nearest even) and return the raw 16-bit patterns."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def make_inputs(kind: int, V: int, r: int, B: int, gamma: int, seed: int = 0) -> dict:
    """W, E (uint16 bf16 patterns, V x r), base (B x gamma x V fp32), s0 (B x r fp32), A, c."""
    W = to_bf16_bits(normal_f32(seed, "W", (V, r), 1.0 / r))
    E = to_bf16_bits(normal_f32(seed, "E", (V, r), 1.0))
    base = normal_f32(seed, "base", (B, gamma, V), 2.0)
    if kind == MARKOV:
        s0 = normal_f32(seed, "u0", (B, r), 1.0)
        A = None
        c = None
    else:
        s0 = normal_f32(seed, "h0", (B, r), 1.0)
        A = normal_f32(seed, "A", (r, r), 1.0 / r)
        c = np.zeros((r,), dtype=np.float32)
    return dict(kind=kind, W=W, E=E, base=base, s0=s0, A=A, c=c)


def workload_inputs(name: str, seed: int = 0) -> dict:
    w = WORKLOADS[name]
    d = make_inputs(w["kind"], w["V"], w["r"], w["B"], w["gamma"], seed)
    d["T"] = w["T"]
    return d
