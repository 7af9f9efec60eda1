"""Seeded synthetic workloads for the fused FP16 MLP.

This module is the one place both the GPU path's tests/benchmark and the CPU
oracle take their inputs from. It holds no arithmetic of the method itself:
only the workload shapes and a counter-based random generator that turns a
seed into FP16 weights, biases and inputs.

Generator (published definition): SplitMix64 (Steele, Lea and Flood, "Fast
splittable pseudorandom number generators", OOPSLA 2014). The i-th output
(i = 1, 2, ...) of the stream with seed s is mix(s + i * 0x9E3779B97F4A7C15),
so any draw can be computed from its index alone. A draw becomes a uniform
double u = (z >> 11) * 2^-53 in [0, 1).

Draw order for one workload: for l = 1..L the weights W_l row-major, then its
biases b_l; then the inputs row-major. U(a, b) = a + (b - a) * u in double,
then rounded to float32 and to float16 (both round to nearest even). Normal
inputs use Box-Muller on two consecutive draws, z = sqrt(-2 ln(1 - u1)) *
cos(2 pi u2), clipped to [-4, 4].

Weights ~ U(-sqrt(6/fan_in), +sqrt(6/fan_in)), biases ~ U(-0.1, 0.1), inputs
~ U(-1, 1) (or the clipped normal), as the workload table below states.
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    """Draws start+1 .. start+count (1-based) of the SplitMix64 stream."""
    with np.errstate(over="ignore"):
        i = np.arange(start + 1, start + count + 1, dtype=np.uint64)
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + i * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def uniform01(seed: int, start: int, count: int) -> np.ndarray:
    return (splitmix64(seed, start, count) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def _to_f16_bits(v64: np.ndarray) -> np.ndarray:
    return v64.astype(np.float32).astype(np.float16).view(np.uint16)


def _uniform_f16(seed, start, count, lo, hi):
    u = uniform01(seed, start, count)
    return _to_f16_bits(lo + (hi - lo) * u)


def _normal_clipped_f16(seed, start, count, clip=4.0):
    u = uniform01(seed, start, 2 * count)
    u1, u2 = u[0::2], u[1::2]
    z = np.sqrt(-2.0 * np.log(1.0 - u1)) * np.cos(2.0 * math.pi * u2)
    return _to_f16_bits(np.clip(z, -clip, clip))


@dataclass(frozen=True)
class Workload:
    """One benchmark/parity workload.

    ``n_unique`` distinct inputs are generated; a dispatch evaluates each of
    them ``repeats`` times (the repeated rows are materialised as copies), so
    one dispatch is ``n_unique * repeats`` network evaluations.
    """
    name: str
    dims: tuple
    seed: int
    n_unique: int
    repeats: int = 1
    input_dist: str = "uniform"          # "uniform" U(-1,1) or "normal4" N(0,1) clipped to +-4
    description: str = field(default="", compare=False)

    @property
    def n_layers(self) -> int:
        return len(self.dims) - 1

    @property
    def n_evals(self) -> int:
        return self.n_unique * self.repeats

    @property
    def param_draws(self) -> int:
        d = self.dims
        return sum(d[l + 1] * d[l] + d[l + 1] for l in range(len(d) - 1))

    @property
    def flops_per_eval(self) -> int:
        d = self.dims
        return 2 * sum(d[l] * d[l + 1] for l in range(len(d) - 1))

    @property
    def hbm_bytes_per_eval(self) -> int:
        return 2 * (self.dims[0] + self.dims[-1])


WORKLOADS = {
    "tiny": Workload(
        "tiny", (32, 32, 32, 32, 32, 32, 32, 32, 16), seed=0, n_unique=65536,
        description="8 affine layers 32x7->16, 65,536 U(-1,1) inputs, one pass, seed 0"),
    "page": Workload(
        "page", (48, 64, 64, 64, 64, 64, 64, 64, 16), seed=1, n_unique=65536, repeats=16,
        description="page-shaped 48->64x7->16, 65,536 inputs x 16 = 1,048,576 evals, seed 1"),
    "ablation": Workload(
        "ablation", (48, 64, 64, 64, 64, 64, 64, 64, 16), seed=1, n_unique=65536, repeats=16,
        description="the page-shaped network and inputs x 16 = 1,048,576 evals (layout/activation ablations)"),
    "tiny_ablation": Workload(
        "tiny_ablation", (32, 32, 32, 32, 32, 32, 32, 32, 16), seed=0, n_unique=65536, repeats=16,
        description="the tiny network and its inputs x 16 = 1,048,576 evals (layout/activation ablations)"),
    "wide": Workload(
        "wide", (64, 128, 128, 128, 128, 128, 128, 128, 16), seed=3, n_unique=16777216,
        description="64->128x7->16, 16,777,216 U(-1,1) inputs, one pass, seed 3"),
    "hetero": Workload(
        "hetero", (64, 128, 256, 256, 128, 128, 64, 64, 16), seed=4, n_unique=4194304,
        input_dist="normal4",
        description="64->128->256->256->128->128->64->64->16, 4,194,304 N(0,1) clipped inputs, seed 4"),
}


def net_params(dims, seed):
    """FP16 bits of W_l ([d_{l+1}, d_l] row-major) and b_l for l = 1..L."""
    W, b = [], []
    pos = 0
    for l in range(len(dims) - 1):
        K, N = int(dims[l]), int(dims[l + 1])
        a = math.sqrt(6.0 / K)
        W.append(_uniform_f16(seed, pos, N * K, -a, a).reshape(N, K))
        pos += N * K
        b.append(_uniform_f16(seed, pos, N, -0.1, 0.1))
        pos += N
    return W, b


def inputs(w: Workload, row_start: int = 0, row_count: int | None = None,
           threads: int = 0) -> np.ndarray:
    """FP16 bits [row_count, d_0] of unique input rows row_start.. of ``w``."""
    if row_count is None:
        row_count = w.n_unique - row_start
    d0 = w.dims[0]
    base = w.param_draws
    out = np.empty((row_count, d0), dtype=np.uint16)

    def fill(r0, r1):
        cnt = (r1 - r0) * d0
        if w.input_dist == "uniform":
            v = _uniform_f16(w.seed, base + (row_start + r0) * d0, cnt, -1.0, 1.0)
        elif w.input_dist == "normal4":
            v = _normal_clipped_f16(w.seed, base + 2 * (row_start + r0) * d0, cnt)
        else:
            raise ValueError(w.input_dist)
        out[r0:r1] = v.reshape(r1 - r0, d0)

    chunk = 1 << 18
    spans = [(r, min(r + chunk, row_count)) for r in range(0, row_count, chunk)]
    if threads == 0:
        import os
        threads = min(16, os.cpu_count() or 1)
    if len(spans) <= 1 or threads <= 1:
        for s in spans:
            fill(*s)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(lambda s: fill(*s), spans))
    return out


def small_net_inputs(dims, seed, n, dist="uniform"):
    """Weights, biases and n inputs of an arbitrary net (for parity sweeps)."""
    w = Workload("adhoc", tuple(int(d) for d in dims), seed=seed, n_unique=n, input_dist=dist)
    W, b = net_params(w.dims, seed)
    return W, b, inputs(w)
