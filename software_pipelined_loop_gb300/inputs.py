"""Seeded synthetic inputs for the GEMM workloads.

This module is the one piece shared by the CPU oracle checks, the GPU parity
tests and the bench: it turns (seed, stream, element index) into matrix
entries and does no GEMM arithmetic.  Both sides of every comparison consume
the very same bytes produced here.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014; public-domain C by S. Vigna), used in its
counter form: draw i of a stream with state s is mix(s + (i + 1) * gamma).

Distributions (matching the workloads' stated value ranges):
  * int8 uniform on [-128, 127]: the top byte of a draw, read as two's
    complement.
  * fp16 uniform on [-1, 1]: u = (draw >> 40) * 2^-24 in [0, 1), value 2u - 1,
    rounded to binary16 (round to nearest even).
  * fp16 normal(0, 1) * scale: Box-Muller (cosine branch) on two consecutive
    draws in fp64, times scale, rounded to binary16.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_STREAM_MUL = 0xD1B54A32D192ED03

# Seeds of the five named workloads: base + workload index.
SEED_BASE = 0x5EED0000
STREAM_A = 0
STREAM_B = 1

_CHUNK = 1 << 22


def stream_state(seed: int, stream: int) -> int:
    """Initial SplitMix64 state of one stream of one seed."""
    return (int(seed) ^ ((int(stream) * _STREAM_MUL) & 0xFFFFFFFFFFFFFFFF)) & 0xFFFFFFFFFFFFFFFF


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def draws(state: int, start: int, count: int) -> np.ndarray:
    """Draws start .. start+count-1 of the stream whose state is `state` (uint64)."""
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(state) + idx * _GAMMA
        return _mix(z)


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def _fill(n: int, fn, dtype) -> np.ndarray:
    out = np.empty(n, dtype=dtype)
    spans = [(s, min(n, s + _CHUNK)) for s in range(0, n, _CHUNK)]
    if len(spans) <= 1:
        for s, e in spans:
            out[s:e] = fn(s, e - s)
        return out

    def work(span):
        s, e = span
        out[s:e] = fn(s, e - s)

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(work, spans))
    return out


def int8_uniform(seed: int, stream: int, rows: int, cols: int) -> np.ndarray:
    """rows x cols int8 matrix, uniform on [-128, 127], row-major."""
    st = stream_state(seed, stream)
    f = lambda s, c: (draws(st, s, c) >> np.uint64(56)).astype(np.uint8).view(np.int8)
    return _fill(rows * cols, f, np.int8).reshape(rows, cols)


def fp16_uniform(seed: int, stream: int, rows: int, cols: int) -> np.ndarray:
    """rows x cols float16 matrix, uniform on [-1, 1], row-major."""
    st = stream_state(seed, stream)

    def f(s, c):
        u = (draws(st, s, c) >> np.uint64(40)).astype(np.float64) * (2.0 ** -24)
        return (2.0 * u - 1.0).astype(np.float16)

    return _fill(rows * cols, f, np.float16).reshape(rows, cols)


def fp16_normal(seed: int, stream: int, rows: int, cols: int, scale: float = 1.0) -> np.ndarray:
    """rows x cols float16 matrix, normal(0, 1) times `scale`, row-major."""
    st = stream_state(seed, stream)

    def f(s, c):
        z = draws(st, 2 * s, 2 * c)
        u1 = ((z[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
        u2 = (z[1::2] >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
        v = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
        return (v * scale).astype(np.float16)

    return _fill(rows * cols, f, np.float16).reshape(rows, cols)


# The five named workloads.  index -> (name, dtype, M, N, K, distribution)
WORKLOADS = {
    0: ("int8_512", "s8", 512, 512, 512, "uniform"),
    1: ("fp16_1024", "f16", 1024, 1024, 1024, "uniform"),
    2: ("int8_4096", "s8", 4096, 4096, 4096, "uniform"),
    3: ("fp16_skinny_16384x128x16384", "f16", 16384, 128, 16384, "normal"),
    4: ("fp16_ragged_4093x3001x4107", "f16", 4093, 3001, 4107, "uniform"),
}


def make_operands(dtype: str, M: int, N: int, K: int, seed: int, dist: str = "uniform"):
    """A (M x K) and B (K x N) for one seed: stream 0 gives A, stream 1 gives B."""
    if dtype == "s8":
        return (int8_uniform(seed, STREAM_A, M, K), int8_uniform(seed, STREAM_B, K, N))
    if dist == "normal":
        sc = 1.0 / np.sqrt(K) if K > 0 else 1.0
        return (fp16_normal(seed, STREAM_A, M, K, sc), fp16_normal(seed, STREAM_B, K, N, sc))
    return (fp16_uniform(seed, STREAM_A, M, K), fp16_uniform(seed, STREAM_B, K, N))


def workload_operands(index: int):
    """(name, dtype, M, N, K, A, B) of one named workload."""
    name, dtype, M, N, K, dist = WORKLOADS[index]
    A, B = make_operands(dtype, M, N, K, SEED_BASE + index, dist)
    return name, dtype, M, N, K, A, B
