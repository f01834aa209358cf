"""Pins of the CPU oracle against what the pages and the mathematics fix.

No GPU is needed.  Every pin is a function of an ``oracle.Oracle`` so that the
last test can rerun the whole set on deliberately broken builds of the C
oracle (a dropped k term, a flipped sign, a wrong index, a wrong exponent
bias, a wrong factor) and show that each such mistake fails at least one pin.

What pins what:
  * brute force with Python integers / exact rationals on tiny non-square
    shapes (the plain definition; non-square so a transposed operand shows);
  * identity operands (C = B, C = A), all-ones operands (column and row sums),
    rank-one operands (C = K a_i b_j), int8 extremes (C = 16384 K) and the
    int32 range limit;
  * linearity in B;
  * the binary16 decoder against numpy's own conversion for all 65536 bit
    patterns;
  * the shared-memory budget against the worked example printed on the
    "Pipeline GPU Kernel" skill page, Step 1 (tests/golden/);
  * the compute/load ratio of Step 2 against a count of multiply-adds and of
    loaded elements by enumeration.
"""
from __future__ import annotations

import json
import os
import re
import tempfile
from fractions import Fraction

import numpy as np
import pytest

import oracle
from software_pipelined_loop_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

TINY_SHAPES = [(m, n, k) for m in (1, 2, 3, 5) for n in (1, 2, 4, 5) for k in (1, 2, 3, 7)] + [
    (7, 11, 13), (8, 3, 16), (4, 9, 16), (13, 1, 5)]


# ----------------------------------------------------------------- helpers

def fraction_to_f32(q: Fraction) -> np.float32:
    """Exact rational -> nearest binary32, ties to even (no double rounding)."""
    if q == 0:
        return np.float32(0.0)
    neg = q < 0
    q = -q if neg else q
    e = q.numerator.bit_length() - q.denominator.bit_length()
    while Fraction(2) ** e > q:
        e -= 1
    while Fraction(2) ** (e + 1) <= q:
        e += 1
    ulp_e = max(e - 23, -149)
    scaled = q / (Fraction(2) ** ulp_e)
    n = scaled.numerator // scaled.denominator
    rem = scaled - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    v = float(n) * 2.0 ** ulp_e
    return np.float32(-v if neg else v)


def exact_f16_gemm(A: np.ndarray, B: np.ndarray) -> np.ndarray:
    M, K = A.shape
    N = B.shape[1]
    Af = [[Fraction(float(x)) for x in row] for row in A]
    Bf = [[Fraction(float(x)) for x in row] for row in B]
    C = np.zeros((M, N), dtype=np.float32)
    for i in range(M):
        for j in range(N):
            C[i, j] = fraction_to_f32(sum((Af[i][k] * Bf[k][j] for k in range(K)), Fraction(0)))
    return C


def exact_int_gemm(A: np.ndarray, B: np.ndarray) -> np.ndarray:
    M, K = A.shape
    N = B.shape[1]
    a = A.astype(object)
    b = B.astype(object)
    C = np.zeros((M, N), dtype=np.int64)
    for i in range(M):
        for j in range(N):
            s = 0
            for k in range(K):
                s += int(a[i, k]) * int(b[k, j])
            C[i, j] = s
    return C


# -------------------------------------------------------------------- pins

def pin_int8_brute_force(o):
    for idx, (M, N, K) in enumerate(TINY_SHAPES):
        A, B = inputs.make_operands("s8", M, N, K, seed=1000 + idx)
        got = o.gemm_s8s8s32(A, B, threads=3)
        assert got.dtype == np.int32 and got.shape == (M, N)
        assert np.array_equal(got.astype(np.int64), exact_int_gemm(A, B)), (M, N, K)


def pin_fp16_brute_force(o):
    # |values| <= 1 and K <= 16: every partial sum is a multiple of 2^-48 below
    # 2^5, so the fp64 accumulation is exact and the one rounding is the
    # correctly rounded value of the exact rational sum.
    for idx, (M, N, K) in enumerate(TINY_SHAPES):
        A, B = inputs.make_operands("f16", M, N, K, seed=2000 + idx)
        got = o.gemm_f16f32(A, B, threads=2)
        assert got.dtype == np.float32 and got.shape == (M, N)
        assert np.array_equal(got, exact_f16_gemm(A, B)), (M, N, K)


def pin_identity(o):
    M, N = 23, 17
    I = np.eye(M, dtype=np.int8)
    _, B = inputs.make_operands("s8", M, N, M, seed=3)
    assert np.array_equal(o.gemm_s8s8s32(I, B), B.astype(np.int32))
    A, _ = inputs.make_operands("s8", M, N, N, seed=4)
    assert np.array_equal(o.gemm_s8s8s32(A, np.eye(N, dtype=np.int8)), A.astype(np.int32))
    Ih = np.eye(M, dtype=np.float16)
    _, Bh = inputs.make_operands("f16", M, N, M, seed=5)
    assert np.array_equal(o.gemm_f16f32(Ih, Bh), Bh.astype(np.float32))
    Ah, _ = inputs.make_operands("f16", M, N, N, seed=6)
    assert np.array_equal(o.gemm_f16f32(Ah, np.eye(N, dtype=np.float16)), Ah.astype(np.float32))


def pin_all_ones(o):
    M, N, K = 9, 31, 70
    A, B = inputs.make_operands("s8", M, N, K, seed=7)
    ones_a = np.ones((M, K), dtype=np.int8)
    ones_b = np.ones((K, N), dtype=np.int8)
    col = B.astype(np.int64).sum(axis=0)
    row = A.astype(np.int64).sum(axis=1)
    assert np.array_equal(o.gemm_s8s8s32(ones_a, B), np.broadcast_to(col, (M, N)))
    assert np.array_equal(o.gemm_s8s8s32(A, ones_b), np.broadcast_to(row[:, None], (M, N)))
    assert np.array_equal(o.gemm_s8s8s32(ones_a, ones_b), np.full((M, N), K))
    Ah, Bh = inputs.make_operands("f16", M, N, K, seed=8)
    # Sums of binary16 values in [-1, 1]: multiples of 2^-24 below 2^7, exact
    # in fp64 in any order; one rounding to fp32.
    colh = Bh.astype(np.float64).sum(axis=0).astype(np.float32)
    rowh = Ah.astype(np.float64).sum(axis=1).astype(np.float32)
    assert np.array_equal(o.gemm_f16f32(np.ones((M, K), np.float16), Bh), np.broadcast_to(colh, (M, N)))
    assert np.array_equal(o.gemm_f16f32(Ah, np.ones((K, N), np.float16)), np.broadcast_to(rowh[:, None], (M, N)))


def pin_rank_one(o):
    M, N, K = 6, 10, 37
    a = np.arange(-3, 3, dtype=np.int8)
    b = np.arange(-5, 5, dtype=np.int8)
    A = np.repeat(a[:, None], K, axis=1)
    B = np.repeat(b[None, :], K, axis=0)
    want = K * np.outer(a.astype(np.int64), b.astype(np.int64))
    assert np.array_equal(o.gemm_s8s8s32(A, B), want)
    ah = np.array([0.5, -0.25, 1.0, 0.125, -1.0, 0.75], dtype=np.float16)
    bh = np.linspace(-1, 1, N).astype(np.float16)
    Ah = np.repeat(ah[:, None], K, axis=1)
    Bh = np.repeat(bh[None, :], K, axis=0)
    wanth = (K * np.outer(ah.astype(np.float64), bh.astype(np.float64))).astype(np.float32)
    assert np.array_equal(o.gemm_f16f32(Ah, Bh), wanth)


def pin_int8_extremes(o):
    K = 1024
    A = np.full((3, K), -128, np.int8)
    B = np.full((K, 5), -128, np.int8)
    assert np.array_equal(o.gemm_s8s8s32(A, B), np.full((3, 5), 16384 * K))
    B2 = np.full((K, 5), 127, np.int8)
    assert np.array_equal(o.gemm_s8s8s32(A, B2), np.full((3, 5), -16256 * K))
    # The int32 limit: 16384 * 131071 fits, 16384 * 131072 = 2^31 does not.
    Kmax = 131071
    assert o.gemm_s8s8s32(np.full((1, Kmax), -128, np.int8), np.full((Kmax, 1), -128, np.int8))[0, 0] == 16384 * Kmax
    with pytest.raises(oracle.OracleError):
        o.gemm_s8s8s32(np.full((1, Kmax + 1), -128, np.int8), np.full((Kmax + 1, 1), -128, np.int8))


def pin_linearity(o):
    M, N, K = 11, 19, 45
    A, _ = inputs.make_operands("s8", M, N, K, seed=9)
    _, B1 = inputs.make_operands("s8", M, N, K, seed=10)
    _, B2 = inputs.make_operands("s8", M, N, K, seed=11)
    B1 = (B1 // 2).astype(np.int8)
    B2 = (B2 // 2).astype(np.int8)
    lhs = o.gemm_s8s8s32(A, (B1 + B2).astype(np.int8)).astype(np.int64)
    rhs = o.gemm_s8s8s32(A, B1).astype(np.int64) + o.gemm_s8s8s32(A, B2)
    assert np.array_equal(lhs, rhs)


def pin_rows_and_threads(o):
    M, N, K = 37, 29, 53
    A, B = inputs.make_operands("f16", M, N, K, seed=12)
    full1 = o.gemm_f16f32(A, B, threads=1)
    full5 = o.gemm_f16f32(A, B, threads=5)
    assert np.array_equal(full1, full5)
    rows = [M - 1, 0, 17, 17]
    assert np.array_equal(o.gemm_f16f32(A, B, rows=rows, threads=3), full1[rows])
    A8, B8 = inputs.make_operands("s8", M, N, K, seed=13)
    f8 = o.gemm_s8s8s32(A8, B8)
    assert np.array_equal(o.gemm_s8s8s32(A8, B8, rows=rows), f8[rows])
    assert np.array_equal(f8.astype(np.int64), exact_int_gemm(A8, B8))


def pin_empty_k(o):
    A = np.zeros((3, 0), np.int8)
    B = np.zeros((0, 4), np.int8)
    assert np.array_equal(o.gemm_s8s8s32(A, B), np.zeros((3, 4), np.int32))
    assert np.array_equal(o.gemm_f16f32(A.astype(np.float16), B.astype(np.float16)),
                          np.zeros((3, 4), np.float32))


def pin_f16_decoder(o):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([o.f16_to_f64(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def pin_smem_budget(o):
    with open(os.path.join(GOLDEN, "smem_budget_example.json")) as f:
        g = json.load(f)
    BM, BN, BK, eb = g["BM"], g["BN"], g["BK"], g["elem_bytes"]
    assert o.smem_a_bytes(BM, BK, eb) == g["single_a_bytes"]
    assert o.smem_b_bytes(BK, BN, eb) == g["single_b_bytes"]
    assert o.smem_a_bytes(BM, BK, eb) + o.smem_b_bytes(BK, BN, eb) == g["single_total_bytes"]
    assert o.smem_doubled_bytes(BM, BN, BK, eb) == g["doubled_total_bytes"]
    assert o.smem_doubled_bytes(BM, BN, BK, eb) < g["ga104_cliff_bytes_per_block"]
    # A and B differ once the tile is not square.
    assert o.smem_doubled_bytes(64, 128, 32, 2) == 2 * (64 * 32 * 2) + 2 * (32 * 128 * 2)


def pin_ratio_by_enumeration(o):
    for BM, BN, BK, eb in [(4, 8, 2, 2), (3, 5, 7, 4), (16, 16, 16, 1), (8, 2, 6, 2), (32, 32, 32, 2)]:
        macs = sum(1 for _m in range(BM) for _n in range(BN) for _k in range(BK))
        loaded = len({("a", m, k) for m in range(BM) for k in range(BK)} |
                     {("b", k, n) for k in range(BK) for n in range(BN)})
        want = 2 * macs / (loaded * eb)
        assert o.compute_load_ratio(BM, BN, BK, eb) == pytest.approx(want, rel=1e-15)


ALL_PINS = [pin_int8_brute_force, pin_fp16_brute_force, pin_identity, pin_all_ones,
            pin_rank_one, pin_int8_extremes, pin_linearity, pin_rows_and_threads,
            pin_empty_k, pin_f16_decoder, pin_smem_budget, pin_ratio_by_enumeration]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin, oracle_lib):
    pin(oracle_lib)


def test_workload_inputs_are_deterministic():
    a1, b1 = inputs.make_operands("f16", 33, 17, 65, seed=inputs.SEED_BASE + 1)
    a2, b2 = inputs.make_operands("f16", 33, 17, 65, seed=inputs.SEED_BASE + 1)
    assert a1.tobytes() == a2.tobytes() and b1.tobytes() == b2.tobytes()
    assert np.abs(a1.astype(np.float64)).max() <= 1.0
    i8, _ = inputs.make_operands("s8", 64, 64, 4096, seed=5)
    assert i8.min() == -128 and i8.max() == 127


def test_splitmix64_published_vector():
    # SplitMix64 seeded with 1234567: the first five outputs of the published
    # reference implementation.
    got = [int(x) for x in inputs.draws(1234567, 0, 5)]
    assert got == [6457827717110365317, 3203168211198807973, 9817491932198370423,
                   4593380528125082431, 16408922859458223821]


# Each mutation is a plausible slip; every one must make some pin fail.
MUTATIONS = [
    ("drop last k term", r"for \(int64_t k = 0; k < K; \+\+k\)", "for (int64_t k = 0; k < K - 1; ++k)"),
    ("sign of accumulation", r"acc\[j\] \+= a \*", "acc[j] -= a *"),
    ("columns reversed on store", r"C\[p \* N \+ j\] = \(float\)acc\[j\]", "C[p * N + j] = (float)acc[N - 1 - j]"),
    ("rows reversed", r"jb->rows\[p\] : p;", "jb->rows[p] : (jb->M - 1 - p);"),
    ("exponent bias", r"e - 25\)", "e - 24)"),
    ("subnormal scale", r"\(double\)f, -24\)", "(double)f, -25)"),
    ("ratio factor", r"double flops = 2\.0 \*", "double flops = 1.0 *"),
    ("ratio B-tile index", r"\(BM \* BK \+ BK \* BN\)", "(BM * BK + BM * BN)"),
    ("budget B not doubled", r"oracle_smem_b_bytes\(BK, BN, elem_bytes\) \* 2", "oracle_smem_b_bytes(BK, BN, elem_bytes) * 1"),
]


@pytest.mark.parametrize("name,pattern,repl", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_mutation(name, pattern, repl, tmp_path):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "gemm_oracle.c")).read()
    mutated, n = re.subn(pattern, repl, src)
    assert n >= 1, f"mutation {name!r} did not apply"
    path = tmp_path / "mutant.c"
    path.write_text(mutated)
    lib = oracle.load_library(oracle.build(force=True, src=str(path), out=str(tmp_path / "libmutant.so")))
    o = oracle.Oracle(lib)
    failed = []
    for pin in ALL_PINS:
        try:
            pin(o)
        except (AssertionError, oracle.OracleError, pytest.fail.Exception):
            failed.append(pin.__name__)
    assert failed, f"no pin caught mutation {name!r}"
