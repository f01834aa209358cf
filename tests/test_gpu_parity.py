"""GPU parity: the CUDA library through the C ABI against the CPU oracle.

INT8 results must equal the oracle bit for bit.  FP16 results (fp32
accumulation on the tensor cores) must be within max-abs 1e-2 and relative
Frobenius 1e-4 of the oracle's fp64-accumulated product.

Every test compares every element of C, the full-size workloads included
(their oracle products are computed once per session, see conftest).
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from software_pipelined_loop_gb300 import gemmpipe, inputs

pytestmark = pytest.mark.gpu

MAX_ABS = 1e-2
MAX_REL_FRO = 1e-4


@pytest.fixture(scope="module")
def dev():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from software_pipelined_loop_gb300 import build
    build.build()
    gemmpipe.load()
    gemmpipe.gemmpipe_set_plan_override(-1, 0, 0)
    yield torch.device("cuda:0")
    gemmpipe.gemmpipe_set_plan_override(-1, 0, 0)


def to_dev(a: np.ndarray, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def run_f16(A: np.ndarray, B: np.ndarray, dev) -> np.ndarray:
    import torch
    M, K = A.shape
    N = B.shape[1]
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
    gemmpipe.gemm_f16f32(M, N, K, to_dev(A, dev), to_dev(B, dev), C)
    assert gemmpipe.gemmpipe_get_device_status() == gemmpipe.OK
    return C.cpu().numpy()


def run_s8(A: np.ndarray, B: np.ndarray, dev) -> np.ndarray:
    import torch
    M, K = A.shape
    N = B.shape[1]
    C = torch.full((M, N), -7, dtype=torch.int32, device=dev)
    gemmpipe.gemm_s8s8s32(M, N, K, to_dev(A, dev), to_dev(B, dev), C)
    assert gemmpipe.gemmpipe_get_device_status() == gemmpipe.OK
    return C.cpu().numpy()


def assert_f16_close(got: np.ndarray, ref: np.ndarray, what=""):
    assert got.shape == ref.shape
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    d = got.astype(np.float64) - ref.astype(np.float64)
    err = np.abs(d).max() if d.size else 0.0
    nrm = np.linalg.norm(ref.astype(np.float64))
    rel = np.linalg.norm(d) / nrm if nrm > 0 else np.linalg.norm(d)
    assert err <= MAX_ABS and rel <= MAX_REL_FRO, f"{what}: max-abs {err:.3g} rel-fro {rel:.3g}"


def sample_rows(M: int, n_random: int = 24, seed: int = 7) -> np.ndarray:
    fixed = {0, 1, 63, 64, 127, 128, 129, 255, 256, M // 2, M - 129, M - 128, M - 2, M - 1}
    rng = np.random.default_rng(seed)
    rnd = set(int(x) for x in rng.integers(0, M, n_random))
    return np.array(sorted(r for r in fixed | rnd if 0 <= r < M), dtype=np.int64)


# --------------------------------------------------------------- small sweeps

SWEEP = [
    # (M, N, K): aligned pitches (TMA producer) and odd ones (bounded loads)
    (1, 8, 8), (1, 1, 1), (17, 24, 64), (128, 128, 64), (129, 136, 72), (300, 264, 192),
    (128, 256, 128), (255, 512, 1000), (64, 8, 4096), (129, 129, 129), (15, 17, 127),
    (16, 16, 16), (127, 1, 65), (200, 300, 17), (33, 513, 250), (300, 7, 1031),
]


@pytest.mark.parametrize("M,N,K", SWEEP)
def test_f16_sweep(dev, M, N, K):
    A, B = inputs.make_operands("f16", M, N, K, seed=100 + M + 7 * N + 13 * K)
    assert_f16_close(run_f16(A, B, dev), oracle.gemm_f16f32(A, B), f"{M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", SWEEP)
def test_s8_sweep(dev, M, N, K):
    A, B = inputs.make_operands("s8", M, N, K, seed=200 + M + 7 * N + 13 * K)
    assert np.array_equal(run_s8(A, B, dev), oracle.gemm_s8s8s32(A, B))


# The page's pitfalls (last K tile dropped, off-by-one in the buffer index):
# number of k-blocks around the ring depth S (4 for 128x256 tiles, 6 for
# 128x128), including the last tile being a partial one.
@pytest.mark.parametrize("num_kb", [1, 2, 3, 4, 5, 6, 7, 9, 13])
@pytest.mark.parametrize("N", [128, 256])
def test_ring_depth_edges(dev, num_kb, N):
    for K in (64 * num_kb, 64 * num_kb - 24):
        A, B = inputs.make_operands("f16", 256, N, K, seed=300 + num_kb + K)
        assert_f16_close(run_f16(A, B, dev), oracle.gemm_f16f32(A, B), f"K={K}")


@pytest.mark.parametrize("producer", [0, 1])
@pytest.mark.parametrize("bn", [128, 256])
def test_forced_producer_and_tile(dev, producer, bn):
    M, N, K = 384, 520, 704
    A, B = inputs.make_operands("f16", M, N, K, seed=400 + bn + producer)
    gemmpipe.gemmpipe_set_plan_override(producer, bn, 0)
    try:
        plan = gemmpipe.gemmpipe_plan(1, M, N, K)
        assert plan["producer"] == producer and plan["BN"] == bn
        got = run_f16(A, B, dev)
    finally:
        gemmpipe.gemmpipe_set_plan_override(-1, 0, 0)
    assert_f16_close(got, oracle.gemm_f16f32(A, B))


def test_misaligned_base_pointers(dev):
    import torch
    # A and B start 2 bytes past a 16-byte boundary, C 4 bytes past: the
    # bounded-load producer and 4-byte stores must take over.
    M, N, K = 200, 136, 264
    A, B = inputs.make_operands("f16", M, N, K, seed=11)
    ab = torch.zeros(M * K + 8, dtype=torch.float16, device=dev)
    bb = torch.zeros(K * N + 8, dtype=torch.float16, device=dev)
    cb = torch.zeros(M * N + 4, dtype=torch.float32, device=dev)
    ab[1:1 + M * K] = to_dev(A.reshape(-1), dev)
    bb[1:1 + K * N] = to_dev(B.reshape(-1), dev)
    a_ptr, b_ptr, c_ptr = ab.data_ptr() + 2, bb.data_ptr() + 2, cb.data_ptr() + 4
    ref = oracle.gemm_f16f32(A, B)
    for forced, producer, copy in ((-1, 0, 2), (1, 1, 0)):
        gemmpipe.gemmpipe_set_plan_override(forced, 0, 0)
        try:
            plan = gemmpipe.gemmpipe_plan(1, M, N, K, a_ptr, b_ptr, c_ptr)
            assert plan["producer"] == producer and plan["operand_copy"] == copy and plan["vector_store"] == 0
            cb.zero_()
            gemmpipe.gemm_f16f32(M, N, K, a_ptr, b_ptr, c_ptr)
            assert gemmpipe.gemmpipe_get_device_status() == gemmpipe.OK
        finally:
            gemmpipe.gemmpipe_set_plan_override(-1, 0, 0)
        got = cb[1:1 + M * N].cpu().numpy().reshape(M, N)
        assert_f16_close(got, ref)
        assert cb[0].item() == 0 and cb[M * N + 1:].abs().sum().item() == 0


@pytest.mark.parametrize("dtype,M,N,K", [("f16", 600, 1000, 512), ("f16", 517, 771, 300),
                                         ("s8", 600, 1000, 1100), ("s8", 300, 517, 200)])
@pytest.mark.parametrize("c_off", [4, 8, 12])
def test_c_rows_off_16_bytes(dev, dtype, M, N, K, c_off):
    """C rows that do not start on 16-byte boundaries (C's base 4, 8 or 12
    bytes past one; N a multiple of 8 or odd, so that the rows' offsets vary)
    on every tile plan, split tiles included: no TMA store can take them, so
    the epilogue writes one row piece per warp store.  Every element against
    the oracle, and nothing written outside C."""
    import torch
    A, B = inputs.make_operands(dtype, M, N, K, seed=71 + c_off)
    ref = oracle.gemm_s8s8s32(A, B) if dtype == "s8" else oracle.gemm_f16f32(A, B)
    pad = 64
    cdt = torch.int32 if dtype == "s8" else torch.float32
    buf = torch.full((pad + M * N + pad,), 777, dtype=cdt, device=dev)
    c_ptr = buf.data_ptr() + 4 * pad + c_off
    assert c_ptr % 16 == c_off
    Ad, Bd = to_dev(A, dev), to_dev(B, dev)
    fn = gemmpipe.gemm_s8s8s32 if dtype == "s8" else gemmpipe.gemm_f16f32
    # (producer, bn, stages, cta_pair, split): default, CTA pair, quad, single CTA, pair with forced split
    plans = [(-1, 0, 0, -1, -1), (-1, 256, 0, 1, -1), (-1, 256, 0, 2, -1), (-1, 128, 0, 0, -1), (-1, 256, 0, 1, 1)]
    for ov in plans:
        gemmpipe.gemmpipe_set_plan_override(*ov)
        try:
            plan = gemmpipe.gemmpipe_plan(0 if dtype == "s8" else 1, M, N, K, Ad, Bd, c_ptr)
            assert plan["vector_store"] == 0
            buf.fill_(777)
            fn(M, N, K, Ad, Bd, c_ptr)
            assert gemmpipe.gemmpipe_get_device_status() == gemmpipe.OK
        finally:
            gemmpipe.gemmpipe_set_plan_override(-1, 0, 0, -1, -1)
        host = buf.cpu().numpy()
        c0 = pad + c_off // 4
        got = host[c0:c0 + M * N].reshape(M, N)
        assert (host[:c0] == 777).all(), (ov, "elements before C written")
        assert (host[c0 + M * N:] == 777).all(), (ov, "elements after C written")
        if dtype == "s8":
            assert np.array_equal(got, ref), (ov, plan)
        else:
            assert_f16_close(got, ref, str((ov, plan["cta_pair"], plan["BN"])))


def test_guard_bands_untouched(dev):
    import torch
    M, N, K = 257, 264, 128
    A, B = inputs.make_operands("f16", M, N, K, seed=12)
    pad = 4096
    buf = torch.full((pad + M * N + pad,), 12345.0, dtype=torch.float32, device=dev)
    c_ptr = buf.data_ptr() + 4 * pad
    gemmpipe.gemm_f16f32(M, N, K, to_dev(A, dev), to_dev(B, dev), c_ptr)
    assert gemmpipe.gemmpipe_get_device_status() == gemmpipe.OK
    host = buf.cpu().numpy()
    assert (host[:pad] == 12345.0).all() and (host[pad + M * N:] == 12345.0).all()
    assert_f16_close(host[pad:pad + M * N].reshape(M, N), oracle.gemm_f16f32(A, B))


def test_empty_shapes(dev):
    import torch
    C = torch.full((5, 9), 3.0, dtype=torch.float32, device=dev)
    A = torch.zeros((5, 0), dtype=torch.float16, device=dev)
    B = torch.zeros((0, 9), dtype=torch.float16, device=dev)
    gemmpipe.gemm_f16f32(5, 9, 0, A, B, C)           # empty sum: zeros
    assert gemmpipe.gemmpipe_get_device_status() == gemmpipe.OK
    assert (C == 0).all()
    Ci = torch.full((5, 9), 3, dtype=torch.int32, device=dev)
    gemmpipe.gemm_s8s8s32(5, 9, 0, A.to(torch.int8), B.to(torch.int8), Ci)
    assert gemmpipe.gemmpipe_get_device_status() == gemmpipe.OK
    assert (Ci == 0).all()
    gemmpipe.gemm_f16f32(0, 9, 4, None, None, None)   # nothing to do
    gemmpipe.gemm_s8s8s32(5, 0, 4, None, None, None)


def test_host_pointer_rejected(dev):
    import torch
    A = torch.zeros((8, 8), dtype=torch.float16)      # host memory
    B = torch.zeros((8, 8), dtype=torch.float16, device=dev)
    C = torch.zeros((8, 8), dtype=torch.float32, device=dev)
    with pytest.raises(gemmpipe.GemmpipeError) as ei:
        gemmpipe.gemm_f16f32(8, 8, 8, A, B, C)
    assert ei.value.status == gemmpipe.ERR_INVALID_VALUE


def test_plan_rejects_tile_counts_beyond_32_bits(dev):
    # 2^24 x 2^24 is 2^34 tiles of 128 x 128: the kernels number tiles in
    # 32 bits, and such a C (2^50 bytes) cannot be device memory.  Only the
    # plan is asked for: nothing is launched.
    for dtype in (0, 1):
        with pytest.raises(gemmpipe.GemmpipeError) as ei:
            gemmpipe.gemmpipe_plan(dtype, 1 << 24, 1 << 24, 64)
        assert ei.value.status == gemmpipe.ERR_INVALID_VALUE
    assert gemmpipe.gemmpipe_plan(1, 1 << 15, 1 << 15, 64)["tiles"] == (1 << 14)


# ----------------------------------------------------------- INT8 exactness

@pytest.mark.parametrize("forced", [-1, 0], ids=["widened_in_workspace", "widened_in_kernel_if_aligned"])
@pytest.mark.parametrize("N", [264, 272])
@pytest.mark.parametrize("K", [1024, 1025, 2048, 3000, 4096, 4112])
def test_s8_chunk_exactness_extremes(dev, K, N, forced):
    # Products of +-127/-128 make every chunk partial an odd or large integer
    # near 2^24 in magnitude: any bit the fp32 accumulation dropped shows.
    # N = 264 is not a multiple of 16 (workspace path); N = 272 with K a
    # multiple of 16 takes the in-kernel widening path.
    M = 130
    rng = np.random.default_rng(K)
    A = rng.choice(np.array([-128, 127, -127], dtype=np.int8), size=(M, K))
    B = rng.choice(np.array([-128, 127, 127], dtype=np.int8), size=(K, N))
    expect_convert = (N % 16 == 0 and K % 16 == 0 and forced == 0)
    gemmpipe.gemmpipe_set_plan_override(forced, 0, 0)
    try:
        assert gemmpipe.gemmpipe_plan(0, M, N, K)["operand_copy"] == (0 if expect_convert else 1)
    finally:
        gemmpipe.gemmpipe_set_plan_override(-1, 0, 0)
    A[0, :] = 127
    B[:, 0] = 127          # C[0,0] = 16129 K: odd partials just below 2^24
    A[1, :] = -128
    B[:, 1] = -128         # C[1,1] = 16384 K: the chunk bound itself
    gemmpipe.gemmpipe_set_plan_override(forced, 0, 0)
    try:
        got = run_s8(A, B, dev)
    finally:
        gemmpipe.gemmpipe_set_plan_override(-1, 0, 0)
    want = oracle.gemm_s8s8s32(A, B)
    assert np.array_equal(got, want)
    assert got[0, 0] == 16129 * K and got[1, 1] == 16384 * K


# ------------------------------------------------------------ the workloads

def test_workload_int8_512(dev):
    _, _, M, N, K, A, B = inputs.workload_operands(0)
    assert np.array_equal(run_s8(A, B, dev), oracle.gemm_s8s8s32(A, B))


def test_workload_fp16_1024(dev):
    _, _, M, N, K, A, B = inputs.workload_operands(1)
    assert_f16_close(run_f16(A, B, dev), oracle.gemm_f16f32(A, B), "fp16 1024^3")


def test_workload_int8_4096(dev, full_size):
    # Every element of the headline workload, bit for bit.
    A, B, want = full_size(2)
    K = A.shape[1]
    got = run_s8(A, B, dev)
    assert np.array_equal(got, want)
    # Any-size property: int8 products are bounded by 2^14 K.
    assert np.abs(got.astype(np.int64)).max() <= 16384 * K


def test_workload_fp16_skinny(dev, full_size):
    # Every element of the 16384 x 128 C (128 whole tiles, A streamed once).
    A, B, want = full_size(3)
    assert_f16_close(run_f16(A, B, dev), want, "skinny")


@pytest.mark.parametrize("forced", [-1, 1], ids=["padded_tma", "bounded_loads"])
def test_workload_fp16_ragged(dev, full_size, forced):
    # Every element of the 4093 x 3001 C: partial last tiles in M, N and K,
    # most tiles split into k-block ranges over the persistent grid.
    A, B, want = full_size(4)
    M, K = A.shape
    N = B.shape[1]
    gemmpipe.gemmpipe_set_plan_override(forced, 0, 0)
    try:
        plan = gemmpipe.gemmpipe_plan(1, M, N, K)
        got = run_f16(A, B, dev)
    finally:
        gemmpipe.gemmpipe_set_plan_override(-1, 0, 0)
    assert plan["k_blocks"] == (K + 63) // 64
    assert_f16_close(got, want, "ragged")


# --------------------------------------------------------- bounded waits

def test_stall_times_out_and_context_survives(dev):
    import torch
    M, N, K = 256, 256, 1024
    A, B = inputs.make_operands("f16", M, N, K, seed=13)
    Ad, Bd = to_dev(A, dev), to_dev(B, dev)
    C = torch.zeros((M, N), dtype=torch.float32, device=dev)
    gemmpipe.gemmpipe_test_inject_stall(3, 200)
    gemmpipe.gemm_f16f32(M, N, K, Ad, Bd, C)
    assert gemmpipe.gemmpipe_get_device_status() == gemmpipe.ERR_TIMEOUT
    # The context is still usable and the hook was one-shot.
    gemmpipe.gemm_f16f32(M, N, K, Ad, Bd, C)
    assert gemmpipe.gemmpipe_get_device_status() == gemmpipe.OK
    assert_f16_close(C.cpu().numpy(), oracle.gemm_f16f32(A, B))


def test_stall_times_out_bounded_load_producer(dev):
    import torch
    M, N, K = 129, 200, 333   # odd pitches; the bounded-load producer is forced
    A, B = inputs.make_operands("f16", M, N, K, seed=14)
    Ad, Bd = to_dev(A, dev), to_dev(B, dev)
    C = torch.zeros((M, N), dtype=torch.float32, device=dev)
    gemmpipe.gemmpipe_set_plan_override(1, 0, 0)
    try:
        assert gemmpipe.gemmpipe_plan(1, M, N, K, Ad, Bd, C)["producer"] == 1
        gemmpipe.gemmpipe_test_inject_stall(1, 200)
        gemmpipe.gemm_f16f32(M, N, K, Ad, Bd, C)
        assert gemmpipe.gemmpipe_get_device_status() == gemmpipe.ERR_TIMEOUT
        gemmpipe.gemm_f16f32(M, N, K, Ad, Bd, C)
        assert gemmpipe.gemmpipe_get_device_status() == gemmpipe.OK
    finally:
        gemmpipe.gemmpipe_set_plan_override(-1, 0, 0)
    assert_f16_close(C.cpu().numpy(), oracle.gemm_f16f32(A, B))


def test_kernel_timing_and_launch_count(dev):
    import torch
    M = N = K = 512
    A, B = inputs.make_operands("s8", M, N, K, seed=15)
    Ad, Bd = to_dev(A, dev), to_dev(B, dev)
    C = torch.zeros((M, N), dtype=torch.int32, device=dev)
    gemmpipe.gemmpipe_timing_read()
    for forced, aux in ((0, 0), (-1, 3)):   # in-kernel widening: 1 kernel; workspace path: 2 per call
        gemmpipe.gemmpipe_set_plan_override(forced, 0, 0)
        n0 = gemmpipe.gemmpipe_launch_count()
        gemmpipe.gemmpipe_timing_enable(True)
        try:
            for _ in range(3):
                gemmpipe.gemm_s8s8s32(M, N, K, Ad, Bd, C)
            gms, gn, ams, an = gemmpipe.gemmpipe_timing_read()
        finally:
            gemmpipe.gemmpipe_timing_enable(False)
            gemmpipe.gemmpipe_set_plan_override(-1, 0, 0)
        assert gemmpipe.gemmpipe_get_device_status() == gemmpipe.OK
        assert gn == 3 and an == aux and gms > 0 and (ams > 0) == (aux > 0)
        assert gemmpipe.gemmpipe_launch_count() - n0 == 3 + aux
        assert np.array_equal(C.cpu().numpy(), oracle.gemm_s8s8s32(A, B))


def test_copy_kernel(dev):
    import torch
    src = torch.arange(1 << 20, dtype=torch.int32, device=dev)
    dst = torch.zeros_like(src)
    gemmpipe.gemmpipe_copy(dst, src, src.numel() * 4)
    assert gemmpipe.gemmpipe_get_device_status() == gemmpipe.OK
    assert torch.equal(src, dst)
    odd = torch.zeros(1001, dtype=torch.uint8, device=dev)
    gemmpipe.gemmpipe_copy(odd.data_ptr() + 1, src.data_ptr() + 3, 999)
    assert gemmpipe.gemmpipe_get_device_status() == gemmpipe.OK
    assert torch.equal(odd[1:1000].cpu(), src.cpu().view(torch.uint8)[3:1002])


# ------------------------------------------------ stream-K (split tiles)

@pytest.mark.parametrize("dtype", ["f16", "s8"])
@pytest.mark.parametrize("wide", [True, False], ids=["bn256", "bn128"])
@pytest.mark.parametrize("n_extra", [0, 8], ids=["n16", "n8"])
def test_tail_wave_split(dev, dtype, wide, n_extra):
    # Tile counts a little above one wave of the persistent grid: the last
    # two waves' tiles are split into equal k-block ranges over all units.
    # Wide shapes run on CTA pairs (256-row tiles), N <= 128 on single CTAs.
    if wide:
        N, K, n_tiles = 496 + n_extra, 144, 2
    else:
        N, K, n_tiles = 112 + n_extra, 208, 1
    probe = gemmpipe.gemmpipe_plan(0 if dtype == "s8" else 1, 1 << 20, N, K)  # more tiles than slots
    units = probe["grid"] // (2 if probe["cta_pair"] else 1)
    tile_m = probe["BM"]
    assert probe["cta_pair"] == (1 if wide else 0)
    m_tiles = -(-(units + max(1, units // 4)) // n_tiles)
    M = m_tiles * tile_m - 5
    plan = gemmpipe.gemmpipe_plan(0 if dtype == "s8" else 1, M, N, K)
    tiles = m_tiles * n_tiles
    rem = tiles % units
    assert plan["tiles"] == tiles and plan["units"] == units
    assert 0 < rem and plan["split_tiles"] == units + rem
    A, B = inputs.make_operands(dtype, M, N, K, seed=500 + M)
    if dtype == "s8":
        assert np.array_equal(run_s8(A, B, dev), oracle.gemm_s8s8s32(A, B))
    else:
        assert_f16_close(run_f16(A, B, dev), oracle.gemm_f16f32(A, B))


# Fewer tiles than the grid holds: every tile's k-blocks are spread over
# several units (one tile over 128 units in the last case; the INT8 ranges
# straddle the 1024-k accumulation chunks).
SPLIT_SHAPES = [(256, 128, 8192), (100, 100, 65536), (512, 512, 4096), (300, 260, 5000), (129, 1000, 3000),
                (1000, 40, 20000)]


@pytest.mark.parametrize("dtype", ["f16", "s8"])
@pytest.mark.parametrize("M,N,K", SPLIT_SHAPES)
def test_split_small_tile_counts(dev, dtype, M, N, K):
    plan = gemmpipe.gemmpipe_plan(0 if dtype == "s8" else 1, M, N, K)
    assert plan["split_tiles"] == plan["tiles"] and plan["units"] > plan["tiles"]
    assert plan["units"] <= -(-plan["tiles"] * plan["k_blocks"] // 8)
    A, B = inputs.make_operands(dtype, M, N, K, seed=900 + M + N + K)
    if dtype == "s8":
        assert np.array_equal(run_s8(A, B, dev), oracle.gemm_s8s8s32(A, B))
    else:
        assert_f16_close(run_f16(A, B, dev), oracle.gemm_f16f32(A, B))


@pytest.mark.parametrize("pair", [1, 0], ids=["pair", "single"])
def test_split_results_repeat_bit_for_bit(dev, pair):
    # The parts of a split tile are added in a fixed order.
    import torch
    M, N, K = 1000, 700, 3000
    A, B = inputs.make_operands("f16", M, N, K, seed=31)
    Ad, Bd = to_dev(A, dev), to_dev(B, dev)
    gemmpipe.gemmpipe_set_plan_override(-1, 0, 0, pair)
    try:
        plan = gemmpipe.gemmpipe_plan(1, M, N, K, Ad, Bd)
        assert plan["split_tiles"] > 0 and plan["cta_pair"] == pair
        outs = []
        for _ in range(3):
            C = torch.empty((M, N), dtype=torch.float32, device=dev)
            gemmpipe.gemm_f16f32(M, N, K, Ad, Bd, C)
            assert gemmpipe.gemmpipe_get_device_status() == gemmpipe.OK
            outs.append(C)
    finally:
        gemmpipe.gemmpipe_set_plan_override(-1, 0, 0)
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    assert_f16_close(outs[0].cpu().numpy(), oracle.gemm_f16f32(A, B))


def test_memory_bound_half_full_grid_keeps_whole_tiles(dev):
    # 100 tiles of 128 x 128 over 152 SMs, 113 flops per byte (memory-bound):
    # whole tiles by default; the split override still splits, same result.
    M, N, K = 12800, 128, 2048
    A, B = inputs.make_operands("f16", M, N, K, seed=43)
    want = oracle.gemm_f16f32(A, B)
    plan = gemmpipe.gemmpipe_plan(1, M, N, K)
    assert plan["tiles"] == 100 and plan["split_tiles"] == 0 and plan["units"] == 100
    assert_f16_close(run_f16(A, B, dev), want)
    gemmpipe.gemmpipe_set_plan_override(-1, 0, 0, -1, 1)
    try:
        forced = gemmpipe.gemmpipe_plan(1, M, N, K)
        assert forced["split_tiles"] == 100 and forced["units"] > 100
        got = run_f16(A, B, dev)
    finally:
        gemmpipe.gemmpipe_set_plan_override(-1, 0, 0)
    assert_f16_close(got, want)


def test_split_plans_share_the_stream_workspace(dev):
    # Split launches with different grids and tile widths take turns on one
    # stream: the flags sit in a fixed region, never where another plan
    # leaves its (small-integer INT8) partial sums.
    import torch
    shapes = [("s8", 1000, 700, 3000), ("f16", 256, 128, 8192), ("s8", 300, 100, 9000), ("f16", 1000, 40, 20000)]
    ops = []
    for dt, M, N, K in shapes:
        A, B = inputs.make_operands(dt, M, N, K, seed=41 + M)
        want = oracle.gemm_s8s8s32(A, B) if dt == "s8" else oracle.gemm_f16f32(A, B)
        assert gemmpipe.gemmpipe_plan(0 if dt == "s8" else 1, M, N, K)["split_tiles"] > 0
        C = torch.empty((M, N), dtype=torch.int32 if dt == "s8" else torch.float32, device=dev)
        ops.append((dt, M, N, K, to_dev(A, dev), to_dev(B, dev), C, want))
    for _ in range(8):
        for dt, M, N, K, Ad, Bd, C, want in ops:
            C.fill_(-1)
            (gemmpipe.gemm_s8s8s32 if dt == "s8" else gemmpipe.gemm_f16f32)(M, N, K, Ad, Bd, C)
            assert gemmpipe.gemmpipe_get_device_status() == gemmpipe.OK
            if dt == "s8":
                assert np.array_equal(C.cpu().numpy(), want)
            else:
                assert_f16_close(C.cpu().numpy(), want)


@pytest.mark.parametrize("dtype", ["f16", "s8"])
def test_split_stall_times_out(dev, dtype):
    # CTA 0 stalls on its first k-block: its own waits and the wait of the
    # unit that adds its partial sums run out of time; nothing hangs, and
    # the next call is correct.
    import torch
    M, N, K = 256, 128, 8192
    A, B = inputs.make_operands(dtype, M, N, K, seed=37)
    Ad, Bd = to_dev(A, dev), to_dev(B, dev)
    plan = gemmpipe.gemmpipe_plan(0 if dtype == "s8" else 1, M, N, K, Ad, Bd)
    assert plan["split_tiles"] == plan["tiles"]
    out_t = torch.int32 if dtype == "s8" else torch.float32
    C = torch.zeros((M, N), dtype=out_t, device=dev)
    call = gemmpipe.gemm_s8s8s32 if dtype == "s8" else gemmpipe.gemm_f16f32
    gemmpipe.gemmpipe_test_inject_stall(0, 200)
    call(M, N, K, Ad, Bd, C)
    assert gemmpipe.gemmpipe_get_device_status() == gemmpipe.ERR_TIMEOUT
    call(M, N, K, Ad, Bd, C)
    assert gemmpipe.gemmpipe_get_device_status() == gemmpipe.OK
    if dtype == "s8":
        assert np.array_equal(C.cpu().numpy(), oracle.gemm_s8s8s32(A, B))
    else:
        assert_f16_close(C.cpu().numpy(), oracle.gemm_f16f32(A, B))


@pytest.mark.parametrize("dtype", ["f16", "s8"])
@pytest.mark.parametrize("M,N,K", [(256, 256, 64), (257, 264, 200), (1000, 776, 1032), (4093, 3000, 136),
                                   (512, 136, 4096), (200, 1024, 64)])
def test_cta_pair_matches_single_cta(dev, dtype, M, N, K):
    # CTA pairs (cta_group::2, 256-row tiles; asked for, since the planner
    # takes single 128 x 128 tiles for small problems) and the single-CTA
    # 128 x 256 variant must both match the oracle.
    A, B = inputs.make_operands(dtype, M, N, K, seed=700 + M + N + K)
    want = oracle.gemm_s8s8s32(A, B) if dtype == "s8" else oracle.gemm_f16f32(A, B)
    run = run_s8 if dtype == "s8" else run_f16
    check = (lambda g: np.testing.assert_array_equal(g, want)) if dtype == "s8" else \
        (lambda g: assert_f16_close(g, want))
    gemmpipe.gemmpipe_set_plan_override(-1, 0, 0, 1)
    try:
        plan = gemmpipe.gemmpipe_plan(0 if dtype == "s8" else 1, M, N, K)
        assert plan["cta_pair"] == 1 and plan["BM"] == 256
        check(run(A, B, dev))
    finally:
        gemmpipe.gemmpipe_set_plan_override(-1, 0, 0)
    gemmpipe.gemmpipe_set_plan_override(-1, 256, 0, 0)
    try:
        plan = gemmpipe.gemmpipe_plan(0 if dtype == "s8" else 1, M, N, K)
        assert plan["cta_pair"] == 0 and plan["BM"] == 128
        got = run(A, B, dev)
    finally:
        gemmpipe.gemmpipe_set_plan_override(-1, 0, 0)
    check(got)


def test_cta_pair_stall_times_out(dev):
    import torch
    M, N, K = 512, 512, 1024
    A, B = inputs.make_operands("f16", M, N, K, seed=17)
    Ad, Bd = to_dev(A, dev), to_dev(B, dev)
    C = torch.zeros((M, N), dtype=torch.float32, device=dev)
    gemmpipe.gemmpipe_set_plan_override(-1, 0, 0, 1)
    try:
        assert gemmpipe.gemmpipe_plan(1, M, N, K, Ad, Bd, C)["cta_pair"] == 1
        gemmpipe.gemmpipe_test_inject_stall(2, 200)
        gemmpipe.gemm_f16f32(M, N, K, Ad, Bd, C)
        assert gemmpipe.gemmpipe_get_device_status() == gemmpipe.ERR_TIMEOUT
        gemmpipe.gemm_f16f32(M, N, K, Ad, Bd, C)
        assert gemmpipe.gemmpipe_get_device_status() == gemmpipe.OK
    finally:
        gemmpipe.gemmpipe_set_plan_override(-1, 0, 0)
    assert_f16_close(C.cpu().numpy(), oracle.gemm_f16f32(A, B))


def test_workload_fp16_4096(dev, full_size):
    # The fp16 half of the headline metric: 4096^3, uniform [-1, 1], every
    # element.  The 256 pair tiles leave a partial last wave, so the last
    # two waves are split into k-block ranges.
    A, B, want = full_size("fp16_4096")
    M, K = A.shape
    N = B.shape[1]
    plan = gemmpipe.gemmpipe_plan(1, M, N, K)
    assert plan["tiles"] % plan["units"] == 0 or plan["split_tiles"] > 0
    assert_f16_close(run_f16(A, B, dev), want, "fp16 4096^3")


@pytest.mark.parametrize("M,N,K", [(128, 128, 64), (300, 272, 1040), (129, 512, 2048), (1000, 256, 4096),
                                   (64, 16, 16), (513, 144, 3088)])
def test_s8_in_kernel_and_workspace_widening_agree(dev, M, N, K):
    A, B = inputs.make_operands("s8", M, N, K, seed=600 + M + N + K)
    want = oracle.gemm_s8s8s32(A, B)
    assert gemmpipe.gemmpipe_plan(0, M, N, K)["operand_copy"] == 1
    assert np.array_equal(run_s8(A, B, dev), want)
    gemmpipe.gemmpipe_set_plan_override(0, 0, 0)
    try:
        assert gemmpipe.gemmpipe_plan(0, M, N, K)["operand_copy"] == 0
        got = run_s8(A, B, dev)
    finally:
        gemmpipe.gemmpipe_set_plan_override(-1, 0, 0)
    assert np.array_equal(got, want)


def test_s8_stall_times_out_in_converter_variant(dev):
    import torch
    M, N, K = 256, 256, 2048
    A, B = inputs.make_operands("s8", M, N, K, seed=16)
    Ad, Bd = to_dev(A, dev), to_dev(B, dev)
    C = torch.zeros((M, N), dtype=torch.int32, device=dev)
    gemmpipe.gemmpipe_set_plan_override(0, 0, 0)
    try:
        assert gemmpipe.gemmpipe_plan(0, M, N, K, Ad, Bd, C)["operand_copy"] == 0
        gemmpipe.gemmpipe_test_inject_stall(5, 200)
        gemmpipe.gemm_s8s8s32(M, N, K, Ad, Bd, C)
        assert gemmpipe.gemmpipe_get_device_status() == gemmpipe.ERR_TIMEOUT
        gemmpipe.gemm_s8s8s32(M, N, K, Ad, Bd, C)
        assert gemmpipe.gemmpipe_get_device_status() == gemmpipe.OK
    finally:
        gemmpipe.gemmpipe_set_plan_override(-1, 0, 0)
    assert np.array_equal(C.cpu().numpy(), oracle.gemm_s8s8s32(A, B))


@pytest.mark.parametrize("stages", [1, 2, 3, 4, 5, 6])
def test_ring_depths_of_cta_pair(dev, stages):
    # S = 1: the producer waits for the MMAs to release the only stage
    # before every load (load, wait, compute -- no overlap); S = 2: the
    # double buffer; deeper rings overlap more k-blocks.  Results must not
    # depend on the depth.
    M, N, K = 520, 776, 1000
    A, B = inputs.make_operands("f16", M, N, K, seed=800 + stages)
    gemmpipe.gemmpipe_set_plan_override(0, 256, stages, 1)
    try:
        plan = gemmpipe.gemmpipe_plan(1, M, N, K)
        assert plan["stages"] == stages and plan["cta_pair"] == 1
        got = run_f16(A, B, dev)
    finally:
        gemmpipe.gemmpipe_set_plan_override(-1, 0, 0)
    assert_f16_close(got, oracle.gemm_f16f32(A, B), f"S={stages}")


# -------------------------------------- warp-level integer MMA (comparison)

@pytest.mark.parametrize("stages", [4, 2], ids=["S4", "S2"])
@pytest.mark.parametrize("M,N,K", [(128, 128, 64), (300, 270, 1040), (1000, 777, 4096), (17, 33, 16),
                                   (513, 129, 208), (2048, 2048, 2048)])
def test_imma_comparison_path_is_bit_exact(dev, M, N, K, stages):
    # The pages' design (mma.sync m16n8k32 s8 with a cp.async ring; S = 2 is
    # their double buffer) on A and a transposed copy of B: bit-exact like
    # the tcgen05 paths.
    A, B = inputs.make_operands("s8", M, N, K, seed=1100 + M + N + K)
    gemmpipe.gemmpipe_set_plan_override(2, 0, stages if stages == 2 else 0)
    try:
        plan = gemmpipe.gemmpipe_plan(0, M, N, K)
        assert plan["producer"] == 2 and plan["operand_copy"] == 3 and plan["stages"] == stages
        assert plan["workspace_bytes"] == N * (-(-K // 16) * 16)
        got = run_s8(A, B, dev)
    finally:
        gemmpipe.gemmpipe_set_plan_override(-1, 0, 0)
    np.testing.assert_array_equal(got, oracle.gemm_s8s8s32(A, B))


def test_imma_comparison_path_extremes_and_fallback(dev):
    M, N, K = 200, 136, 4096
    A = np.full((M, K), -128, dtype=np.int8)
    B = np.full((K, N), -128, dtype=np.int8)
    gemmpipe.gemmpipe_set_plan_override(2, 0, 0)
    try:
        got = run_s8(A, B, dev)
        # K not a multiple of 16: the comparison path does not apply and the
        # call takes the default widening path.
        plan = gemmpipe.gemmpipe_plan(0, 64, 64, 100)
        assert plan["producer"] == 0 and plan["operand_copy"] == 1
        A2, B2 = inputs.make_operands("s8", 64, 64, 100, seed=5)
        got2 = run_s8(A2, B2, dev)
    finally:
        gemmpipe.gemmpipe_set_plan_override(-1, 0, 0)
    assert (got == 16384 * K).all()
    np.testing.assert_array_equal(got2, oracle.gemm_s8s8s32(A2, B2))


# ------------------------------------------- int32 wrap and 64-bit indexing

@pytest.mark.parametrize("path", ["tcgen05", "imma"])
def test_s8_sums_wrap_modulo_2_32(dev, path):
    # K = 2^17 + 64 with extreme operands: exact sums up to 16384 * K exceed
    # int32 and wrap modulo 2^32, as integer hardware does.  One 64 x 64
    # tile over 2049 k-blocks: the tcgen05 path splits it over the whole
    # grid (a finisher adding up to ~150 partial sums).
    M, N, K = 64, 64, (1 << 17) + 64
    rng = np.random.default_rng(11)
    A = np.where(rng.random((M, K)) < 0.9, -128, 127).astype(np.int8)
    B = np.where(rng.random((K, N)) < 0.9, -128, 127).astype(np.int8)
    A[0, :] = -128
    B[:, 0] = -128
    want = oracle.gemm_s8s8s32(A, B, allow_overflow=True)
    assert want[0, 0] == np.int32(np.int64(16384 * K) - (1 << 32))
    gemmpipe.gemmpipe_set_plan_override(2 if path == "imma" else -1, 0, 0)
    try:
        plan = gemmpipe.gemmpipe_plan(0, M, N, K)
        if path == "tcgen05":
            assert plan["split_tiles"] == 1 and plan["units"] > 100
        got = run_s8(A, B, dev)
    finally:
        gemmpipe.gemmpipe_set_plan_override(-1, 0, 0)
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("dtype", ["f16", "s8"])
def test_c_beyond_2_31_elements(dev, dtype):
    # C of 600000 x 4096 = 2.46e9 elements (9.8 GB): row offsets past 2^31
    # elements on every path (TMA store coordinates, partial sums, widening).
    import torch
    M, N, K = 600000, 4096, 64
    A, B = inputs.make_operands(dtype, M, N, K, seed=77)
    Ad, Bd = to_dev(A, dev), to_dev(B, dev)
    C = torch.empty((M, N), dtype=torch.int32 if dtype == "s8" else torch.float32, device=dev)
    C[-1].fill_(-7)
    (gemmpipe.gemm_s8s8s32 if dtype == "s8" else gemmpipe.gemm_f16f32)(M, N, K, Ad, Bd, C)
    assert gemmpipe.gemmpipe_get_device_status() == gemmpipe.OK
    rows = sample_rows(M)
    idx = torch.from_numpy(rows).to(dev)
    got = C.index_select(0, idx).cpu().numpy()
    del C
    if dtype == "s8":
        np.testing.assert_array_equal(got, oracle.gemm_s8s8s32(A, B, rows=rows))
    else:
        assert_f16_close(got, oracle.gemm_f16f32(A, B, rows=rows))


# ------------------------------------------------------ extreme aspect ratios

@pytest.mark.parametrize("dtype", ["f16", "s8"])
@pytest.mark.parametrize("M,N,K", [(1, 65536, 64),      # one row, 256+ column tiles, split tail
                                   (65536, 16, 32),     # tall and thin: 512 row tiles of a 128-wide variant
                                   (2, 3, 200000),      # a single tile split over the whole grid
                                   (128, 128, 131071)])  # the largest K whose int8 sums cannot wrap
def test_extreme_aspect_ratios(dev, dtype, M, N, K):
    A, B = inputs.make_operands(dtype, M, N, K, seed=2100 + M + N + K)
    if dtype == "s8":
        assert np.array_equal(run_s8(A, B, dev), oracle.gemm_s8s8s32(A, B))
    else:
        assert_f16_close(run_f16(A, B, dev), oracle.gemm_f16f32(A, B), f"{M}x{N}x{K}")


# ------------------------------------------------- 512-wide CTA-pair tiles

@pytest.mark.parametrize("split", [-1, 0, 1], ids=["auto", "whole", "split"])
@pytest.mark.parametrize("M,N,K", [(256, 512, 64),        # one tile, one k-block
                                   (520, 1030, 1000),     # ragged M, N, K; several tiles
                                   (300, 600, 4107),      # two column tiles, the second mostly empty
                                   (1024, 2048, 2048),    # more tiles than one pass of each pair
                                   (2000, 3000, 257)])    # ragged everything, 5 k-blocks
def test_bn512_pair_tiles(dev, M, N, K, split):
    # 256 x 512 tiles: two N = 256 MMAs per k-step into one 512-column
    # accumulator, drained in two passes; whole tiles and stream-K splits.
    A, B = inputs.make_operands("f16", M, N, K, seed=900 + M + N + K)
    gemmpipe.gemmpipe_set_plan_override(-1, 512, 0, 1, split)
    try:
        plan = gemmpipe.gemmpipe_plan(1, M, N, K)
        assert plan["BN"] == 512 and plan["cta_pair"] == 1 and plan["stages"] == 4
        if split == 0:
            assert plan["split_tiles"] == 0
        got = run_f16(A, B, dev)
    finally:
        gemmpipe.gemmpipe_set_plan_override(-1, 0, 0, -1, -1)
    assert_f16_close(got, oracle.gemm_f16f32(A, B), f"{M}x{N}x{K} split={split}")


def test_bn512_falls_back_for_int8_and_narrow_shapes(dev):
    # No 512-wide INT8 variant (its epilogue keeps int32 sums per thread)
    # and no pair for a single row tile: the override then takes 256.
    gemmpipe.gemmpipe_set_plan_override(-1, 512, 0, -1, -1)
    try:
        assert gemmpipe.gemmpipe_plan(0, 1024, 1024, 1024)["BN"] == 256
        p = gemmpipe.gemmpipe_plan(1, 100, 1024, 256)
        assert p["BN"] == 256 and p["cta_pair"] == 0
        A, B = inputs.make_operands("s8", 300, 700, 300, seed=931)
        np.testing.assert_array_equal(run_s8(A, B, dev), oracle.gemm_s8s8s32(A, B))
    finally:
        gemmpipe.gemmpipe_set_plan_override(-1, 0, 0, -1, -1)


def test_bn512_stall_times_out(dev):
    import torch
    M, N, K = 512, 1024, 1024
    A, B = inputs.make_operands("f16", M, N, K, seed=933)
    Ad, Bd = to_dev(A, dev), to_dev(B, dev)
    C = torch.zeros((M, N), dtype=torch.float32, device=dev)
    gemmpipe.gemmpipe_set_plan_override(-1, 512, 0, 1, -1)
    try:
        assert gemmpipe.gemmpipe_plan(1, M, N, K, Ad, Bd, C)["BN"] == 512
        gemmpipe.gemmpipe_test_inject_stall(2, 200)
        gemmpipe.gemm_f16f32(M, N, K, Ad, Bd, C)
        assert gemmpipe.gemmpipe_get_device_status() == gemmpipe.ERR_TIMEOUT
        gemmpipe.gemm_f16f32(M, N, K, Ad, Bd, C)
        assert gemmpipe.gemmpipe_get_device_status() == gemmpipe.OK
    finally:
        gemmpipe.gemmpipe_set_plan_override(-1, 0, 0, -1, -1)
    assert_f16_close(C.cpu().numpy(), oracle.gemm_f16f32(A, B))


@pytest.mark.parametrize("dtype", ["f16", "s8"])
@pytest.mark.parametrize("M,N,K,small", [(512, 512, 512, True), (1024, 1024, 1024, True), (300, 2000, 700, True),
                                         (1280, 1280, 256, False), (2048, 2048, 128, False)])
def test_small_problems_take_single_cta_tiles(dev, dtype, M, N, K, small):
    # At most a quarter of the SM pairs' worth of 256 x 256 tiles: single
    # CTAs on 128 x 128 tiles (more SMs, a quarter of the epilogue each);
    # larger problems keep the pairs.  Results match the oracle either way.
    plan = gemmpipe.gemmpipe_plan(0 if dtype == "s8" else 1, M, N, K)
    if small:
        assert plan["cta_pair"] == 0 and plan["BM"] == 128 and plan["BN"] == 128
    else:
        assert plan["cta_pair"] == 1 and plan["BM"] == 256
    A, B = inputs.make_operands(dtype, M, N, K, seed=950 + M + N + K)
    if dtype == "s8":
        np.testing.assert_array_equal(run_s8(A, B, dev), oracle.gemm_s8s8s32(A, B))
    else:
        assert_f16_close(run_f16(A, B, dev), oracle.gemm_f16f32(A, B))


@pytest.mark.parametrize("dtype", ["f16", "s8"])
@pytest.mark.parametrize("M,N,K,split", [(1024, 1024, 2048, False), (1024, 1024, 3072, True),
                                         (1000, 1000, 4100, True), (1024, 896, 4096, True)])
def test_single_cta_tiles_split_long_k(dev, dtype, M, N, K, split):
    # Fewer single-CTA tiles than SMs: the planner spreads the k-blocks over
    # all SMs when that takes at least 1536 k values off each unit (whole
    # tiles otherwise).  Results match the oracle either way.
    plan = gemmpipe.gemmpipe_plan(0 if dtype == "s8" else 1, M, N, K)
    assert plan["cta_pair"] == 0 and plan["BN"] == 128
    if split:
        assert plan["split_tiles"] == plan["tiles"] and plan["units"] > plan["tiles"]
    else:
        assert plan["split_tiles"] == 0 and plan["units"] == plan["tiles"]
    A, B = inputs.make_operands(dtype, M, N, K, seed=970 + M + K)
    if dtype == "s8":
        np.testing.assert_array_equal(run_s8(A, B, dev), oracle.gemm_s8s8s32(A, B))
    else:
        assert_f16_close(run_f16(A, B, dev), oracle.gemm_f16f32(A, B))


# ------------------------------------------- quads: two CTA pairs sharing A

@pytest.mark.parametrize("split", [-1, 0, 1], ids=["auto", "whole", "split"])
@pytest.mark.parametrize("M,N,K", [(256, 512, 64),        # one tile, one k-block
                                   (520, 1030, 1000),     # ragged M, N, K
                                   (300, 300, 4107),      # the second pair's columns mostly past N
                                   (512, 256, 640),       # the second pair's columns all past N
                                   (1024, 2048, 2048),    # several tiles per quad
                                   (2000, 3000, 257)])    # ragged everything, 5 k-blocks
@pytest.mark.parametrize("dtype", ["f16", "s8"])
def test_quad_tiles(dev, dtype, M, N, K, split):
    # Quads (cluster of four CTAs): two CTA pairs compute a 256 x 512 tile
    # over the same 256 rows; each CTA loads half of its A rows of a k-block
    # and multicasts it to its counterpart in the other pair.
    A, B = inputs.make_operands(dtype, M, N, K, seed=970 + M + N + K)
    gemmpipe.gemmpipe_set_plan_override(-1, 0, 0, 2, split)
    try:
        plan = gemmpipe.gemmpipe_plan(0 if dtype == "s8" else 1, M, N, K)
        assert plan["cta_pair"] == 2 and plan["BM"] == 256 and plan["BN"] == 512
        assert plan["grid"] == 4 * plan["units"]
        if split == 0:
            assert plan["split_tiles"] == 0
        got = run_s8(A, B, dev) if dtype == "s8" else run_f16(A, B, dev)
    finally:
        gemmpipe.gemmpipe_set_plan_override(-1, 0, 0, -1, -1)
    if dtype == "s8":
        np.testing.assert_array_equal(got, oracle.gemm_s8s8s32(A, B))
    else:
        assert_f16_close(got, oracle.gemm_f16f32(A, B), f"quad {M}x{N}x{K} split={split}")


@pytest.mark.parametrize("dtype", ["f16", "s8"])
def test_quad_stall_times_out(dev, dtype):
    import torch
    M, N, K = 512, 1024, 2048
    A, B = inputs.make_operands(dtype, M, N, K, seed=977)
    Ad, Bd = to_dev(A, dev), to_dev(B, dev)
    C = torch.zeros((M, N), dtype=torch.int32 if dtype == "s8" else torch.float32, device=dev)
    call = gemmpipe.gemm_s8s8s32 if dtype == "s8" else gemmpipe.gemm_f16f32
    gemmpipe.gemmpipe_set_plan_override(-1, 0, 0, 2, -1)
    try:
        assert gemmpipe.gemmpipe_plan(0 if dtype == "s8" else 1, M, N, K, Ad, Bd, C)["cta_pair"] == 2
        gemmpipe.gemmpipe_test_inject_stall(2, 200)
        call(M, N, K, Ad, Bd, C)
        assert gemmpipe.gemmpipe_get_device_status() == gemmpipe.ERR_TIMEOUT
        call(M, N, K, Ad, Bd, C)
        assert gemmpipe.gemmpipe_get_device_status() == gemmpipe.OK
    finally:
        gemmpipe.gemmpipe_set_plan_override(-1, 0, 0, -1, -1)
    want = oracle.gemm_s8s8s32(A, B) if dtype == "s8" else oracle.gemm_f16f32(A, B)
    if dtype == "s8":
        np.testing.assert_array_equal(C.cpu().numpy(), want)
    else:
        assert_f16_close(C.cpu().numpy(), want)


@pytest.mark.parametrize("dtype", ["f16", "s8"])
@pytest.mark.parametrize("N,quad", [(3001, True), (3004, False), (1030, True), (1032, False)])
def test_quads_by_default_for_c_rows_off_16_bytes(dev, dtype, N, quad):
    # C rows off 16-byte boundaries take 4-byte stores; there the planner
    # takes quads by default, elsewhere CTA pairs.
    M, K = 1500, 700
    plan = gemmpipe.gemmpipe_plan(0 if dtype == "s8" else 1, M, N, K)
    assert plan["cta_pair"] == (2 if quad else 1)
    A, B = inputs.make_operands(dtype, M, N, K, seed=990 + N)
    if dtype == "s8":
        np.testing.assert_array_equal(run_s8(A, B, dev), oracle.gemm_s8s8s32(A, B))
    else:
        assert_f16_close(run_f16(A, B, dev), oracle.gemm_f16f32(A, B))


@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (1000, 128, 4107), (16384, 128, 2048), (300, 100, 129),
                                   (520, 64, 1000)])
def test_bk128_single_cta_tiles(dev, M, N, K):
    # Single CTAs on 128 x 128 tiles with 128 k per stage (A as two 64-k
    # sub-tiles per stage): one k-block, ragged K tails, N below 128.
    A, B = inputs.make_operands("f16", M, N, K, seed=1100 + M + N + K)
    gemmpipe.gemmpipe_set_plan_override(-1, 128, 0, 0, -1)
    gemmpipe.gemmpipe_set_plan_bk(128)
    try:
        plan = gemmpipe.gemmpipe_plan(1, M, N, K)
        assert plan["BK"] == 128 and plan["stages"] == 3 and plan["cta_pair"] == 0 and plan["BN"] == 128
        got = run_f16(A, B, dev)
    finally:
        gemmpipe.gemmpipe_set_plan_bk(0)
        gemmpipe.gemmpipe_set_plan_override(-1, 0, 0, -1, -1)
    assert_f16_close(got, oracle.gemm_f16f32(A, B), f"{M}x{N}x{K}")


def test_quad_split_rule(dev):
    # Quads split only a last wave at most half full after two full waves.
    for M, N, K in ((4093, 3001, 4107), (2000, 3001, 2000), (3000, 5001, 4000), (8191, 6001, 4096)):
        p = gemmpipe.gemmpipe_plan(1, M, N, K)
        assert p["cta_pair"] == 2
        T, G = p["tiles"], p["units"]
        want = G + T % G if (T > G and T % G and 2 * (T % G) <= G and T >= 2 * G) else 0
        assert p["split_tiles"] == want, (M, N, K, p)


# ----------------------------------------------- 128 k per stage (CTA pairs)

@pytest.mark.parametrize("split", [-1, 0, 1], ids=["auto", "whole", "split"])
@pytest.mark.parametrize("M,N,K", [(256, 256, 128), (520, 1030, 1000), (300, 600, 4107), (1024, 2048, 4160),
                                   (2000, 3000, 257), (777, 512, 64)])
@pytest.mark.parametrize("dtype", ["f16", "s8"])
def test_bk128_pair_tiles(dev, dtype, M, N, K, split):
    # Stages of 128 k (A as two 64-k sub-tiles, B as 64-column atoms of 128
    # rows), three deep; ragged K tails, one k-block, INT8 chunks of eight
    # k-blocks.
    A, B = inputs.make_operands(dtype, M, N, K, seed=1010 + M + N + K)
    gemmpipe.gemmpipe_set_plan_override(-1, 256, 0, 1, split)
    gemmpipe.gemmpipe_set_plan_bk(128)
    try:
        plan = gemmpipe.gemmpipe_plan(0 if dtype == "s8" else 1, M, N, K)
        assert plan["BK"] == 128 and plan["stages"] == 3 and plan["cta_pair"] == 1
        assert plan["k_blocks"] == (K + 127) // 128
        got = run_s8(A, B, dev) if dtype == "s8" else run_f16(A, B, dev)
    finally:
        gemmpipe.gemmpipe_set_plan_bk(0)
        gemmpipe.gemmpipe_set_plan_override(-1, 0, 0, -1, -1)
    if dtype == "s8":
        np.testing.assert_array_equal(got, oracle.gemm_s8s8s32(A, B))
    else:
        assert_f16_close(got, oracle.gemm_f16f32(A, B), f"bk128 {M}x{N}x{K} split={split}")


def test_bk128_int8_chunk_extremes(dev):
    # Partial sums of 1024 k just below 2^24 with odd values: exact only if
    # every accumulation chunk stays within 1024 k (eight 128-k blocks).
    M, N, K = 300, 520, 4096
    rng = np.random.default_rng(23)
    A = np.where(rng.random((M, K)) < 0.97, -128, 127).astype(np.int8)
    B = np.where(rng.random((K, N)) < 0.97, -128, 127).astype(np.int8)
    gemmpipe.gemmpipe_set_plan_override(-1, 256, 0, 1, -1)
    gemmpipe.gemmpipe_set_plan_bk(128)
    try:
        assert gemmpipe.gemmpipe_plan(0, M, N, K)["BK"] == 128
        got = run_s8(A, B, dev)
    finally:
        gemmpipe.gemmpipe_set_plan_bk(0)
        gemmpipe.gemmpipe_set_plan_override(-1, 0, 0, -1, -1)
    np.testing.assert_array_equal(got, oracle.gemm_s8s8s32(A, B))
