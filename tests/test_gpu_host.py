"""GPU parity of the host-buffer calls (gemm_s8s8s32_host, gemm_f16f32_host)
against the CPU oracle: A, B and C in host memory, row panels copied in,
computed and copied back with overlap.

INT8 bit-exact; FP16 within max-abs 1e-2 and relative Frobenius 1e-4.  The
shapes give one panel, several panels with a ragged last one, odd pitches,
K = 0, page-locked and pageable buffers, and calls queued back to back on
one stream (the library's device buffers are reused by the next call).
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
    gemmpipe.gemmpipe_set_plan_override(-1, 0, 0, -1, -1)
    yield torch.device("cuda:0")
    gemmpipe.gemmpipe_set_plan_override(-1, 0, 0, -1, -1)


def host(a: np.ndarray, pinned: bool):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    return t.pin_memory() if pinned else t.clone()


def out(shape, dtype, fill, pinned: bool):
    import torch
    return torch.full(shape, fill, dtype=dtype, pin_memory=pinned)


def run_host(dtype: str, A: np.ndarray, B: np.ndarray, pinned: bool) -> np.ndarray:
    import torch
    M, K = A.shape
    N = B.shape[1]
    Ah, Bh = host(A, pinned), host(B, pinned)  # referenced until the synchronization below
    if dtype == "s8":
        C = out((M, N), torch.int32, -7, pinned)
        gemmpipe.gemm_s8s8s32_host(M, N, K, Ah, Bh, C)
    else:
        C = out((M, N), torch.float32, float("nan"), pinned)
        gemmpipe.gemm_f16f32_host(M, N, K, Ah, Bh, C)
    assert gemmpipe.gemmpipe_get_device_status() == gemmpipe.OK
    return C.numpy()


def assert_f16_close(got, ref, what=""):
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    d = got.astype(np.float64) - ref.astype(np.float64)
    err = np.abs(d).max() if d.size else 0.0
    nrm = np.linalg.norm(ref.astype(np.float64))
    rel = np.linalg.norm(d) / nrm if nrm > 0 else np.linalg.norm(d)
    assert err <= MAX_ABS and rel <= MAX_REL_FRO, f"{what}: max-abs {err:.3g} rel-fro {rel:.3g}"


SHAPES = [
    (7, 9, 11),          # one panel, nothing aligned
    (512, 256, 128),     # exactly one panel
    (513, 64, 100),      # two panels, the second one row
    (1300, 1000, 777),   # three panels, ragged last one, odd K
    (2100, 520, 2048),   # three panels of 768 rows, the last 564
    # B of at least 4 MiB with N a multiple of 32: the first panel is
    # computed in column parts as B's parts arrive
    (1100, 2048, 2080),  # INT8 and FP16 split
    (600, 4096, 1024),   # one panel, split
    (700, 2048, 2051),   # INT8 split (any K); FP16 not (K not a multiple of 8)
    (700, 1024, 16384),  # long K (16 MiB of int8 B), first panel in halves
]


@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_host_s8(dev, M, N, K, pinned):
    A, B = inputs.make_operands("s8", M, N, K, seed=900 + M + 3 * N + 7 * K)
    assert np.array_equal(run_host("s8", A, B, pinned), oracle.gemm_s8s8s32(A, B))


@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_host_f16(dev, M, N, K, pinned):
    A, B = inputs.make_operands("f16", M, N, K, seed=950 + M + 3 * N + 7 * K)
    assert_f16_close(run_host("f16", A, B, pinned), oracle.gemm_f16f32(A, B), f"{M}x{N}x{K}")


def test_host_numpy_buffers(dev):
    M, N, K = 1100, 300, 260
    A, B = inputs.make_operands("s8", M, N, K, seed=991)
    C = np.full((M, N), 5, dtype=np.int32)
    gemmpipe.gemm_s8s8s32_host(M, N, K, A, B, C)
    assert gemmpipe.gemmpipe_get_device_status() == gemmpipe.OK
    assert np.array_equal(C, oracle.gemm_s8s8s32(A, B))


def test_host_k_zero(dev):
    import torch
    for dtype in ("s8", "f16"):
        C = out((600, 40), torch.int32 if dtype == "s8" else torch.float32, 3, True)
        fn = gemmpipe.gemm_s8s8s32_host if dtype == "s8" else gemmpipe.gemm_f16f32_host
        fn(600, 40, 0, None, None, C)
        assert gemmpipe.gemmpipe_get_device_status() == gemmpipe.OK
        assert (C.numpy() == 0).all()


def test_host_calls_back_to_back(dev):
    """Several calls queued on one stream before any synchronization: each
    reuses the library's device buffers, so the later copies in must wait
    for the earlier panels' GEMMs and copies out."""
    import torch
    shapes = [(1300, 700, 500), (900, 700, 500), (1300, 700, 500), (2000, 64, 300)]
    ops, outs, keep = [], [], []
    for i, (M, N, K) in enumerate(shapes):
        A, B = inputs.make_operands("s8", M, N, K, seed=1200 + i)
        ops.append((A, B))
        C = out((M, N), torch.int32, -1, True)
        outs.append(C)
        # The page-locked inputs stay referenced until the stream is
        # synchronized: the copies read them asynchronously.
        keep.append((host(A, True), host(B, True)))
        gemmpipe.gemm_s8s8s32_host(M, N, K, keep[-1][0], keep[-1][1], C)
    assert gemmpipe.gemmpipe_get_device_status() == gemmpipe.OK
    for (A, B), C in zip(ops, outs):
        assert np.array_equal(C.numpy(), oracle.gemm_s8s8s32(A, B))


def test_host_after_device_work_on_the_stream(dev):
    """The copies in start after earlier work on the caller's stream: a
    device-to-host copy into A, queued before the call, is what the call
    reads."""
    import torch
    M, N, K = 1030, 200, 300
    A, B = inputs.make_operands("s8", M, N, K, seed=1300)
    Ah = host(np.zeros_like(A), True)
    Ad = torch.from_numpy(A).to(dev)
    torch.cuda._sleep(2_000_000)  # keep the stream busy so the copy lands late
    Ah.copy_(Ad, non_blocking=True)
    C = out((M, N), torch.int32, -1, True)
    Bh = host(B, True)
    gemmpipe.gemm_s8s8s32_host(M, N, K, Ah, Bh, C)
    assert gemmpipe.gemmpipe_get_device_status() == gemmpipe.OK
    assert np.array_equal(C.numpy(), oracle.gemm_s8s8s32(A, B))


@pytest.mark.parametrize("producer", [0, 2], ids=["in-kernel-widening", "comparison-path"])
def test_host_s8_other_int8_paths(dev, producer):
    M, N, K = 1100, 256, 512
    A, B = inputs.make_operands("s8", M, N, K, seed=1400 + producer)
    gemmpipe.gemmpipe_set_plan_override(producer, 0, 0, -1, -1)
    try:
        got = run_host("s8", A, B, True)
    finally:
        gemmpipe.gemmpipe_set_plan_override(-1, 0, 0, -1, -1)
    assert np.array_equal(got, oracle.gemm_s8s8s32(A, B))


def test_host_s8_full_size(dev, full_size):
    """INT8 4096^3 (four panels of 1024 rows, the first in column halves)
    through host buffers, every element bit for bit."""
    A, B, want = full_size(2)
    assert np.array_equal(run_host("s8", A, B, True), want)


def test_host_f16_full_size(dev, full_size):
    """FP16 4096^3 through host buffers (four panels, the first in column
    halves), every element within the FP16 tolerance."""
    A, B, want = full_size("fp16_4096")
    assert_f16_close(run_host("f16", A, B, True), want, "fp16 4096^3 host")
