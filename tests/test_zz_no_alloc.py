"""gemm_s8s8s32_noalloc, the INT8 entry point for callers that cannot let
the library allocate device memory (a process whose device memory is all
planned up front, or a call path on which a cudaMalloc/cudaFree stall of the
whole device is not acceptable).  Its fp16 operand copies live in a fixed
static scratch array instead of a cudaMalloc'd workspace.

Checked here: on calls in a row of different shapes (a CTA-pair plan,
single-CTA plans, and K = 0, which must zero C) the result
equals the CPU oracle's and gemm_s8s8s32's bit for bit -- no call depends on
what the one before left in the shared scratch; once the library's code is
loaded on the device, a call on a fresh stream leaves the device's free
memory unchanged; and problems beyond the scratch are refused before
anything runs.  This file is collected last, so a run that stops at the
first failure has run every other test already.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from software_pipelined_loop_gb300 import gemmpipe, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from software_pipelined_loop_gb300 import build
    build.build()
    return gemmpipe.load()


def _dev(a, torch):
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda:0")


def _fits(M, N, K):
    Kp, Np = -(-K // 8) * 8, -(-N // 8) * 8
    return 2 * (M * Kp + K * Np) <= gemmpipe.NOALLOC_SCRATCH_BYTES


def test_noalloc_matches_oracle_and_allocating_entry_point(lib):
    import torch
    stream = torch.cuda.current_stream().cuda_stream
    # CTA pairs (24 tiles of 256 x 256), a single CTA per 128 x 128 tile
    # (N <= 128), K = 0, then single CTAs again (a small problem: at most a
    # quarter of the SM pairs' worth of pair tiles), all back to back on one
    # stream.
    cases = [(1000, 1500, 2000, 71), (300, 64, 1000, 72), (257, 190, 0, 73), (777, 300, 3001, 74)]
    for M, N, K, seed in cases:
        assert _fits(M, N, K)
        A, B = inputs.make_operands("s8", M, N, K, seed=seed)
        want = oracle.gemm_s8s8s32(A, B) if K > 0 else np.zeros((M, N), dtype=np.int32)
        Ad, Bd = _dev(A, torch), _dev(B, torch)
        ref = torch.full((M, N), -1, dtype=torch.int32, device="cuda:0")
        got = torch.full((M, N), -2, dtype=torch.int32, device="cuda:0")
        assert lib.gemm_s8s8s32(M, N, K, Ad.data_ptr(), Bd.data_ptr(), ref.data_ptr(), stream) == gemmpipe.OK
        assert lib.gemm_s8s8s32_noalloc(M, N, K, Ad.data_ptr(), Bd.data_ptr(), got.data_ptr(),
                                        stream) == gemmpipe.OK
        assert lib.gemmpipe_get_device_status(stream) == gemmpipe.OK
        assert np.array_equal(got.cpu().numpy(), want), (M, N, K)
        assert torch.equal(got, ref), (M, N, K)


def test_noalloc_call_leaves_free_device_memory_unchanged(lib):
    import torch
    M, N, K = 1024, 1024, 2048
    A, B = inputs.make_operands("s8", M, N, K, seed=75)
    Ad, Bd = _dev(A, torch), _dev(B, torch)
    C = torch.full((M, N), -3, dtype=torch.int32, device="cuda:0")
    s0 = torch.cuda.current_stream().cuda_stream
    # The first call on a device loads the library's code there (the static
    # scratch array included): that is set-up, done once.
    assert lib.gemm_s8s8s32_noalloc(M, N, K, Ad.data_ptr(), Bd.data_ptr(), C.data_ptr(), s0) == gemmpipe.OK
    assert lib.gemmpipe_get_device_status(s0) == gemmpipe.OK
    side = torch.cuda.Stream()
    C.fill_(-4)
    lib.gemmpipe_release_workspaces()
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    assert lib.gemm_s8s8s32_noalloc(M, N, K, Ad.data_ptr(), Bd.data_ptr(), C.data_ptr(),
                                    side.cuda_stream) == gemmpipe.OK
    assert lib.gemmpipe_get_device_status(side.cuda_stream) == gemmpipe.OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, (free0, free1)
    assert np.array_equal(C.cpu().numpy(), oracle.gemm_s8s8s32(A, B))


def test_noalloc_refuses_problems_beyond_its_scratch(lib):
    import torch
    stream = torch.cuda.current_stream().cuda_stream
    M = N = K = 4096   # needs 64 MiB of scratch
    assert not _fits(M, N, K)
    A = torch.zeros((M, K), dtype=torch.int8, device="cuda:0")
    B = torch.zeros((K, N), dtype=torch.int8, device="cuda:0")
    C = torch.full((M, N), 5, dtype=torch.int32, device="cuda:0")
    assert lib.gemm_s8s8s32_noalloc(M, N, K, A.data_ptr(), B.data_ptr(), C.data_ptr(),
                                    stream) == gemmpipe.ERR_INVALID_VALUE
    assert lib.gemmpipe_get_device_status(stream) == gemmpipe.OK
    assert bool((C == 5).all())   # nothing was launched
