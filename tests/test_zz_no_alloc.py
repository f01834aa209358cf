"""gemm_s8s8s32_noalloc, the INT8 entry point for callers that cannot let
the library allocate device memory (a fixed device-memory budget, or no
allocator stalls allowed on the call path).  Its fp16 operand copies live in
a fixed static scratch array instead of a cudaMalloc'd workspace.

The results must equal gemm_s8s8s32's bit for bit (INT8 is exact), on two
calls in a row of different shapes -- the second call must not depend on
what the first left in the shared scratch.  This file is collected last, so
a run that stops at the first failure has run every other test already.
"""
from __future__ import annotations

import numpy as np
import pytest

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


def test_noalloc_matches_allocating_entry_point(lib):
    import torch
    stream = torch.cuda.current_stream().cuda_stream
    # Both shapes fit the fixed scratch: 2 * (M * Kp + K * Np) bytes.
    for M, N, K, seed in [(1000, 1500, 2000, 71), (777, 300, 3001, 72)]:
        Kp, Np = -(-K // 8) * 8, -(-N // 8) * 8
        assert 2 * (M * Kp + K * Np) <= gemmpipe.NOALLOC_SCRATCH_BYTES
        A, B = inputs.make_operands("s8", M, N, K, seed=seed)
        Ad, Bd = _dev(A, torch), _dev(B, torch)
        ref = torch.full((M, N), -1, dtype=torch.int32, device="cuda:0")
        got = torch.full((M, N), -2, dtype=torch.int32, device="cuda:0")
        assert lib.gemm_s8s8s32(M, N, K, Ad.data_ptr(), Bd.data_ptr(), ref.data_ptr(), stream) == gemmpipe.OK
        assert lib.gemm_s8s8s32_noalloc(M, N, K, Ad.data_ptr(), Bd.data_ptr(), got.data_ptr(),
                                        stream) == gemmpipe.OK
        assert lib.gemmpipe_get_device_status(stream) == gemmpipe.OK
        assert torch.equal(got, ref), (M, N, K)


def test_noalloc_refuses_problems_beyond_its_scratch(lib):
    import torch
    stream = torch.cuda.current_stream().cuda_stream
    M = N = K = 4096   # needs 64 MiB of scratch
    A = torch.zeros((M, K), dtype=torch.int8, device="cuda:0")
    B = torch.zeros((K, N), dtype=torch.int8, device="cuda:0")
    C = torch.full((M, N), 5, dtype=torch.int32, device="cuda:0")
    assert lib.gemm_s8s8s32_noalloc(M, N, K, A.data_ptr(), B.data_ptr(), C.data_ptr(),
                                    stream) == gemmpipe.ERR_INVALID_VALUE
    assert lib.gemmpipe_get_device_status(stream) == gemmpipe.OK
    assert bool((C == 5).all())   # nothing was launched
