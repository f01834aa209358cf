"""The pipelining itself, observed on the device ("Pipeline GPU Kernel",
Steps 3-4: the loads of the next K-tiles are issued while the tensor cores
work on the current one; Step 6 compares against the non-pipelined
load / wait / compute loop).

The trace hook makes CTA 0 (the leader of pair 0) stamp %globaltimer when
its producer has issued the copies of each k-block and when its MMA thread
finds that k-block's data ready.  With the default 6-stage ring the MMA
thread finds k-blocks ready at the tensor-core rate and the next k-block's
copies are already on their way; with a single stage every k-block waits for
its own load, which is issued only after the previous k-block's MMAs have
read their stage.
"""
from __future__ import annotations

import numpy as np
import pytest

from software_pipelined_loop_gb300 import gemmpipe, inputs

pytestmark = pytest.mark.gpu

N_TRACE = 256


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


def traced(dev, stages: int):
    """(producer stamps, MMA-ready stamps, plan) of one FP16 4096^3 call on
    CTA pairs with the given ring depth."""
    import torch
    M = N = K = 4096
    A, B = inputs.make_operands("f16", M, N, K, seed=77)
    Ad, Bd = torch.from_numpy(A).to(dev), torch.from_numpy(B).to(dev)
    C = torch.empty((M, N), dtype=torch.float32, device=dev)
    gemmpipe.gemmpipe_set_plan_override(0, 256, stages, 1, -1)
    try:
        plan = gemmpipe.gemmpipe_plan(1, M, N, K, Ad, Bd, C)
        gemmpipe.gemm_f16f32(M, N, K, Ad, Bd, C)  # warm
        buf = torch.zeros(3 * N_TRACE, dtype=torch.int64, device=dev)
        gemmpipe.gemmpipe_test_trace(buf, N_TRACE)
        gemmpipe.gemm_f16f32(M, N, K, Ad, Bd, C)
        assert gemmpipe.gemmpipe_get_device_status() == gemmpipe.OK
    finally:
        gemmpipe.gemmpipe_set_plan_override(-1, 0, 0, -1, -1)
    t = buf.cpu().numpy()
    return t[:N_TRACE], t[N_TRACE:2 * N_TRACE], t[2 * N_TRACE:], plan


def stats(prod, mma):
    used = int((prod > 0).sum())
    assert used > 32 and (mma[:used] > 0).all()
    # Causality: a k-block's data is found ready only after its copies were issued.
    assert (mma[:used] >= prod[:used]).all()
    assert (np.diff(prod[:used]) >= 0).all() and (np.diff(mma[:used]) >= 0).all()
    steady = range(8, used - 8)
    next_first = np.mean([prod[j + 1] < mma[j] for j in steady])
    gap = np.median(np.diff(mma[8:used - 8])) / 1e3  # microseconds per k-block
    return next_first, gap


def test_ring_overlaps_loads_with_mma(dev):
    p6, m6, c6, plan6 = traced(dev, 6)
    p1, m1, c1, plan1 = traced(dev, 1)
    assert plan6["stages"] == 6 and plan1["stages"] == 1 and plan6["cta_pair"] == plan1["cta_pair"] == 1
    next6, gap6 = stats(p6, m6)
    next1, gap1 = stats(p1, m1)
    # One stage: the copies of k-block j+1 go out only after k-block j's
    # MMAs have read the single stage -- never before its data was found.
    assert next1 == 0.0
    # Six stages: mostly the next k-block is already being copied, and
    # k-blocks come at least twice as fast.
    assert next6 >= 0.5, next6
    assert gap1 >= 2 * gap6, (gap1, gap6)


def test_trace_cycle_stamps_follow_the_clock(dev):
    """The %clock64 stamps beside the MMA-ready times count SM cycles: they
    increase with every k-block, and cycles over nanoseconds between the
    first and last stamp is an SM clock between 0.5 and 2.2 GHz."""
    prod, mma, cyc, _ = traced(dev, 6)
    used = int((prod > 0).sum())
    assert used > 32
    assert (np.diff(cyc[:used]) > 0).all()
    ghz = (cyc[used - 1] - cyc[0]) / (mma[used - 1] - mma[0])
    assert 0.5 <= ghz <= 2.2, ghz
