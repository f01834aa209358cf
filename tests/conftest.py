import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")


def gpu_available() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    return oracle.default()


# Whole-C oracle results of the full-size workloads, computed once per test
# session (several tests compare against the same product) with their wall
# times, which the terminal summary prints so the suite's cost stays visible.
_ORACLE_TIMES: list[tuple[str, float, int]] = []


def _full_operands(key):
    from software_pipelined_loop_gb300 import inputs
    if key == "fp16_4096":
        # FP16 4096^3, uniform on [-1, 1]: the fp16 half of the headline metric.
        A, B = inputs.make_operands("f16", 4096, 4096, 4096, inputs.SEED_BASE + 5)
        return "fp16_4096", "f16", A, B
    name, dtype, _, _, _, A, B = inputs.workload_operands(key)
    return name, dtype, A, B


@pytest.fixture(scope="session")
def full_size():
    """get(key) -> (A, B, C_oracle) for a workload index of inputs.WORKLOADS
    or "fp16_4096"; the oracle computes every element of C once."""
    import time

    import oracle
    cache = {}

    def get(key):
        if key not in cache:
            name, dtype, A, B = _full_operands(key)
            threads = oracle.default_threads()
            t = time.perf_counter()
            C = oracle.gemm_s8s8s32(A, B, threads=threads) if dtype == "s8" else \
                oracle.gemm_f16f32(A, B, threads=threads)
            _ORACLE_TIMES.append((name, time.perf_counter() - t, threads))
            cache[key] = (A, B, C)
        return cache[key]

    return get


def pytest_terminal_summary(terminalreporter):
    for name, secs, threads in _ORACLE_TIMES:
        terminalreporter.write_line(f"oracle, whole C of {name}: {secs:.1f} s on {threads} threads")
