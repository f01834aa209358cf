"""The C ABI without a GPU: the library loads, exports what the header
declares, and rejects bad arguments on the host before touching a device."""
from __future__ import annotations

import ctypes
import subprocess

import pytest

import oracle
from software_pipelined_loop_gb300 import build, gemmpipe


@pytest.fixture(scope="module")
def lib():
    build.build()
    return gemmpipe.load()


def test_exports_every_declared_symbol(lib):
    names = gemmpipe.header_functions()
    assert len(names) >= 14
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", gemmpipe.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    assert set(names) <= exported
    # Nothing else leaks out (the statically linked CUDA runtime stays hidden).
    assert {s for s in exported if not s.startswith("_")} == set(names)


def test_binding_covers_header(lib):
    for n in gemmpipe.header_functions():
        assert callable(getattr(gemmpipe, n)), n


def test_ratio_and_budget_helpers(lib):
    # Step 1 worked example: 32x32x32 fp16, two stages = the doubled 8 KB.
    assert gemmpipe.gemmpipe_stage_smem_bytes(32, 32, 32, 2, 1) == 4096
    assert gemmpipe.gemmpipe_stage_smem_bytes(32, 32, 32, 2, 2) == oracle.smem_doubled_bytes(32, 32, 32, 2) == 8192
    for t in [(32, 32, 32, 2), (128, 256, 64, 2), (128, 128, 64, 2), (128, 256, 128, 1), (3, 5, 7, 4)]:
        assert gemmpipe.gemmpipe_compute_load_ratio(*t) == pytest.approx(oracle.compute_load_ratio(*t), rel=1e-15)
    assert gemmpipe.gemmpipe_compute_load_ratio(0, 1, 1, 1) < 0
    assert gemmpipe.gemmpipe_stage_smem_bytes(1, 1, 1, 1, 0) == -1
    # The ring of the 128x256x64 fp16 kernel, four stages: 192 KiB.
    assert gemmpipe.gemmpipe_stage_smem_bytes(128, 256, 64, 2, 4) == 196608


def test_status_strings(lib):
    for code in range(7):
        assert gemmpipe.gemmpipe_status_string(code)
    assert gemmpipe.gemmpipe_status_string(99) == "unknown status"


def test_host_side_argument_checks(lib):
    f16 = lib.gemm_f16f32
    s8 = lib.gemm_s8s8s32
    fake = 1 << 20  # never dereferenced: these fail before any device call
    assert f16(-1, 4, 4, fake, fake, fake, None) == gemmpipe.ERR_INVALID_VALUE
    assert s8(4, 4, -2, fake, fake, fake, None) == gemmpipe.ERR_INVALID_VALUE
    assert f16(1 << 31, 4, 4, fake, fake, fake, None) == gemmpipe.ERR_INVALID_VALUE
    big = (1 << 31) - 1
    assert s8(big, 8, big, fake, fake, fake, None) == gemmpipe.ERR_INVALID_VALUE    # 2^62 elements of A
    assert f16(big, big, 8, fake, fake, fake, None) == gemmpipe.ERR_INVALID_VALUE   # 2^62 elements of C
    # 2^32 tiles of 128 x 128 (C of 2^46 values, under the 2^56-element rule)
    assert f16(1 << 23, 1 << 23, 8, fake, fake, fake, None) == gemmpipe.ERR_INVALID_VALUE
    assert s8(1 << 23, 1 << 23, 8, fake, fake, fake, None) == gemmpipe.ERR_INVALID_VALUE
    assert f16(4, 4, 4, None, fake, fake, None) == gemmpipe.ERR_INVALID_VALUE
    assert s8(4, 4, 4, fake, fake, None, None) == gemmpipe.ERR_INVALID_VALUE
    assert f16(4, 4, 4, fake + 1, fake, fake, None) == gemmpipe.ERR_INVALID_VALUE   # fp16 misaligned
    assert s8(4, 4, 4, fake + 1, fake + 3, fake + 2, None) == gemmpipe.ERR_INVALID_VALUE  # int32 C misaligned
    assert f16(0, 4, 4, None, None, None, None) == gemmpipe.OK
    assert s8(4, 0, 4, None, None, None, None) == gemmpipe.OK
    assert lib.gemmpipe_set_plan_override(3, 0, 0, -1, -1) == gemmpipe.ERR_INVALID_VALUE
    assert lib.gemmpipe_set_plan_override(-1, 192, 0, -1, -1) == gemmpipe.ERR_INVALID_VALUE
    assert lib.gemmpipe_set_plan_override(-1, 0, 0, 3, -1) == gemmpipe.ERR_INVALID_VALUE
    assert lib.gemmpipe_set_plan_override(-1, 0, 0, -1, 2) == gemmpipe.ERR_INVALID_VALUE
    assert lib.gemmpipe_set_plan_override(-1, 0, 0, -1, -1) == gemmpipe.OK
    assert lib.gemmpipe_test_inject_stall(3, 0) == gemmpipe.ERR_INVALID_VALUE
    assert lib.gemmpipe_test_inject_stall(-1, 0) == gemmpipe.OK
    assert lib.gemmpipe_copy(None, None, -1, None) == gemmpipe.ERR_INVALID_VALUE
    assert lib.gemmpipe_test_trace(None, -1) == gemmpipe.ERR_INVALID_VALUE
    assert lib.gemmpipe_test_trace(fake, 1 << 21) == gemmpipe.ERR_INVALID_VALUE
    assert lib.gemmpipe_test_trace(None, 0) == gemmpipe.OK
    # Host-buffer calls: the same checks, before any device call.
    for fn in (lib.gemm_s8s8s32_host, lib.gemm_f16f32_host):
        assert fn(-1, 4, 4, fake, fake, fake, None) == gemmpipe.ERR_INVALID_VALUE
        assert fn(4, 4, 4, fake, fake, None, None) == gemmpipe.ERR_INVALID_VALUE
        assert fn(4, 4, 4, fake, fake, fake + 2, None) == gemmpipe.ERR_INVALID_VALUE  # C misaligned
        assert fn(big, 8, big, fake, fake, fake, None) == gemmpipe.ERR_INVALID_VALUE
        assert fn(0, 4, 4, None, None, None, None) == gemmpipe.OK
    assert lib.gemm_f16f32_host(4, 4, 4, fake + 1, fake, fake, None) == gemmpipe.ERR_INVALID_VALUE


def test_host_panel_rows(lib):
    rows = gemmpipe.gemmpipe_host_panel_rows
    # At least 512 rows; M / 4 rounded up to 256 beyond that.
    assert [rows(m) for m in (0, 1, 512, 513, 2048, 2049, 4096, 4097, 8192, 16384, 100000)] == \
        [512, 512, 512, 512, 512, 768, 1024, 1280, 2048, 4096, 25088]
    for m in range(1, 20000, 97):
        r = rows(m)
        assert r % 256 == 0 and r >= 512
        panels = -(-m // r)
        assert panels <= 4 and (panels == 1 or r * (panels - 1) < m)


def test_no_gpu_fails_loudly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    fake = 1 << 20
    # Valid arguments but no usable device: an error, never a CPU fallback.
    assert lib.gemm_f16f32(8, 8, 8, fake, fake, fake, None) == gemmpipe.ERR_UNSUPPORTED_DEVICE
    assert lib.gemm_s8s8s32(8, 8, 8, fake, fake, fake, None) == gemmpipe.ERR_UNSUPPORTED_DEVICE
    with pytest.raises(gemmpipe.GemmpipeError):
        gemmpipe.gemm_f16f32(8, 8, 8, fake, fake, fake, stream=0)
    assert lib.gemm_s8s8s32_host(8, 8, 8, fake, fake, fake, None) == gemmpipe.ERR_UNSUPPORTED_DEVICE
    assert lib.gemm_f16f32_host(8, 8, 8, fake, fake, fake, None) == gemmpipe.ERR_UNSUPPORTED_DEVICE


def test_header_parses():
    names = gemmpipe.header_functions()
    assert "gemm_s8s8s32" in names and "gemm_f16f32" in names and "gemmpipe_get_device_status" in names
