"""Python binding of libgemmpipe (include/gemmpipe.h): argument marshalling only.

Every function has the C entry point's name and arguments.  Matrix arguments
may be torch tensors (their ``data_ptr()`` is passed) or raw device
addresses (ints).  ``stream`` may be None (torch's current CUDA stream), a
``torch.cuda.Stream`` or a raw ``cudaStream_t`` value.  A non-OK status
raises :class:`GemmpipeError`.  All GEMM work runs in the CUDA library; when
the library is missing the calls raise instead of computing anything.
"""
from __future__ import annotations

import ctypes
import os
import re

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgemmpipe.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "gemmpipe.h")

STATUS = {0: "GEMMPIPE_OK", 1: "GEMMPIPE_ERR_INVALID_VALUE", 2: "GEMMPIPE_ERR_UNSUPPORTED_DEVICE",
          3: "GEMMPIPE_ERR_LAUNCH", 4: "GEMMPIPE_ERR_TIMEOUT", 5: "GEMMPIPE_ERR_INTERNAL",
          6: "GEMMPIPE_ERR_OUT_OF_MEMORY"}
NOALLOC_SCRATCH_BYTES = 16 << 20  # GEMMPIPE_NOALLOC_SCRATCH_BYTES
OK, ERR_INVALID_VALUE, ERR_UNSUPPORTED_DEVICE, ERR_LAUNCH, ERR_TIMEOUT, ERR_INTERNAL, ERR_OUT_OF_MEMORY = range(7)


class GemmpipeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


class PlanT(ctypes.Structure):
    _fields_ = [("producer", ctypes.c_int), ("BM", ctypes.c_int), ("BN", ctypes.c_int), ("BK", ctypes.c_int),
                ("stages", ctypes.c_int), ("k_chunk", ctypes.c_int), ("threads", ctypes.c_int),
                ("cta_pair", ctypes.c_int), ("grid", ctypes.c_int), ("tiles", ctypes.c_int64), ("units", ctypes.c_int64),
                ("split_tiles", ctypes.c_int64),
                ("k_blocks", ctypes.c_int64),
                ("smem_bytes", ctypes.c_int64), ("vector_store", ctypes.c_int),
                ("operand_copy", ctypes.c_int), ("workspace_bytes", ctypes.c_int64)]


_lib = None
_i64, _vp, _int = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Opens the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with software_pipelined_loop_gb300.build.build()")
    lib = ctypes.CDLL(path)
    sig = {
        "gemm_s8s8s32": (_int, [_i64, _i64, _i64, _vp, _vp, _vp, _vp]),
        "gemm_f16f32": (_int, [_i64, _i64, _i64, _vp, _vp, _vp, _vp]),
        "gemm_s8s8s32_noalloc": (_int, [_i64, _i64, _i64, _vp, _vp, _vp, _vp]),
        "gemm_s8s8s32_host": (_int, [_i64, _i64, _i64, _vp, _vp, _vp, _vp]),
        "gemm_f16f32_host": (_int, [_i64, _i64, _i64, _vp, _vp, _vp, _vp]),
        "gemmpipe_host_panel_rows": (_i64, [_i64]),
        "gemmpipe_test_trace": (_int, [_vp, _i64]),
        "gemmpipe_get_device_status": (_int, [_vp]),
        "gemmpipe_status_string": (ctypes.c_char_p, [_int]),
        "gemmpipe_compute_load_ratio": (ctypes.c_double, [_int, _int, _int, _int]),
        "gemmpipe_stage_smem_bytes": (_i64, [_int, _int, _int, _int, _int]),
        "gemmpipe_plan": (_int, [_int, _i64, _i64, _i64, _vp, _vp, _vp, ctypes.POINTER(PlanT)]),
        "gemmpipe_set_plan_override": (_int, [_int, _int, _int, _int, _int]),
        "gemmpipe_set_plan_bk": (_int, [_int]),
        "gemmpipe_release_workspaces": (_int, []),
        "gemmpipe_timing_enable": (_int, [_int]),
        "gemmpipe_timing_read": (_int, [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(_i64),
                                        ctypes.POINTER(ctypes.c_double), ctypes.POINTER(_i64)]),
        "gemmpipe_launch_count": (_i64, []),
        "gemmpipe_copy": (_int, [_vp, _vp, _i64, _vp]),
        "gemmpipe_test_inject_stall": (_int, [_i64, _int]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def header_functions(path: str = HEADER) -> list[str]:
    """Names of the entry points include/gemmpipe.h declares."""
    text = open(path).read()
    return re.findall(r"^GEMMPIPE_API\s+[\w\s\*]*?\b(\w+)\s*\(", text, flags=re.M)


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return int(x.data_ptr())
    if hasattr(x, "__array_interface__"):
        return int(x.__array_interface__["data"][0])
    raise TypeError(f"expected a tensor or an address, got {type(x)!r}")


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def _check(status: int, where: str) -> None:
    if status != OK:
        raise GemmpipeError(status, where)


def gemm_s8s8s32(M, N, K, A, B, C, stream=None) -> None:
    """C (M x N int32) = A (M x K int8) @ B (K x N int8), enqueued on `stream`."""
    _check(load().gemm_s8s8s32(M, N, K, _ptr(A), _ptr(B), _ptr(C), _stream(stream)), "gemm_s8s8s32")


def gemm_f16f32(M, N, K, A, B, C, stream=None) -> None:
    """C (M x N fp32) = A (M x K fp16) @ B (K x N fp16), enqueued on `stream`."""
    _check(load().gemm_f16f32(M, N, K, _ptr(A), _ptr(B), _ptr(C), _stream(stream)), "gemm_f16f32")


def gemm_s8s8s32_noalloc(M, N, K, A, B, C, stream=None) -> None:
    """gemm_s8s8s32 that never allocates: the fp16 operand copies use the
    library's fixed device scratch (NOALLOC_SCRATCH_BYTES), so problems
    needing more are refused; calls overlapping on the GPU race on it."""
    _check(load().gemm_s8s8s32_noalloc(M, N, K, _ptr(A), _ptr(B), _ptr(C), _stream(stream)),
           "gemm_s8s8s32_noalloc")


def gemm_s8s8s32_host(M, N, K, A, B, C, stream=None) -> None:
    """gemm_s8s8s32 with A, B and C in host memory (CPU tensors or numpy
    arrays): copies in, GEMM and copies out overlapped by row panels.
    Asynchronous for page-locked buffers: synchronize `stream` before
    reading C."""
    _check(load().gemm_s8s8s32_host(M, N, K, _ptr(A), _ptr(B), _ptr(C), _stream(stream)), "gemm_s8s8s32_host")


def gemm_f16f32_host(M, N, K, A, B, C, stream=None) -> None:
    """gemm_f16f32 with A, B and C in host memory (see gemm_s8s8s32_host)."""
    _check(load().gemm_f16f32_host(M, N, K, _ptr(A), _ptr(B), _ptr(C), _stream(stream)), "gemm_f16f32_host")


def gemmpipe_host_panel_rows(M: int) -> int:
    """Rows per panel of the host-buffer calls (no GPU needed)."""
    return int(load().gemmpipe_host_panel_rows(M))


def gemmpipe_get_device_status(stream=None) -> int:
    """Synchronizes `stream`; returns (and clears) the device status code."""
    return load().gemmpipe_get_device_status(_stream(stream))


def gemmpipe_status_string(status: int) -> str:
    return load().gemmpipe_status_string(status).decode()


def gemmpipe_compute_load_ratio(BM: int, BN: int, BK: int, elem_bytes: int) -> float:
    return load().gemmpipe_compute_load_ratio(BM, BN, BK, elem_bytes)


def gemmpipe_stage_smem_bytes(BM: int, BN: int, BK: int, elem_bytes: int, stages: int) -> int:
    return load().gemmpipe_stage_smem_bytes(BM, BN, BK, elem_bytes, stages)


def gemmpipe_plan(dtype: int, M, N, K, A=None, B=None, C=None) -> dict:
    """Kernel plan for gemm_s8s8s32 (dtype 0) or gemm_f16f32 (dtype 1)."""
    p = PlanT()
    _check(load().gemmpipe_plan(dtype, M, N, K, _ptr(A), _ptr(B), _ptr(C), ctypes.byref(p)), "gemmpipe_plan")
    return {name: getattr(p, name) for name, _ in PlanT._fields_}


def gemmpipe_set_plan_override(producer: int = -1, bn: int = 0, stages: int = 0, cta_pair: int = -1,
                               split: int = -1) -> None:
    _check(load().gemmpipe_set_plan_override(producer, bn, stages, cta_pair, split), "gemmpipe_set_plan_override")


def gemmpipe_set_plan_bk(bk: int) -> None:
    _check(load().gemmpipe_set_plan_bk(bk), "gemmpipe_set_plan_bk")


def gemmpipe_release_workspaces() -> None:
    _check(load().gemmpipe_release_workspaces(), "gemmpipe_release_workspaces")


def gemmpipe_timing_enable(enable: bool) -> None:
    _check(load().gemmpipe_timing_enable(1 if enable else 0), "gemmpipe_timing_enable")


def gemmpipe_timing_read() -> tuple[float, int, float, int]:
    """(gemm_ms, gemm_launches, aux_ms, aux_launches) since the last read."""
    gm, am = ctypes.c_double(), ctypes.c_double()
    gn, an = ctypes.c_int64(), ctypes.c_int64()
    _check(load().gemmpipe_timing_read(ctypes.byref(gm), ctypes.byref(gn), ctypes.byref(am), ctypes.byref(an)),
           "gemmpipe_timing_read")
    return gm.value, gn.value, am.value, an.value


def gemmpipe_launch_count() -> int:
    return load().gemmpipe_launch_count()


def gemmpipe_copy(dst, src, nbytes: int, stream=None) -> None:
    _check(load().gemmpipe_copy(_ptr(dst), _ptr(src), nbytes, _stream(stream)), "gemmpipe_copy")


def gemmpipe_test_trace(buffer, entries: int) -> None:
    """Arms the pipelining trace for the next GEMM launch (see the C header):
    `buffer` is a device array of 2 * entries uint64."""
    _check(load().gemmpipe_test_trace(_ptr(buffer), entries), "gemmpipe_test_trace")


def gemmpipe_test_inject_stall(k_block: int, timeout_ms: int = 0) -> None:
    _check(load().gemmpipe_test_inject_stall(k_block, timeout_ms), "gemmpipe_test_inject_stall")
