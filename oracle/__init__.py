"""CPU oracle for the pipelined tiled GEMM -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the bench's CPU-baseline and
reference legs may import this package.  The GPU library never does, and this
package never imports the GPU library.

The arithmetic lives in ``gemm_oracle.c`` (plain C, pthreads, no BLAS, no
CUDA), compiled by :func:`build` with gcc into ``liboracle.so`` next to it.
What each function follows in the pages ("Pipeline GPU Kernel" skill page):

* :func:`gemm_s8s8s32`, :func:`gemm_f16f32` -- the plain matrix product that
  Step 5 item 4 says pipelining must reproduce: it reorders loads and leaves
  the arithmetic as it was.  INT8 sums exactly in int64; FP16 sums in fp64
  and rounds once to fp32.
* :func:`smem_a_bytes`, :func:`smem_b_bytes`, :func:`smem_doubled_bytes` --
  the Step 1 shared-memory budget.
* :func:`compute_load_ratio` -- the Step 2 flop-per-byte ratio of one tile.

Every function here is pinned by tests in ``tests/test_oracle.py`` against
brute force, closed forms and the page's worked example.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_i64 = ctypes.c_int64
_vp = ctypes.c_void_p


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the C oracle into a shared library (gcc -O2, no fast-math)."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           "-ffp-contract=off", "-fno-fast-math", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def load_library(path: str) -> ctypes.CDLL:
    """Open one build of the C oracle and declare its signatures."""
    lib = ctypes.CDLL(path)
    lib.oracle_f16_to_f64.restype = ctypes.c_double
    lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
    for name in ("oracle_gemm_s8s8s32", "oracle_gemm_f16f32"):
        fn = getattr(lib, name)
        fn.restype = ctypes.c_int
        fn.argtypes = [_i64, _i64, _i64, _vp, _vp, _vp, _i64, _vp, ctypes.c_int]
    lib.oracle_smem_a_bytes.restype = _i64
    lib.oracle_smem_a_bytes.argtypes = [_i64, _i64, _i64]
    lib.oracle_smem_b_bytes.restype = _i64
    lib.oracle_smem_b_bytes.argtypes = [_i64, _i64, _i64]
    lib.oracle_smem_doubled_bytes.restype = _i64
    lib.oracle_smem_doubled_bytes.argtypes = [_i64, _i64, _i64, _i64]
    lib.oracle_compute_load_ratio.restype = ctypes.c_double
    lib.oracle_compute_load_ratio.argtypes = [_i64, _i64, _i64, _i64]
    return lib


def default_threads() -> int:
    return os.cpu_count() or 1


class OracleError(RuntimeError):
    pass


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p) if a.size else None


def _rows_arg(rows, M):
    if rows is None:
        return None, M
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    return r, int(r.size)


class Oracle:
    """The oracle's entry points bound to one compiled library."""

    def __init__(self, lib: ctypes.CDLL):
        self.lib = lib

    def gemm_s8s8s32(self, A, B, rows=None, threads=None, allow_overflow=False):
        """C = A @ B for int8 A (M x K), B (K x N), exact, as int32.

        With ``rows`` only those rows of C are computed (returned packed).
        Raises OracleError if an entry does not fit int32 (unless allowed)."""
        A = np.ascontiguousarray(A, dtype=np.int8)
        B = np.ascontiguousarray(B, dtype=np.int8)
        M, K = A.shape
        K2, N = B.shape
        if K != K2:
            raise ValueError("inner dimensions differ")
        r, n = _rows_arg(rows, M)
        C = np.zeros((n, N), dtype=np.int32)
        rc = self.lib.oracle_gemm_s8s8s32(M, N, K, _ptr(A), _ptr(B),
                                          _ptr(r) if r is not None else None, n,
                                          _ptr(C), threads or default_threads())
        if rc < 0 or (rc == 1 and not allow_overflow):
            raise OracleError(f"oracle_gemm_s8s8s32 returned {rc}")
        return C

    def gemm_f16f32(self, A, B, rows=None, threads=None):
        """C = A @ B for float16 A (M x K), B (K x N): fp64 sums, one rounding to fp32."""
        A = np.ascontiguousarray(A, dtype=np.float16)
        B = np.ascontiguousarray(B, dtype=np.float16)
        M, K = A.shape
        K2, N = B.shape
        if K != K2:
            raise ValueError("inner dimensions differ")
        r, n = _rows_arg(rows, M)
        C = np.zeros((n, N), dtype=np.float32)
        rc = self.lib.oracle_gemm_f16f32(M, N, K, _ptr(A.view(np.uint16)), _ptr(B.view(np.uint16)),
                                         _ptr(r) if r is not None else None, n,
                                         _ptr(C), threads or default_threads())
        if rc != 0:
            raise OracleError(f"oracle_gemm_f16f32 returned {rc}")
        return C

    def f16_to_f64(self, bits: int) -> float:
        """Value of one binary16 bit pattern (the oracle's own decoder)."""
        return self.lib.oracle_f16_to_f64(int(bits) & 0xFFFF)

    def smem_a_bytes(self, BM, BK, elem_bytes):
        return self.lib.oracle_smem_a_bytes(BM, BK, elem_bytes)

    def smem_b_bytes(self, BK, BN, elem_bytes):
        return self.lib.oracle_smem_b_bytes(BK, BN, elem_bytes)

    def smem_doubled_bytes(self, BM, BN, BK, elem_bytes):
        return self.lib.oracle_smem_doubled_bytes(BM, BN, BK, elem_bytes)

    def compute_load_ratio(self, BM, BN, BK, elem_bytes):
        return self.lib.oracle_compute_load_ratio(BM, BN, BK, elem_bytes)


_default = None


def default() -> Oracle:
    """The oracle built from gemm_oracle.c (compiled on first use)."""
    global _default
    if _default is None:
        _default = Oracle(load_library(build()))
    return _default


def gemm_s8s8s32(A, B, rows=None, threads=None, allow_overflow=False):
    return default().gemm_s8s8s32(A, B, rows, threads, allow_overflow)


def gemm_f16f32(A, B, rows=None, threads=None):
    return default().gemm_f16f32(A, B, rows, threads)


def f16_to_f64(bits: int) -> float:
    return default().f16_to_f64(bits)


def smem_a_bytes(BM: int, BK: int, elem_bytes: int) -> int:
    return default().smem_a_bytes(BM, BK, elem_bytes)


def smem_b_bytes(BK: int, BN: int, elem_bytes: int) -> int:
    return default().smem_b_bytes(BK, BN, elem_bytes)


def smem_doubled_bytes(BM: int, BN: int, BK: int, elem_bytes: int) -> int:
    return default().smem_doubled_bytes(BM, BN, BK, elem_bytes)


def compute_load_ratio(BM: int, BN: int, BK: int, elem_bytes: int) -> float:
    return default().compute_load_ratio(BM, BN, BK, elem_bytes)
