"""CPU oracle for the fused row softmax (FP64, one final cast).

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package. The CUDA
product path (``memory_bound_row_rows_gb300``) never imports it, and the two
share no code: ``softmax_oracle.c`` is self-contained plain C.

The definition it follows (row max, exponentiate, sum, divide; FP64, one
rounding to the dtype) is stated and cited at the top of ``softmax_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

F32, BF16, F16 = 0, 1, 2
_STORAGE = {F32: np.float32, BF16: np.uint16, F16: np.uint16}

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "softmax_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

CFLAGS = ["-O2", "-std=gnu11", "-fPIC", "-shared", "-pthread",
          "-ffp-contract=off", "-fno-fast-math"]


def compile_library(src: str, dst: str) -> str:
    """Compile an oracle source file into a shared library (also used on mutants)."""
    tmp = dst + ".tmp%d" % os.getpid()
    subprocess.check_call(["gcc", *CFLAGS, src, "-o", tmp, "-lm"])
    os.replace(tmp, dst)
    return dst


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(SOURCE):
        compile_library(SOURCE, _LIB)
    return _LIB


class Oracle:
    """ctypes view of one compiled oracle library (the real one, or a test mutant)."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        i64, c_int, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        for name in ("oracle_softmax_rows", "oracle_softmax_rows_f64"):
            fn = getattr(lib, name)
            fn.restype = c_int
            fn.argtypes = [vp, vp, i64, i64, i64, i64, c_int, c_int]
        fn = lib.oracle_softmax_rows_masked
        fn.restype = c_int
        fn.argtypes = [vp, vp, i64, i64, i64, i64, c_int, vp, i64, c_int]
        fn = lib.oracle_softmax_backward
        fn.restype = c_int
        fn.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, c_int]
        fn = lib.oracle_rmsnorm_residual
        fn.restype = c_int
        fn.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, ctypes.c_double, c_int]
        for name in ("oracle_cast", "oracle_decode"):
            fn = getattr(lib, name)
            fn.restype = c_int
            fn.argtypes = [vp, vp, i64, c_int]
        self.lib = lib

    def softmax_rows(self, x: np.ndarray, M: int, N: int, ld_in: int, ld_out: int,
                     dtype: int, out: np.ndarray | None = None, nthreads: int = 1) -> np.ndarray:
        """Softmax of the first N columns of each of M rows; returns an (M, ld_out) array.

        ``x`` holds M*ld_in elements of the dtype's storage type (float32, or uint16
        patterns for bf16/f16). Pad columns of a freshly made output are zero.
        """
        x = np.ascontiguousarray(x)
        assert x.dtype == _STORAGE[dtype] and x.size >= M * ld_in
        if out is None:
            out = np.zeros((M, ld_out), dtype=_STORAGE[dtype])
        assert out.flags["C_CONTIGUOUS"] and out.dtype == _STORAGE[dtype]
        rc = self.lib.oracle_softmax_rows(x.ctypes.data, out.ctypes.data, M, N, ld_in,
                                          ld_out, dtype, nthreads)
        if rc != 0:
            raise ValueError("oracle_softmax_rows returned %d" % rc)
        return out

    def softmax_rows_masked(self, x: np.ndarray, M: int, N: int, ld_in: int, ld_out: int,
                            dtype: int, lens=None, causal_period: int = 0,
                            nthreads: int = 1) -> np.ndarray:
        """Masked softmax (entries past each row's valid length are -inf, never read)."""
        x = np.ascontiguousarray(x)
        assert x.dtype == _STORAGE[dtype] and x.size >= M * ld_in
        out = np.zeros((M, ld_out), dtype=_STORAGE[dtype])
        lp = None
        if lens is not None:
            lens = np.ascontiguousarray(lens, dtype=np.int32)
            assert lens.size >= M
            lp = lens.ctypes.data
        rc = self.lib.oracle_softmax_rows_masked(x.ctypes.data, out.ctypes.data, M, N, ld_in,
                                                 ld_out, dtype, lp, causal_period, nthreads)
        if rc != 0:
            raise ValueError("oracle_softmax_rows_masked returned %d" % rc)
        return out

    def softmax_backward(self, y: np.ndarray, dy: np.ndarray, M: int, N: int, ld_y: int,
                         ld_dy: int, ld_dx: int, dtype: int) -> np.ndarray:
        """dx = y * (dy - sum(y * dy)) per row, FP64, one cast; an (M, ld_dx) array."""
        y = np.ascontiguousarray(y)
        dy = np.ascontiguousarray(dy)
        assert y.dtype == _STORAGE[dtype] and dy.dtype == _STORAGE[dtype]
        assert y.size >= M * ld_y and dy.size >= M * ld_dy
        dx = np.zeros((M, ld_dx), dtype=_STORAGE[dtype])
        rc = self.lib.oracle_softmax_backward(y.ctypes.data, dy.ctypes.data, dx.ctypes.data, M, N,
                                              ld_y, ld_dy, ld_dx, dtype)
        if rc != 0:
            raise ValueError("oracle_softmax_backward returned %d" % rc)
        return dx

    def rmsnorm_residual(self, x: np.ndarray, r: np.ndarray, w: np.ndarray, M: int, N: int,
                         ld_x: int, ld_r: int, ld_y: int, eps: float, dtype: int) -> np.ndarray:
        """y = dtype(h * w / sqrt(mean(h^2) + eps)), h = dtype(x + r); an (M, ld_y) array."""
        x, r, w = (np.ascontiguousarray(a) for a in (x, r, w))
        for a in (x, r, w):
            assert a.dtype == _STORAGE[dtype]
        assert x.size >= M * ld_x and r.size >= M * ld_r and w.size >= N
        y = np.zeros((M, ld_y), dtype=_STORAGE[dtype])
        rc = self.lib.oracle_rmsnorm_residual(x.ctypes.data, r.ctypes.data, w.ctypes.data,
                                              y.ctypes.data, M, N, ld_x, ld_r, ld_y, float(eps),
                                              dtype)
        if rc != 0:
            raise ValueError("oracle_rmsnorm_residual returned %d" % rc)
        return y

    def softmax_rows_f64(self, x: np.ndarray, M: int, N: int, ld_in: int, dtype: int,
                         nthreads: int = 1) -> np.ndarray:
        """The FP64 values before the final cast, as an (M, N) float64 array."""
        x = np.ascontiguousarray(x)
        assert x.dtype == _STORAGE[dtype] and x.size >= M * ld_in
        out = np.zeros((M, N), dtype=np.float64)
        rc = self.lib.oracle_softmax_rows_f64(x.ctypes.data, out.ctypes.data, M, N, ld_in,
                                              N, dtype, nthreads)
        if rc != 0:
            raise ValueError("oracle_softmax_rows_f64 returned %d" % rc)
        return out

    def cast(self, v: np.ndarray, dtype: int) -> np.ndarray:
        v = np.ascontiguousarray(v, dtype=np.float64)
        out = np.zeros(v.shape, dtype=_STORAGE[dtype])
        rc = self.lib.oracle_cast(v.ctypes.data, out.ctypes.data, v.size, dtype)
        if rc != 0:
            raise ValueError("oracle_cast returned %d" % rc)
        return out

    def decode(self, a: np.ndarray, dtype: int) -> np.ndarray:
        a = np.ascontiguousarray(a, dtype=_STORAGE[dtype])
        out = np.zeros(a.shape, dtype=np.float64)
        rc = self.lib.oracle_decode(a.ctypes.data, out.ctypes.data, a.size, dtype)
        if rc != 0:
            raise ValueError("oracle_decode returned %d" % rc)
        return out


def load() -> Oracle:
    global _lib
    if _lib is None:
        _lib = Oracle(build())
    return _lib


def softmax_rows(x, M, N, ld_in, ld_out, dtype, out=None, nthreads=1):
    return load().softmax_rows(x, M, N, ld_in, ld_out, dtype, out=out, nthreads=nthreads)


def softmax_rows_f64(x, M, N, ld_in, dtype, nthreads=1):
    return load().softmax_rows_f64(x, M, N, ld_in, dtype, nthreads=nthreads)
