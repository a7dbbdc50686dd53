"""Seeded synthetic inputs for the row-softmax workloads.

This module makes input matrices and nothing else: it holds none of the
softmax arithmetic. The CPU oracle tests, the CUDA parity tests and the
benchmark all draw their inputs from here. ``gen.c`` states the generator
(SplitMix64 + Box-Muller, counter-based, so any row range is generated
identically and independently of the thread count).

The five workloads are the logit and attention-score shapes the source pages
measure softmax on ("Fused Softmax on GPU: From Naive PyTorch to Persistent
Triton Kernels", Results; "Triton: Writing GPU Kernels in Python, Measured",
Step 2; "Measured optimization case studies", Wide rows), fixed here with
their value laws:

  f32_1024x256          N(0, 1)                                   seed 0
  f32_4096x4096         N(0, variance 4); rows i % 16 == 0 U[-100, 100)  seed 1
  bf16_16384x1000_ld1024  N(0, 1), input pitch 1024 (NaN pad), output pitch 1000  seed 2
  bf16_1024x131072      N(0, variance 2)                          seed 3
  f16_causal_524288x2048  N(0, 1)/sqrt(128); entry (r, j) = -inf when j > r mod 2048  seed 4
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from dataclasses import dataclass

import numpy as np

F32, BF16, F16 = 0, 1, 2
DTYPE_NAMES = {F32: "f32", BF16: "bf16", F16: "f16"}
ELEM_BYTES = {F32: 4, BF16: 2, F16: 2}
NP_STORAGE = {F32: np.float32, BF16: np.uint16, F16: np.uint16}

DIST_NORMAL, DIST_UNIFORM = 0, 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB = os.path.join(_HERE, "libsynth.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile gen.c into libsynth.so beside it (gcc, no fast-math, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(
            ["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", "-pthread",
             "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.synth_generate.restype = ctypes.c_int
        lib.synth_generate.argtypes = [
            ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_int, ctypes.c_uint64, ctypes.c_int, ctypes.c_double, ctypes.c_double,
            ctypes.c_int64, ctypes.c_double, ctypes.c_double,
            ctypes.c_int64, ctypes.c_int, ctypes.c_int]
        lib.synth_splitmix64_at.restype = ctypes.c_uint64
        lib.synth_splitmix64_at.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
        _lib = lib
    return _lib


def host_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def splitmix64_at(seed: int, k: int) -> int:
    """k-th output (k >= 0) of SplitMix64 seeded with ``seed``."""
    return int(_load().synth_splitmix64_at(seed & (2**64 - 1), k))


def generate_into(buf: np.ndarray, row0: int, M: int, N: int, ld: int, dtype: int, seed: int,
                  dist: int = DIST_NORMAL, p0: float = 0.0, p1: float = 1.0,
                  alt_every: int = 0, alt_lo: float = 0.0, alt_hi: float = 0.0,
                  causal_period: int = 0, pad_nan: bool = False, nthreads: int | None = None):
    """Fill ``buf`` (C-contiguous, >= M*ld elements) with rows [row0, row0+M) of the matrix."""
    assert buf.flags["C_CONTIGUOUS"] and buf.dtype == NP_STORAGE[dtype]
    assert buf.size >= M * ld
    rc = _load().synth_generate(
        buf.ctypes.data, row0, M, N, ld, dtype, seed & (2**64 - 1), dist, p0, p1,
        alt_every, alt_lo, alt_hi, causal_period, int(pad_nan),
        nthreads or host_threads())
    if rc != 0:
        raise ValueError("synth_generate rejected its arguments")
    return buf


def generate(M: int, N: int, ld: int | None = None, dtype: int = F32, seed: int = 0,
             row0: int = 0, **kw) -> np.ndarray:
    """An (M, ld) array in the dtype's storage type (uint16 bits for bf16/f16); pad columns 0."""
    ld = N if ld is None else ld
    buf = np.zeros((M, ld), dtype=NP_STORAGE[dtype])
    return generate_into(buf.reshape(-1), row0, M, N, ld, dtype, seed, **kw).reshape(M, ld)


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: int
    M: int
    N: int
    ld_in: int
    ld_out: int
    seed: int
    dist: int
    p0: float
    p1: float
    alt_every: int = 0
    alt_lo: float = 0.0
    alt_hi: float = 0.0
    causal_period: int = 0
    pad_nan: bool = False

    @property
    def elem_bytes(self) -> int:
        return ELEM_BYTES[self.dtype]

    @property
    def fused_bytes(self) -> int:
        """Algorithmic HBM bytes: one read and one write of each of the M x N elements."""
        return 2 * self.M * self.N * self.elem_bytes

    def gen_kwargs(self) -> dict:
        return dict(dist=self.dist, p0=self.p0, p1=self.p1, alt_every=self.alt_every,
                    alt_lo=self.alt_lo, alt_hi=self.alt_hi,
                    causal_period=self.causal_period, pad_nan=self.pad_nan)

    def with_rows(self, M: int) -> "Workload":
        """The same value law on the first M rows (a smaller parity case)."""
        d = dict(self.__dict__)
        d["M"] = M
        return Workload(**d)

    def rows(self, row0: int, count: int, nthreads: int | None = None) -> np.ndarray:
        """Rows [row0, row0+count) of the input matrix as a (count, ld_in) array."""
        count = max(0, min(count, self.M - row0))
        buf = np.zeros((count, self.ld_in), dtype=NP_STORAGE[self.dtype])
        if count:
            generate_into(buf.reshape(-1), row0, count, self.N, self.ld_in, self.dtype,
                          self.seed, nthreads=nthreads, **self.gen_kwargs())
        return buf

    def generate(self, nthreads: int | None = None) -> np.ndarray:
        """The whole M x ld_in input matrix."""
        return self.rows(0, self.M, nthreads)

    def generate_rows(self, row_ids, nthreads: int | None = 1) -> np.ndarray:
        """Selected rows, each exactly as it appears in the whole matrix."""
        out = np.zeros((len(row_ids), self.ld_in), dtype=NP_STORAGE[self.dtype])
        for k, r in enumerate(row_ids):
            out[k] = self.rows(int(r), 1, nthreads)[0]
        return out


WORKLOADS = {
    w.name: w
    for w in [
        Workload("f32_1024x256", F32, 1024, 256, 256, 256, 0, DIST_NORMAL, 0.0, 1.0),
        Workload("f32_4096x4096", F32, 4096, 4096, 4096, 4096, 1, DIST_NORMAL, 0.0, 2.0,
                 alt_every=16, alt_lo=-100.0, alt_hi=100.0),
        Workload("bf16_16384x1000_ld1024", BF16, 16384, 1000, 1024, 1000, 2, DIST_NORMAL,
                 0.0, 1.0, pad_nan=True),
        Workload("bf16_1024x131072", BF16, 1024, 131072, 131072, 131072, 3, DIST_NORMAL,
                 0.0, math.sqrt(2.0)),
        Workload("f16_causal_524288x2048", F16, 524288, 2048, 2048, 2048, 4, DIST_NORMAL,
                 0.0, 1.0 / math.sqrt(128.0), causal_period=2048),
    ]
}

# Few, wide rows (the wide-row shapes of "Measured optimization case studies",
# FP16, N(0, 1)), for the split plan.
WIDE_FEW = {
    w.name: w
    for w in [
        Workload("f16_4x32769", F16, 4, 32769, 32769, 32769, 5, DIST_NORMAL, 0.0, 1.0),
        Workload("f16_64x131072", F16, 64, 131072, 131072, 131072, 6, DIST_NORMAL, 0.0, 1.0),
        Workload("f16_128x32769", F16, 128, 32769, 32769, 32769, 7, DIST_NORMAL, 0.0, 1.0),
        Workload("f16_1024x16384", F16, 1024, 16384, 16384, 16384, 8, DIST_NORMAL, 0.0, 1.0),
        # Rows wider than a 16-block cluster's registers (800 KB, 1 MiB and 16 MiB).
        Workload("bf16_512x400008", BF16, 512, 400008, 400008, 400008, 11, DIST_NORMAL, 0.0,
                 1.0),
        Workload("bf16_128x524288", BF16, 128, 524288, 524288, 524288, 9, DIST_NORMAL, 0.0, 1.0),
        Workload("f32_32x4194304", F32, 32, 4194304, 4194304, 4194304, 10, DIST_NORMAL, 0.0,
                 1.0),
    ]
}

@dataclass(frozen=True)
class BackwardWorkload:
    """Inputs of the softmax backward: y (a stand-in for softmax output, U[0, 2/N),
    so rows sum to about one) and the incoming gradient dy ~ N(0, 1); both M x N
    with pitch ``ld``."""
    name: str
    dtype: int
    M: int
    N: int
    ld: int
    seed: int

    @property
    def elem_bytes(self) -> int:
        return ELEM_BYTES[self.dtype]

    @property
    def fused_bytes(self) -> int:
        """Algorithmic HBM bytes: y and dy read once, dx written once."""
        return 3 * self.M * self.N * self.elem_bytes

    def with_rows(self, M: int) -> "BackwardWorkload":
        d = dict(self.__dict__)
        d["M"] = M
        return BackwardWorkload(**d)

    def _rows(self, which: int, row0: int, count: int, nthreads=None) -> np.ndarray:
        count = max(0, min(count, self.M - row0))
        buf = np.zeros((count, self.ld), dtype=NP_STORAGE[self.dtype])
        if count:
            if which == 0:
                kw = dict(dist=DIST_UNIFORM, p0=0.0, p1=2.0 / self.N)
            else:
                kw = dict(dist=DIST_NORMAL, p0=0.0, p1=1.0)
            generate_into(buf.reshape(-1), row0, count, self.N, self.ld, self.dtype,
                          self.seed * 2 + which, nthreads=nthreads, **kw)
        return buf

    def y_rows(self, row0: int, count: int, nthreads=None) -> np.ndarray:
        return self._rows(0, row0, count, nthreads)

    def dy_rows(self, row0: int, count: int, nthreads=None) -> np.ndarray:
        return self._rows(1, row0, count, nthreads)


# Softmax-backward shapes: the FP16 training-step shapes of "Measured
# optimization case studies" (Training), plus the 4096 x 4096 FP32 square.
BACKWARD = {
    w.name: w
    for w in [
        BackwardWorkload("f16_16384x4096", F16, 16384, 4096, 4096, 20),
        BackwardWorkload("f32_4096x4096", F32, 4096, 4096, 4096, 21),
        BackwardWorkload("f16_64x131072", F16, 64, 131072, 131072, 22),
        BackwardWorkload("f16_4x32769", F16, 4, 32769, 32769, 23),
        BackwardWorkload("f16_512x4097", F16, 512, 4097, 4097, 24),
        BackwardWorkload("f16_1024x1024", F16, 1024, 1024, 1024, 25),
        BackwardWorkload("f16_32x127", F16, 32, 127, 127, 26),
    ]
}
BACKWARD_HEADLINE = "f16_16384x4096"

@dataclass(frozen=True)
class RmsNormWorkload:
    """Inputs of the residual RMSNorm: x ~ N(0, 1), residual ~ N(0, 1) (M x N,
    pitch ``ld``), weight ~ U[0.5, 1.5) (N), and eps."""
    name: str
    dtype: int
    M: int
    N: int
    ld: int
    seed: int
    eps: float = 1e-6

    @property
    def elem_bytes(self) -> int:
        return ELEM_BYTES[self.dtype]

    @property
    def fused_bytes(self) -> int:
        """Algorithmic HBM bytes: x and the residual read once, y written once, weights once."""
        return (3 * self.M * self.N + self.N) * self.elem_bytes

    def with_rows(self, M: int) -> "RmsNormWorkload":
        d = dict(self.__dict__)
        d["M"] = M
        return RmsNormWorkload(**d)

    def _rows(self, which: int, row0: int, count: int, nthreads=None) -> np.ndarray:
        count = max(0, min(count, self.M - row0))
        buf = np.zeros((count, self.ld), dtype=NP_STORAGE[self.dtype])
        if count:
            generate_into(buf.reshape(-1), row0, count, self.N, self.ld, self.dtype,
                          self.seed * 3 + which, nthreads=nthreads)
        return buf

    def x_rows(self, row0: int, count: int, nthreads=None) -> np.ndarray:
        return self._rows(0, row0, count, nthreads)

    def residual_rows(self, row0: int, count: int, nthreads=None) -> np.ndarray:
        return self._rows(1, row0, count, nthreads)

    def weight(self) -> np.ndarray:
        buf = np.zeros(self.N, dtype=NP_STORAGE[self.dtype])
        generate_into(buf, 0, 1, self.N, self.N, self.dtype, self.seed * 3 + 2,
                      dist=DIST_UNIFORM, p0=0.5, p1=1.5)
        return buf


# Residual RMSNorm shapes: the FP16 shapes of "Measured optimization case
# studies" (Residual RMSNorm) and the BF16 batch x hidden shapes of the
# "Warpline" README (K1).
RMSNORM = {
    w.name: w
    for w in [
        RmsNormWorkload("f16_16384x4096", F16, 16384, 4096, 4096, 30),
        RmsNormWorkload("bf16_16384x4096", BF16, 16384, 4096, 4096, 42),
        RmsNormWorkload("f16_1024x1024", F16, 1024, 1024, 1024, 31),
        RmsNormWorkload("f16_512x4097", F16, 512, 4097, 4097, 32),
        RmsNormWorkload("f16_32x127", F16, 32, 127, 127, 33),
        RmsNormWorkload("f16_4x32769", F16, 4, 32769, 32769, 34),
        RmsNormWorkload("f16_64x131072", F16, 64, 131072, 131072, 35),
        RmsNormWorkload("bf16_1x1024", BF16, 1, 1024, 1024, 36),
        RmsNormWorkload("bf16_8x1024", BF16, 8, 1024, 1024, 37),
        RmsNormWorkload("bf16_16x2048", BF16, 16, 2048, 2048, 38),
        RmsNormWorkload("bf16_32x4096", BF16, 32, 4096, 4096, 39),
        RmsNormWorkload("bf16_64x4096", BF16, 64, 4096, 4096, 40),
        RmsNormWorkload("bf16_64x8192", BF16, 64, 8192, 8192, 41),
    ]
}
RMSNORM_HEADLINE = "f16_16384x4096"

# The workload the headline throughput is quoted on: the largest, the FP16
# causal attention-score matrix (524288 x 2048, 4.29 GB moved per call).
HEADLINE = "f16_causal_524288x2048"


def storage_to_float64(a: np.ndarray, dtype: int) -> np.ndarray:
    """Decode storage (float32, or uint16 bits of bf16/f16) to float64, exactly."""
    if dtype == F32:
        return a.astype(np.float64)
    if dtype == BF16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    with np.errstate(invalid="ignore"):  # NaN payloads warn on some platforms
        return a.view(np.float16).astype(np.float64)
