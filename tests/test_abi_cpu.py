"""The C-ABI library without a GPU: it loads, exports every declared entry
point, and its host-side argument checks and plan choice behave as declared."""
import ctypes
import glob
import os
import re

import pytest

import memory_bound_row_rows_gb300 as sr
import synth
from memory_bound_row_rows_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return sr.load()


def declared_functions():
    names = set()
    for path in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(path).read()
        names |= set(re.findall(r"SR_API\s+[\w\s\*]+?\b(\w+)\s*\(", text))
    return sorted(names)


def test_header_declares_entry_points():
    names = declared_functions()
    for must in ("softmax_rows", "softmax_rows_ex", "softmax_rows_plan",
                 "softmax_rows_last_device_error", "softmax_rows_strerror"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    raw = ctypes.CDLL(sr.lib_path())
    missing = [n for n in declared_functions() if not hasattr(raw, n)]
    assert not missing, missing


def test_version_and_strerror(lib):
    assert sr.softmax_rows_version() >= 100
    for st in range(7):
        assert sr.softmax_rows_strerror(st)
    assert sr.softmax_rows_strerror(99) == "unknown status"


ALIGNED_IN, ALIGNED_OUT = 0x7F0000000000, 0x7F0100000000


def test_rejected_arguments_touch_no_device(lib):
    L = lib
    # No device exists here: each of these must return before any CUDA call.
    assert L.softmax_rows(None, None, 0, 8, 8, 8, 0, None) == sr.SR_OK  # empty
    assert L.softmax_rows(ALIGNED_IN, ALIGNED_OUT, 4, 0, 8, 8, 0, None) == sr.SR_EINVAL
    assert L.softmax_rows(ALIGNED_IN, ALIGNED_OUT, -1, 8, 8, 8, 0, None) == sr.SR_EINVAL
    assert L.softmax_rows(ALIGNED_IN, ALIGNED_OUT, 4, 8, 7, 8, 0, None) == sr.SR_EINVAL
    assert L.softmax_rows(ALIGNED_IN, ALIGNED_OUT, 4, 8, 8, 7, 0, None) == sr.SR_EINVAL
    assert L.softmax_rows(None, ALIGNED_OUT, 4, 8, 8, 8, 0, None) == sr.SR_EINVAL
    assert L.softmax_rows(ALIGNED_IN, None, 4, 8, 8, 8, 0, None) == sr.SR_EINVAL
    assert L.softmax_rows(ALIGNED_IN, ALIGNED_OUT, 4, 8, 8, 8, 3, None) == sr.SR_EDTYPE
    assert L.softmax_rows(ALIGNED_IN, ALIGNED_OUT, 2**40, 2**30, 2**30, 2**30, 0,
                          None) == sr.SR_EINVAL  # index arithmetic would overflow
    assert L.softmax_rows_ex(ALIGNED_IN, ALIGNED_OUT, 4, 4096, 4096, 4096, 0, sr.SR_PLAN_WARP,
                             None) == sr.SR_EPLAN
    assert L.softmax_rows_ex(ALIGNED_IN, ALIGNED_OUT, 4, 8, 8, 8, 0, 9, None) == sr.SR_EPLAN
    assert L.softmax_rows_ex(ALIGNED_IN, ALIGNED_OUT, 4, 8, 8, 8, 0, 8, None) == sr.SR_EPLAN
    assert L.softmax_rows_test_expiry(ALIGNED_IN, ALIGNED_OUT, 4, 8, 8, 8, 0, sr.SR_PLAN_WARP,
                                      1000, None) == sr.SR_EPLAN


EXPECTED_PLANS = {
    "f32_1024x256": sr.SR_PLAN_WARP,
    "f32_4096x4096": sr.SR_PLAN_ROW,
    "bf16_16384x1000_ld1024": sr.SR_PLAN_WARP,
    "bf16_1024x131072": sr.SR_PLAN_WIDE,
    "f16_causal_524288x2048": sr.SR_PLAN_ROW,
}


@pytest.mark.parametrize("name", sorted(EXPECTED_PLANS))
def test_plan_for_each_workload(lib, name):
    w = synth.WORKLOADS[name]
    got = sr.softmax_rows_plan(ALIGNED_IN, ALIGNED_OUT, w.M, w.N, w.ld_in, w.ld_out, w.dtype)
    assert got == EXPECTED_PLANS[name]


def test_plan_depends_on_alignment_and_width(lib):
    P = sr.softmax_rows_plan
    A, B = ALIGNED_IN, ALIGNED_OUT
    assert P(A, B, 10, 4096, 4096, 4096, 0) == sr.SR_PLAN_ROW
    assert P(A, B, 10, 1024, 1024, 1024, 0) == sr.SR_PLAN_ROW          # 256 vectors
    assert P(A, B, 10, 1020, 1020, 1020, 0) == sr.SR_PLAN_WARP         # 255 vectors
    assert P(A + 4, B, 10, 4096, 4096, 4096, 0) == sr.SR_PLAN_ONLINE   # misaligned input
    assert P(A, B, 10, 4096, 4097, 4096, 0) == sr.SR_PLAN_ONLINE       # odd pitch
    # Rows that share their offset from a 16-byte boundary (odd widths, equal
    # pitches, or bases equally misaligned) are read as shifted vectors: ROW up
    # to 64 KiB (FP32) or 32 KiB (16-bit), WIDE beyond.
    assert P(A, B, 4, 32769, 32769, 32769, 2) == sr.SR_PLAN_WIDE
    assert P(A + 4, B + 4, 10, 4096, 4097, 4097, 0) == sr.SR_PLAN_ROW
    assert P(A, B, 10, 4097, 4097, 4097, 2) == sr.SR_PLAN_ROW
    assert P(A + 4, B + 4, 10, 40000, 40001, 40001, 0) == sr.SR_PLAN_WIDE
    assert P(A + 2, B + 4, 10, 4096, 4096, 4096, 2) == sr.SR_PLAN_ONLINE  # not congruent
    assert P(A, B, 10, 8192, 8192, 8192, 0) == sr.SR_PLAN_ROW          # 32 KiB rows
    assert P(A, B, 10, 16384, 16384, 16384, 0) == sr.SR_PLAN_ROW       # 64 KiB f32 rows
    assert P(A, B, 10, 16388, 16388, 16388, 0) == sr.SR_PLAN_WIDE      # just over 64 KiB
    assert P(A, B, 10, 16384, 16384, 16384, 2) == sr.SR_PLAN_ROW       # 32 KiB f16 rows
    assert P(A, B, 10, 16392, 16392, 16392, 1) == sr.SR_PLAN_WIDE      # just over 32 KiB
    assert P(A, B, 10, 262144, 262144, 262144, 1) == sr.SR_PLAN_WIDE   # 512 KiB bf16
    assert P(A, B, 10, 262152, 262152, 262152, 1) == sr.SR_PLAN_WIDE   # streamed by a cluster
    assert P(A, B, 10, 1 << 24, 1 << 24, 1 << 24, 0) == sr.SR_PLAN_WIDE  # 64 MiB rows
    assert P(A + 2, B + 2, 10, 262152, 262153, 262153, 1) == sr.SR_PLAN_ONLINE  # shifted, too wide
    assert P(A, B, 10, 2048, 2048, 2048, 2) == sr.SR_PLAN_ROW
    assert P(A, B, 10, 2040, 2040, 2040, 2) == sr.SR_PLAN_WARP         # 255 vectors
    assert P(A + 2, B, 10, 2048, 2048, 2048, 2) == sr.SR_PLAN_WARP     # scalar warp variant
    assert P(A, B, 10, 0, 8, 8, 0) == -sr.SR_EINVAL
    assert P(A, B, 10, 8, 8, 8, 5) == -sr.SR_EDTYPE


def test_forced_plan_checks(lib):
    C = sr.softmax_rows_plan_check
    A, B = ALIGNED_IN, ALIGNED_OUT
    assert C(A, B, 5, 4096, 4096, 4096, 0, sr.SR_PLAN_CLUSTER) == sr.SR_PLAN_CLUSTER
    assert C(A, B, 5, 4096, 4096, 4096, 0, sr.SR_PLAN_WARP) == -sr.SR_EPLAN
    assert C(A, B, 5, 131072, 131072, 131072, 1, sr.SR_PLAN_CTA) == -sr.SR_EPLAN
    assert C(A + 2, B, 5, 1000, 1000, 1000, 1, sr.SR_PLAN_CTA) == -sr.SR_EPLAN
    assert C(A + 2, B, 5, 1000, 1000, 1000, 1, sr.SR_PLAN_ONLINE) == sr.SR_PLAN_ONLINE
    assert C(A, B, 5, 8, 8, 8, 1, sr.SR_PLAN_CLUSTER) == -sr.SR_EPLAN  # one vector per row
    assert C(A, B, 5, 8, 8, 8, 1, sr.SR_PLAN_SMEM) == sr.SR_PLAN_SMEM
    assert C(A, B, 5, 16384, 16384, 16384, 1, sr.SR_PLAN_SMEM) == sr.SR_PLAN_SMEM
    assert C(A, B, 5, 16392, 16392, 16392, 1, sr.SR_PLAN_SMEM) == -sr.SR_EPLAN  # > 32 KiB
    assert C(A, B, 5, 8, 8, 8, 1, 8) == -sr.SR_EPLAN  # no such plan
    assert C(A, B, 5, 8, 8, 8, 1, sr.SR_PLAN_WIDE) == sr.SR_PLAN_WIDE
    assert C(A, B, 5, 131072, 131072, 131072, 1, sr.SR_PLAN_WIDE) == sr.SR_PLAN_WIDE
    assert C(A, B, 5, 262144, 262144, 262144, 1, sr.SR_PLAN_WIDE) == sr.SR_PLAN_WIDE  # 512 KiB
    assert C(A, B, 5, 262152, 262152, 262152, 1, sr.SR_PLAN_WIDE) == sr.SR_PLAN_WIDE  # streamed
    assert C(A + 2, B + 2, 5, 262152, 262153, 262153, 1, sr.SR_PLAN_WIDE) == -sr.SR_EPLAN
    assert C(A + 2, B, 5, 131072, 131072, 131072, 1, sr.SR_PLAN_WIDE) == -sr.SR_EPLAN
    assert C(A, B, 5, 4096, 4096, 4096, 0, sr.SR_PLAN_ROW) == sr.SR_PLAN_ROW
    assert C(A, B, 5, 16384, 16384, 16384, 1, sr.SR_PLAN_ROW) == sr.SR_PLAN_ROW
    assert C(A, B, 5, 16392, 16392, 16392, 1, sr.SR_PLAN_ROW) == -sr.SR_EPLAN
    assert C(A + 2, B, 5, 4096, 4096, 4096, 1, sr.SR_PLAN_ROW) == -sr.SR_EPLAN
    assert C(A + 2, B + 2, 5, 4096, 4096, 4096, 1, sr.SR_PLAN_ROW) == sr.SR_PLAN_ROW  # shifted


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setenv("SOFTMAX_ROWS_LIB", str(tmp_path / "absent.so"))
    monkeypatch.setattr(sr, "_lib", None)
    with pytest.raises(RuntimeError, match="not found"):
        sr.softmax_rows(1, 2, 1, 8, 8, 8, 0, 0)


def test_split_workspace_is_host_logic(lib):
    A, B = ALIGNED_IN, ALIGNED_OUT
    W = sr.softmax_rows_split_workspace_bytes
    # A fixed size: four steps of tagged 16-byte pairs for up to 4096 blocks.
    for args in [(4, 32769, 32769, 32769, 2), (64, 131072, 131072, 131072, 2),
                 (100000, 64, 64, 64, 1), (32, 1 << 22, 1 << 22, 1 << 22, 0)]:
        assert W(A, B, *args) == 4 * 4096 * 16 == 262144
    assert W(A, B, 4, 0, 8, 8, 0) == -sr.SR_EINVAL
    assert W(A, B, 4, 8, 8, 8, 9) == -sr.SR_EDTYPE
    L = lib
    assert L.softmax_rows_split(A, B, 0, 8, 8, 8, 0, None, 0, None) == sr.SR_OK
    assert L.softmax_rows_split(A, B, 4, 8, 8, 8, 0, None, 1024, None) == sr.SR_EINVAL
    assert L.softmax_rows_split(A, B, 4, 8, 8, 8, 0, A + 4096, 262144 - 16, None) == sr.SR_EINVAL


# A device holding 608 blocks of the split kernel, with a 126.5 MiB L2 (half:
# 66322432 bytes).
SPLIT_BLOCKS, SPLIT_L2 = 608, 132644864


@pytest.mark.parametrize("M,N,dtype,aligned,expect", [
    # 16 MiB rows: three of them exceed half the L2 -> one group of all 608 blocks;
    # 1048576 vectors in parts of ceil(1048576 / 608) = 1725.
    (32, 1 << 22, 0, True, (1, 608, 1725, 4)),
    # 1 MiB rows: the L2 allows 66322432 // (3 * 1048576) = 21 groups, eight rows
    # per group allow 128 // 8 = 16; 608 // 16 = 38 blocks; 65536 vectors -> 1725 x 38.
    (128, 1 << 19, 1, True, (16, 38, 1725, 8)),
    # 64 rows of 256 KiB (16 MiB: fits in half the L2): a group per row, 608 // 64 = 9
    # blocks each; 16384 vectors -> 1821 x 9.
    (64, 131072, 2, True, (64, 9, 1821, 8)),
    # Four unaligned rows of 32769 f16: a group per row of 152 blocks, but no part
    # under 256 elements -> 129 parts of 255 elements.
    (4, 32769, 2, False, (4, 129, 255, 1)),
    # Many short rows (25.6 MB): a group per block, one part per row.
    (100000, 64, 0, True, (608, 1, 16, 4)),
    # Three rows of 250 vectors: a group per row, one part.
    (3, 1000, 0, True, (3, 1, 250, 4)),
])
def test_split_shape_is_host_logic(lib, M, N, dtype, aligned, expect):
    A, B = ALIGNED_IN, ALIGNED_OUT
    if not aligned:
        B += 2
    sh = sr.softmax_rows_split_shape(A, B, M, N, N, N, dtype, SPLIT_BLOCKS, SPLIT_L2)
    assert (sh["lanes"], sh["parts"], sh["part_units"], sh["unit_elems"]) == expect
    # Every part non-empty, the parts cover the row, and the grid fits the device.
    units = N // sh["unit_elems"]
    assert (sh["parts"] - 1) * sh["part_units"] < units <= sh["parts"] * sh["part_units"]
    assert sh["lanes"] * sh["parts"] <= SPLIT_BLOCKS and sh["lanes"] <= M


def test_split_shape_caps_and_errors(lib):
    A, B = ALIGNED_IN, ALIGNED_OUT
    sh = sr.softmax_rows_split_shape(A, B, 8, 1 << 22, 1 << 22, 1 << 22, 0, 100000, SPLIT_L2)
    assert sh["lanes"] * sh["parts"] <= 4096  # the workspace's block limit
    with pytest.raises(sr.SoftmaxRowsError):
        sr.softmax_rows_split_shape(A, B, 8, 0, 8, 8, 0, SPLIT_BLOCKS, SPLIT_L2)
    assert lib.softmax_rows_split_shape(A, B, 8, 64, 64, 64, 0, SPLIT_BLOCKS, SPLIT_L2,
                                        None) == sr.SR_EINVAL


ALIGNED_DY = 0x7F0200000000


def test_backward_rejected_arguments_touch_no_device(lib):
    L = lib
    y, g, x = ALIGNED_IN, ALIGNED_DY, ALIGNED_OUT
    assert L.softmax_rows_backward(None, None, None, 0, 8, 8, 8, 8, 0, None) == sr.SR_OK
    assert L.softmax_rows_backward(y, g, x, 4, 0, 8, 8, 8, 0, None) == sr.SR_EINVAL
    assert L.softmax_rows_backward(y, g, x, -1, 8, 8, 8, 8, 0, None) == sr.SR_EINVAL
    for lds in ((7, 8, 8), (8, 7, 8), (8, 8, 7)):
        assert L.softmax_rows_backward(y, g, x, 4, 8, *lds, 0, None) == sr.SR_EINVAL
    assert L.softmax_rows_backward(y, None, x, 4, 8, 8, 8, 8, 0, None) == sr.SR_EINVAL
    assert L.softmax_rows_backward(y, g, y, 4, 8, 8, 8, 8, 0, None) == sr.SR_EINVAL  # dx is y
    assert L.softmax_rows_backward(y, g, g, 4, 8, 8, 8, 8, 0, None) == sr.SR_EINVAL  # dx is dy
    assert L.softmax_rows_backward(y, g, x, 4, 8, 8, 8, 8, 3, None) == sr.SR_EDTYPE
    assert L.softmax_rows_backward(y, g, x, 2**40, 2**30, 2**30, 2**30, 2**30, 0,
                                   None) == sr.SR_EINVAL  # last byte beyond int64
    assert L.softmax_rows_backward_ex(y, g, x, 4, 8, 8, 8, 8, 0, 9, None) == sr.SR_EPLAN
    assert L.softmax_rows_backward_ex(y, g, x, 0, 8, 8, 8, 8, 0, sr.SR_PLAN_WARP,
                                      None) == sr.SR_EPLAN
    # Empty, with a plan that takes the shape: nothing is launched.
    assert L.softmax_rows_backward_ex(y, g, x, 0, 8, 8, 8, 8, 0, sr.SR_PLAN_ROW,
                                      None) == sr.SR_OK


def _bwd_plan(M, N, dtype, plan=sr.SR_PLAN_AUTO, sm=152, ld=None, offset=0):
    ld = N if ld is None else ld
    return sr.softmax_rows_backward_plan(ALIGNED_IN + offset, ALIGNED_DY, ALIGNED_OUT, M, N, ld,
                                         ld, ld, dtype, plan, sm)


def test_backward_plan_choice(lib):
    F32, BF16, F16 = sr.SR_F32, sr.SR_BF16, sr.SR_F16
    ROW, CL, ON = sr.SR_PLAN_ROW, sr.SR_PLAN_CLUSTER, sr.SR_PLAN_ONLINE
    # Many rows that fit one team: ROW.
    assert _bwd_plan(4096, 4096, F32) == ROW
    assert _bwd_plan(16384, 4096, F16) == ROW
    assert _bwd_plan(1024, 1024, F16) == ROW
    assert _bwd_plan(32, 127, F16) == ROW          # short rows, even if few
    assert _bwd_plan(512, 4097, F16) == ROW        # unaligned, 4097 elements
    # Team limits: 16384 elements of any dtype when aligned, 8192 unaligned.
    assert _bwd_plan(1024, 16384, F32, ROW) == ROW
    assert _bwd_plan(1024, 16384, F16, ROW) == ROW
    assert _bwd_plan(1024, 16392, F16, ROW) == -sr.SR_EPLAN
    # Odd widths with the same pitch in all three matrices: rows share their
    # offset from a 16-byte boundary and are loaded as vectors.
    assert _bwd_plan(1024, 8193, F16, ROW) == ROW
    assert _bwd_plan(1024, 16391, F16, ROW) == ROW
    # Incongruent layouts (y 2 bytes off, dy and dx aligned) load elements:
    # 8192 elements per team at most.
    assert _bwd_plan(1024, 8192, F16, ROW, offset=2) == ROW
    assert _bwd_plan(1024, 8193, F16, ROW, offset=2) == -sr.SR_EPLAN
    # Wide or few rows: CLUSTER; beyond its limit: ONLINE.
    assert _bwd_plan(64, 131072, F16) == CL
    assert _bwd_plan(4, 32769, F16) == CL
    assert _bwd_plan(1024, 131072, BF16) == CL
    assert _bwd_plan(8, 4096, F32) == CL           # too few rows for one team each
    assert _bwd_plan(64, 131080, F16) == CL        # aligned: streamed by a cluster
    assert _bwd_plan(64, 131080, F16, offset=2) == ON
    # Rows that would need a 512-thread team run on CLUSTER.
    assert _bwd_plan(4096, 16384, F16) == CL
    assert _bwd_plan(1024, 16384, F32) == CL
    assert _bwd_plan(16384, 8192, F32) == CL
    assert _bwd_plan(16384, 4096, BF16) == ROW
    assert _bwd_plan(4, 65537, F16) == CL
    assert _bwd_plan(4, 65537, F16, offset=2) == ON
    assert _bwd_plan(4, 65536, F16, offset=2) == CL
    assert _bwd_plan(64, 131080, F16, CL) == CL
    assert _bwd_plan(64, 131080, F16, CL, offset=2) == -sr.SR_EPLAN
    # ONLINE takes anything.
    assert _bwd_plan(3, 1 << 22, F32, ON) == ON
    # A misaligned y base makes every row unaligned (element units).
    assert _bwd_plan(1024, 16384, F16, ROW, offset=2) == -sr.SR_EPLAN
    # Query errors.
    assert _bwd_plan(4, 8, 7) == -sr.SR_EDTYPE
    assert _bwd_plan(4, 8, F32, plan=sr.SR_PLAN_SMEM) == -sr.SR_EPLAN


def test_rmsnorm_rejected_arguments_touch_no_device(lib):
    L = lib
    x, r, y, w = ALIGNED_IN, ALIGNED_DY, ALIGNED_OUT, 0x7F0300000000
    ok = (x, r, w, y, 4, 8, 8, 8, 8)
    assert L.rmsnorm_residual_rows(None, None, None, None, 0, 8, 8, 8, 8, 1e-6, 0, None) == sr.SR_OK
    assert L.rmsnorm_residual_rows(*ok, 1e-6, 3, None) == sr.SR_EDTYPE
    assert L.rmsnorm_residual_rows(x, r, None, y, 4, 8, 8, 8, 8, 1e-6, 0, None) == sr.SR_EINVAL
    assert L.rmsnorm_residual_rows(x, r, w + 1, y, 4, 8, 8, 8, 8, 1e-6, 1, None) == sr.SR_EINVAL
    assert L.rmsnorm_residual_rows(x, r, w, x, 4, 8, 8, 8, 8, 1e-6, 0, None) == sr.SR_EINVAL
    assert L.rmsnorm_residual_rows(x, r, w, r, 4, 8, 8, 8, 8, 1e-6, 0, None) == sr.SR_EINVAL
    assert L.rmsnorm_residual_rows(x, r, w, y, 4, 8, 7, 8, 8, 1e-6, 0, None) == sr.SR_EINVAL
    for eps in (-1.0, float("nan"), float("inf")):
        assert L.rmsnorm_residual_rows(*ok, eps, 0, None) == sr.SR_EINVAL
    assert L.rmsnorm_residual_rows_ex(*ok, 1e-6, 0, sr.SR_PLAN_SMEM, None) == sr.SR_EPLAN
    assert sr.rmsnorm_residual_rows_plan(*ok, 1e-6, 0, sr.SR_PLAN_AUTO, 152) == sr.SR_PLAN_ROW
    assert sr.rmsnorm_residual_rows_plan(x, r, w, y, 64, 131072, 131072, 131072, 131072, 1e-6,
                                         2, sr.SR_PLAN_AUTO, 152) == sr.SR_PLAN_CLUSTER


def test_host_mapped_refuses_without_a_device(lib):
    # No device here: the pointer check fails and nothing is launched.
    assert lib.softmax_rows_host_mapped(ALIGNED_IN, ALIGNED_OUT, 4, 8, 8, 8, 0, None) == \
        sr.SR_EINVAL
    assert lib.softmax_rows_host_mapped(None, None, 0, 8, 8, 8, 0, None) == sr.SR_OK
    assert lib.softmax_rows_host_mapped(ALIGNED_IN, ALIGNED_OUT, 4, 8, 7, 8, 0, None) == \
        sr.SR_EINVAL


def test_wide_shapes(lib):
    """The WIDE plan's launch shape (host logic, 152 SMs)."""
    S = lambda M, N, dt: sr.softmax_rows_wide_shape(M, N, dt, 152)
    # bf16 1024 x 131072: 8-block clusters, 2048 vectors per block, 8 per thread.
    assert S(1024, 131072, 1) == {"csize": 8, "kv": 8, "slice": 2048, "streamed": False}
    # Few rows: clusters grow (up to 8) while each thread keeps a vector.
    assert S(4, 32769, 2)["csize"] == 8
    assert S(64, 131072, 2) == {"csize": 8, "kv": 8, "slice": 2048, "streamed": False}
    # Slices that would half fill 8 vectors per thread take the 5- and 6-vector kernels.
    assert S(4096, 16392, 1) == {"csize": 2, "kv": 5, "slice": 1025, "streamed": False}
    assert S(2730, 24576, 2) == {"csize": 2, "kv": 6, "slice": 1536, "streamed": False}
    assert S(2048, 16388, 0) == {"csize": 4, "kv": 5, "slice": 1025, "streamed": False}
    # 512 KiB is the most 16 blocks hold in registers; rows of exactly 1 MiB
    # are staged (kv 16: 8 vectors per thread in registers, 8 in shared
    # memory), other wider rows are streamed.
    assert S(256, 262144, 1) == {"csize": 16, "kv": 8, "slice": 2048, "streamed": False}
    assert S(128, 524288, 1) == {"csize": 16, "kv": 16, "slice": 4096, "streamed": False}
    assert S(128, 262144, 0) == {"csize": 16, "kv": 16, "slice": 4096, "streamed": False}
    assert S(128, 262152, 1) == {"csize": 8, "kv": 0, "slice": 4097, "streamed": True}
    assert S(128, 524296, 1) == {"csize": 8, "kv": 0, "slice": 8193, "streamed": True}
    # Streamed rows too few for a wave of 8-block clusters double to 16.
    assert S(32, 4194304, 0) == {"csize": 16, "kv": 0, "slice": 65536, "streamed": True}
    for bad in ((4, 0, 1, 152), (-1, 8, 1, 152), (4, 8, 9, 152), (4, 8, 1, 0)):
        with pytest.raises(sr.SoftmaxRowsError):
            sr.softmax_rows_wide_shape(*bad)


def test_host_workspace_is_host_logic(lib):
    """Workspace for full pipeline depth: 4 slots of up to 8 MiB of input rows
    (rows padded to 16 bytes on the device), input and output per slot."""
    W = sr.softmax_rows_host_workspace_bytes
    # f32 4096 x 4096: 512 rows of 16 KiB make 8 MiB.
    assert W(4096, 4096, 0) == 4 * 512 * 2 * 4096 * 4
    # Fewer rows than a chunk: the chunk shrinks to the matrix.
    assert W(10, 4096, 0) == 4 * 10 * 2 * 4096 * 4
    # bf16 1000 columns pad to 1000 (2000 bytes is a multiple of 16); 1001 to 1008.
    assert W(16384, 1000, 1) == 4 * ((8 << 20) // 2000) * 2 * 1000 * 2
    assert W(16384, 1001, 1) == 4 * ((8 << 20) // 2016) * 2 * 1008 * 2
    # A row larger than the chunk target still gets one row per slot.
    assert W(4, 4 << 20, 0) == 4 * 1 * 2 * (4 << 20) * 4
    assert W(4, 8, 9) == -sr.SR_EDTYPE
    assert W(-1, 8, 0) == -sr.SR_EINVAL


def test_last_launch_without_a_launch(lib):
    # No kernel has been launched from a fresh host thread: nothing to describe.
    import threading
    got = []
    th = threading.Thread(target=lambda: got.append(
        lib.softmax_rows_last_launch(ctypes.byref(sr.LaunchInfo()))))
    th.start()
    th.join()
    assert got == [sr.SR_EINVAL]
    assert lib.softmax_rows_last_launch(None) == sr.SR_EINVAL


def test_product_build_flags(lib):
    # The product library is not the bounds-checking build; its hooks refuse.
    assert lib.softmax_rows_build_flags() == 0
    assert lib.softmax_rows_test_bounds_shrink(8) == sr.SR_EINVAL
    assert sr.softmax_rows_strerror(sr.SR_EBOUNDS).startswith("a device access")


def test_copy_ceiling_rejects_before_any_device_call(lib):
    C = lib.softmax_rows_copy_ceiling
    assert C(None, None, 0, 16, 16, 16, None) == sr.SR_OK
    assert C(ALIGNED_IN, ALIGNED_OUT, -1, 16, 16, 16, None) == sr.SR_EINVAL
    assert C(ALIGNED_IN, ALIGNED_OUT, 4, 0, 16, 16, None) == sr.SR_EINVAL
    assert C(ALIGNED_IN, ALIGNED_OUT, 4, 32, 16, 32, None) == sr.SR_EINVAL
    assert C(ALIGNED_IN, ALIGNED_OUT, 4, 32, 32, 31, None) == sr.SR_EINVAL
    assert C(None, ALIGNED_OUT, 4, 32, 32, 32, None) == sr.SR_EINVAL
    assert C(ALIGNED_IN, ALIGNED_OUT, 2, 16, 2**63 - 8, 16, None) == sr.SR_EINVAL


def test_copy_ceiling2_rejects_before_any_device_call(lib):
    C = lib.softmax_rows_copy_ceiling2
    A, B, O = ALIGNED_IN, ALIGNED_OUT, ALIGNED_DY
    assert C(None, None, None, 0, 16, 16, 16, 16, None) == sr.SR_OK
    assert C(A, B, O, -1, 16, 16, 16, 16, None) == sr.SR_EINVAL
    assert C(A, B, O, 4, 0, 16, 16, 16, None) == sr.SR_EINVAL
    assert C(A, B, O, 4, 32, 16, 32, 32, None) == sr.SR_EINVAL
    assert C(A, B, O, 4, 32, 32, 31, 32, None) == sr.SR_EINVAL
    assert C(A, B, O, 4, 32, 32, 32, 31, None) == sr.SR_EINVAL
    assert C(A, None, O, 4, 32, 32, 32, 32, None) == sr.SR_EINVAL
    assert C(A, B, None, 4, 32, 32, 32, 32, None) == sr.SR_EINVAL
    assert C(A, B, O, 2, 16, 16, 2**63 - 8, 16, None) == sr.SR_EINVAL
