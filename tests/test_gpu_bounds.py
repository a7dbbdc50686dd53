"""The bounds-checking build (libsoftmax_rows_check.so): every kernel checks
each global load, store and bulk copy against the matrices of its call and
refuses, and reports, any access outside them.

Here a representative part of the GPU suite runs on that build (every plan on
every workload's value law, the edge and misaligned widths, special rows, in
place, masked, split, backward and RMSNorm calls); each must match the oracle
as before and leave the error word clear. A positive control shrinks the
writable extents by a few bytes: the checker must then refuse the last stores
of a correct kernel, report SR_EBOUNDS and the first refused address, and
leave those elements unwritten. The refused accesses are inside the caller's
buffers, so the control cannot touch invalid memory whatever happens. The
whole suite runs on the checking build with SOFTMAX_ROWS_LIB set to it (the
conftest then checks the error word after every test).
"""
import inspect

import numpy as np
import pytest

import memory_bound_row_rows_gb300 as sr
import oracle
import synth
from memory_bound_row_rows_gb300 import _build
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

from tests import test_gpu_backward as tb  # noqa: E402
from tests import test_gpu_masked as tm  # noqa: E402
from tests import test_gpu_parity as tp  # noqa: E402
from tests import test_gpu_rmsnorm as tr  # noqa: E402
from tests import test_gpu_split as ts  # noqa: E402


@pytest.fixture(scope="module")
def checked():
    """Route the binding to the checking build for this module's tests."""
    lib = sr.open_library(_build.build_checked())
    assert lib.softmax_rows_build_flags() == sr.SR_BUILD_BOUNDS_CHECK
    saved = sr._lib
    sr._lib = lib
    yield lib
    sr._lib = saved


def _clean(lib):
    st = lib.softmax_rows_last_device_error(None)
    addr = lib.softmax_rows_bounds_address()
    assert st == sr.SR_OK, "%s (first refused address 0x%x)" % (sr.softmax_rows_strerror(st), addr)


def test_product_build_checks_nothing():
    lib = sr.open_library(_build.LIB)
    assert lib.softmax_rows_build_flags() == 0
    assert lib.softmax_rows_bounds_address() == 0
    assert lib.softmax_rows_test_bounds_shrink(8) == sr.SR_EINVAL


@pytest.mark.parametrize("name,row0,rows", tp.SMALL_CASES, ids=lambda v: str(v))
@pytest.mark.parametrize("plan", tp.PLANS, ids=lambda p: sr.PLAN_NAMES[p])
def test_every_plan_inside(checked, name, row0, rows, plan):
    tp.test_small_parity(name, row0, rows, plan)
    _clean(checked)


@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16, synth.F16], ids=["f32", "bf16", "f16"])
@pytest.mark.parametrize("N", [1, 7, 33, 255, 1000, 2048, 4097, 16392, 40000])
def test_edge_widths_inside(checked, dtype, N):
    tp.test_edge_shapes(dtype, N)
    _clean(checked)


@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16, synth.F16], ids=["f32", "bf16", "f16"])
@pytest.mark.parametrize("N", [100, 5000, 40000])
def test_misaligned_and_special_inside(checked, dtype, N):
    tp.test_misaligned_rows(dtype, N)
    tp.test_special_rows(dtype, N)
    _clean(checked)


def test_wide_streamed_in_place_guards_inside(checked):
    tp.test_wide_shifted_rows(synth.BF16, 32769, 4)
    tp.test_streamed_wide_rows(synth.BF16, 3, 600008)
    tp.test_wide_staged_rows(synth.F16, 3, 524288, 16)
    tp.test_wide_staged_in_place()
    tp.test_in_place("bf16_16384x1000_ld1024")
    tp.test_guard_regions_untouched()
    _clean(checked)


def test_other_entry_points_inside(checked):
    for name, fn in [(n, getattr(m, n)) for m in (tm, ts, tb, tr) for n in dir(m)
                     if n.startswith("test_") and not hasattr(getattr(m, n), "pytestmark")]:
        if inspect.signature(fn).parameters:
            continue  # parametrised tests are run by their own modules
        fn()
        _clean(checked)


def test_checker_refuses_stores_past_a_shrunken_extent(checked):
    lib = checked
    for dtype, plan, N in [(synth.F32, sr.SR_PLAN_ROW, 4096), (synth.BF16, sr.SR_PLAN_ONLINE, 1001),
                           (synth.F16, sr.SR_PLAN_WARP, 1000)]:
        M = 8
        x = synth.generate(M, N, dtype=dtype, seed=77)
        xd = gu.to_device(x, dtype)
        y = torch.full((M, N), float("nan"), dtype=gu.torch_dtype(dtype), device="cuda")
        es = synth.ELEM_BYTES[dtype]
        assert lib.softmax_rows_test_bounds_shrink(es) == sr.SR_OK  # the last element is outside
        try:
            st = lib.softmax_rows_ex(xd.data_ptr(), y.data_ptr(), M, N, N, N, dtype, plan,
                                     torch.cuda.current_stream().cuda_stream)
            assert st == sr.SR_OK
            assert lib.softmax_rows_last_device_error(None) == sr.SR_EBOUNDS
            addr = lib.softmax_rows_bounds_address()
        finally:
            assert lib.softmax_rows_test_bounds_shrink(0) == sr.SR_OK
        base = y.data_ptr()
        assert base <= addr < base + M * N * es
        row, col = divmod((addr - base) // es, N)
        # a scalar store is refused at the last element, a vector store at the last vector
        assert N - (16 // es) <= col < N, (row, col)
        g = synth.storage_to_float64(gu.to_host(y, dtype), dtype)
        assert np.isnan(g[:, col:]).all(), "a refused store was executed"
        # every row before the refused columns is the softmax
        ref = synth.storage_to_float64(oracle.softmax_rows(x.reshape(-1), M, N, N, N, dtype),
                                       dtype)
        ok, nbad, _ = gu.gate(g[:, :col], ref[:, :col], dtype)
        assert ok, nbad
    # exact extents again: nothing refused
    tp.test_small_parity("f32_4096x4096", 0, 8, sr.SR_PLAN_ROW)
    _clean(lib)
