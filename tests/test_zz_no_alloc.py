"""softmax_rows_split_noalloc: the split plan for callers that cannot allocate
device memory (fixed memory budgets, foreign memory pools, code that must not
trigger the implicit device synchronisation of a cudaMalloc). Its statistics
live in scratch built into the library instead of a caller workspace.

Each check calls the allocation-free entry point through the C ABI on two
calls in a row on different data (the built-in scratch keeps the previous
call's contents) and compares its output with the CPU oracle at the parity
tolerance (and the 1-ulp diagnostic of the 16-bit types), and with the
workspace entry point (softmax_rows_split) on the same input: the two run the
same kernel on the same cut of the rows, so their outputs agree bit for bit.
The split plan's workspace has a fixed size, so the built-in scratch takes
every problem. This file is collected last so that a run stopping at its
first failure has already run every other test; it also passes on its own in
a fresh process.
"""
import numpy as np
import pytest

import memory_bound_row_rows_gb300 as sr
import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

def _with_workspace(xd, M, N, ld_in, ld_out, dtype):
    y = torch.full((M, ld_out), float("nan"), dtype=xd.dtype, device="cuda")
    need = sr.softmax_rows_split_workspace_bytes(xd, y, M, N, ld_in, ld_out, dtype)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    sr.softmax_rows_split(xd, y, M, N, ld_in, ld_out, dtype, ws, need)
    return y


def _no_alloc(xd, M, N, ld_in, ld_out, dtype):
    y = torch.full((M, ld_out), float("nan"), dtype=xd.dtype, device="cuda")
    st = sr.load().softmax_rows_split_noalloc(xd.data_ptr(), y.data_ptr(), M, N, ld_in, ld_out,
                                              dtype, torch.cuda.current_stream().cuda_stream)
    assert st == sr.SR_OK, sr.softmax_rows_strerror(st)
    return y


@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16, synth.F16], ids=["f32", "bf16", "f16"])
def test_no_alloc_matches_workspace_entry_point_twice(dtype):
    shapes = [(4, 32769, 32769, 32769), (37, 12345, 12350, 12345)]
    for call, (M, N, ld_in, ld_out) in enumerate(shapes):
        x = synth.generate(M, N, ld=ld_in, dtype=dtype, seed=1000 + 17 * call + dtype, p1=2.5)
        xd = gu.to_device(x, dtype)
        ref = _with_workspace(xd, M, N, ld_in, ld_out, dtype)
        got = _no_alloc(xd, M, N, ld_in, ld_out, dtype)
        torch.cuda.synchronize()
        got_h = gu.to_host(got, dtype)
        gu.check_rows(got_h, x, N, ld_in, dtype, "no-alloc call %d" % call)
        assert np.array_equal(got_h[:, :N], gu.to_host(ref, dtype)[:, :N]), (
            "call %d: output differs from softmax_rows_split" % call)
        assert torch.isnan(got[:, N:]).all() if ld_out > N else True


def test_no_alloc_takes_many_rows_and_wide_rows():
    # 70000 short rows (one group per block, many rows per group) and 16 MiB
    # rows (one group of every block): the fixed scratch serves both.
    for M, N, dtype, seed in [(70000, 64, synth.F16, 5), (3, 1 << 22, synth.F32, 6)]:
        x = synth.generate(M, N, dtype=dtype, seed=seed, p1=2.0)
        xd = gu.to_device(x, dtype)
        assert sr.softmax_rows_split_workspace_bytes(xd, xd, M, N, N, N, dtype) == 262144
        ref = _with_workspace(xd, M, N, N, N, dtype)
        got = _no_alloc(xd, M, N, N, N, dtype)
        torch.cuda.synchronize()
        got_h = gu.to_host(got, dtype)
        gu.check_rows(got_h, x, N, N, dtype, "no-alloc %dx%d" % (M, N))
        assert np.array_equal(got_h, gu.to_host(ref, dtype)), "output differs from softmax_rows_split"
