"""softmax_rows_split (wide rows across any number of blocks of one cooperative
grid; statistics through a workspace) against the oracle."""
import math

import numpy as np
import pytest

import memory_bound_row_rows_gb300 as sr
import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def run_split(x, M, N, ld_in, ld_out, dtype, ws_extra=0):
    xd = gu.to_device(x, dtype)
    y = torch.full((M, ld_out), float("nan"), dtype=gu.torch_dtype(dtype), device="cuda")
    need = sr.softmax_rows_split_workspace_bytes(xd, y, M, N, ld_in, ld_out, dtype)
    assert need > 0
    ws = torch.full((need + ws_extra,), 0xFF, dtype=torch.uint8, device="cuda")  # garbage
    sr.softmax_rows_split(xd, y, M, N, ld_in, ld_out, dtype, ws, need + ws_extra)
    torch.cuda.synchronize()
    return gu.to_host(y, dtype)


# The few-row, wide shapes of "Measured optimization case studies" (Wide rows),
# plus single huge rows and padded pitches; and rows wide enough that a group
# of blocks takes several rows in turn, so that the four-step ring of pairs and
# counters wraps: 1 MiB rows of bf16 / f16 (about 21 groups, 7 steps), 4 MiB
# f32 rows at a padded pitch (5 groups, 5 steps) and 16 MiB f32 rows (one
# group of every block, 9 steps).
SHAPES = [(4, 32769, 32769), (64, 131072, 131072), (128, 32769, 32776), (1, 1 << 20, 1 << 20),
          (3, 1000, 1000), (37, 12345, 12350), (2, 524288 + 8, 524288 + 8),
          (130, 1 << 19, 1 << 19), (23, 1 << 20, (1 << 20) + 8), (9, 1 << 22, 1 << 22)]


@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16, synth.F16], ids=["f32", "bf16", "f16"])
@pytest.mark.parametrize("M,N,ld", SHAPES, ids=lambda v: str(v))
def test_split_matches_oracle(dtype, M, N, ld):
    x = synth.generate(M, N, ld=ld, dtype=dtype, seed=M * 31 + N, p1=2.0)
    out = run_split(x, M, N, ld, N, dtype)
    gu.check_rows(out, x, N, ld, dtype, "split %dx%d ld %d" % (M, N, ld))


def test_split_special_rows_and_causal():
    from tests import pins
    N = 40000
    rows = [np.full(N, -math.inf), np.linspace(-3, 3, N), np.zeros(N)]
    r = np.full(N, -math.inf); r[:7] = 1.0; rows.append(r)           # masked prefix-heavy row
    r = np.linspace(-2, 2, N); r[N - 1] = math.nan; rows.append(r)   # NaN in the last chunk
    r = np.full(N, -math.inf); r[-1] = 0.5; rows.append(r)           # one finite entry at the end
    for dtype in (synth.F32, synth.BF16, synth.F16):
        vals = pins.to_grid(np.array(rows), dtype)
        x = pins.encode_exact(vals, dtype)
        out = run_split(x, len(rows), N, N, N, dtype, ws_extra=64)
        gu.check_rows(out, x, N, N, dtype, "split special")
        g = synth.storage_to_float64(out, dtype)
        assert np.isnan(g[0]).all() and np.isnan(g[4]).all()
        assert np.all(g[3][7:] == 0.0) and g[5][-1] == 1.0


def test_split_rejects_bad_workspace_and_in_place():
    M, N = 4, 4096
    x = torch.randn(M, N, device="cuda")
    y = torch.empty_like(x)
    need = sr.softmax_rows_split_workspace_bytes(x, y, M, N, N, N, synth.F32)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    L = sr.load()
    st = torch.cuda.current_stream().cuda_stream
    assert L.softmax_rows_split(x.data_ptr(), y.data_ptr(), M, N, N, N, 0, ws.data_ptr(),
                                need - 8, st) == sr.SR_EINVAL
    assert L.softmax_rows_split(x.data_ptr(), y.data_ptr(), M, N, N, N, 0, None, need,
                                st) == sr.SR_EINVAL
    assert L.softmax_rows_split(x.data_ptr(), y.data_ptr(), M, N, N, N, 0, ws.data_ptr() + 4,
                                need, st) == sr.SR_EINVAL
    assert L.softmax_rows_split(x.data_ptr(), x.data_ptr(), M, N, N, N, 0, ws.data_ptr(),
                                need, st) == sr.SR_EINVAL
    assert L.softmax_rows_split(x.data_ptr(), y.data_ptr(), M, N, N, N, 0, ws.data_ptr(),
                                need, st) == sr.SR_OK
    torch.cuda.synchronize()
    assert torch.allclose(y, torch.softmax(x, dim=1), atol=1e-6, rtol=1e-5)


def test_split_launch_shape_matches_host_query():
    M, N, dtype = 130, 1 << 19, synth.BF16
    x = torch.zeros(M, N, dtype=torch.bfloat16, device="cuda")
    y = torch.empty_like(x)
    sh = sr.softmax_rows_split_shape(x, y, M, N, N, N, dtype)
    assert sh["lanes"] > 1 and -(-M // sh["lanes"]) > 4, sh  # the ring wraps
    ws = torch.empty(sr.softmax_rows_split_workspace_bytes(x, y, M, N, N, N, dtype),
                     dtype=torch.uint8, device="cuda")
    sr.softmax_rows_split(x, y, M, N, N, N, dtype, ws, ws.numel())
    torch.cuda.synchronize()
    info = sr.softmax_rows_last_launch()
    assert "split_bulk_kernel" in info["name"]  # aligned rows: the bulk-copy kernel
    assert info["grid"] == sh["lanes"] * sh["parts"] and info["block"] == 288
    if sr.load().softmax_rows_build_flags() == 0:  # the product build spills nothing
        assert info["local_bytes"] == 0
    assert torch.allclose(y.float(), torch.full_like(y.float(), 1.0 / N))


def test_split_wait_expiry():
    M, N, dtype = 6, 1 << 20, synth.F16
    x = synth.generate(M, N, dtype=dtype, seed=91, p1=2.0)
    xd = gu.to_device(x, dtype)
    y = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    need = sr.softmax_rows_split_workspace_bytes(xd, y, M, N, N, N, dtype)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    assert sr.softmax_rows_last_device_error() == sr.SR_OK
    st = sr.softmax_rows_split_test_expiry(xd, y, M, N, N, N, dtype, ws, need, 2_000_000)
    assert st == sr.SR_OK
    assert sr.softmax_rows_last_device_error() == sr.SR_EDEVICE_TIMEOUT
    assert torch.isnan(y).all(), "an expired kernel wrote output"
    sr.softmax_rows_split(xd, y, M, N, N, N, dtype, ws, need)
    torch.cuda.synchronize()
    gu.check_rows(gu.to_host(y, dtype), x, N, N, dtype, "split after expiry")
    assert sr.softmax_rows_last_device_error() == sr.SR_OK
