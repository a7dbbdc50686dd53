"""softmax_rows_split (few, wide rows; statistics through a workspace) against the oracle."""
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
# plus single huge rows and padded pitches.
SHAPES = [(4, 32769, 32769), (64, 131072, 131072), (128, 32769, 32776), (1, 1 << 20, 1 << 20),
          (3, 1000, 1000), (37, 12345, 12350), (2, 524288 + 8, 524288 + 8)]


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
