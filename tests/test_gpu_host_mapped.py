"""softmax_rows_host_mapped: the kernel reads and writes mapped page-locked host memory."""
import numpy as np
import pytest

import memory_bound_row_rows_gb300 as sr
import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.mark.parametrize("name,rows", [("f32_4096x4096", 64), ("bf16_16384x1000_ld1024", 300),
                                       ("bf16_1024x131072", 6), ("f16_causal_524288x2048", 300),
                                       ("f32_1024x256", 1024),
                                       # 8 MiB and more: these run on the WIDE plan
                                       ("f32_4096x4096", 1024), ("bf16_16384x1000_ld1024", 8192),
                                       ("f16_causal_524288x2048", 4096)])
def test_mapped_matches_oracle(name, rows):
    w = synth.WORKLOADS[name].with_rows(rows)
    x = w.generate()
    tdt = gu.torch_dtype(w.dtype)
    xt = torch.from_numpy(x)
    if w.dtype != synth.F32:
        xt = xt.view(torch.int16).view(tdt)
    x_pin = xt.pin_memory()
    y_pin = torch.full((w.M, w.ld_out), float("nan"), dtype=tdt).pin_memory()
    sr.softmax_rows_host_mapped(x_pin, y_pin, w.M, w.N, w.ld_in, w.ld_out, w.dtype)
    torch.cuda.synchronize()
    y = y_pin.numpy() if w.dtype == synth.F32 else y_pin.view(torch.int16).numpy().view(np.uint16)
    gu.check_rows(y, x, w.N, w.ld_in, w.dtype, "%s mapped" % name)
    assert sr.softmax_rows_last_device_error() == sr.SR_OK


def test_unmapped_host_memory_is_refused():
    x = np.zeros((4, 256), dtype=np.float32)  # ordinary pageable memory
    y = np.full((4, 256), np.nan, dtype=np.float32)
    st = sr.load().softmax_rows_host_mapped(x.ctypes.data, y.ctypes.data, 4, 256, 256, 256, 0,
                                            torch.cuda.current_stream().cuda_stream)
    assert st == sr.SR_EINVAL
    assert np.isnan(y).all()
    # A device pointer is not host memory either.
    d = torch.zeros(4, 256, device="cuda")
    st = sr.load().softmax_rows_host_mapped(d.data_ptr(), y.ctypes.data, 4, 256, 256, 256, 0,
                                            torch.cuda.current_stream().cuda_stream)
    assert st == sr.SR_EINVAL
