"""softmax_rows_host: host buffers streamed through a device workspace (GPU required)."""
import numpy as np
import pytest

import memory_bound_row_rows_gb300 as sr
import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def pinned_copy(a: np.ndarray, dtype: int):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype != synth.F32:
        t = t.view(torch.int16).view(gu.torch_dtype(dtype))
    return t.pin_memory()


@pytest.mark.parametrize("name,rows", [("f32_4096x4096", 300), ("bf16_16384x1000_ld1024", 2000),
                                       ("bf16_1024x131072", 40), ("f16_causal_524288x2048", 5000)])
@pytest.mark.parametrize("workspace", ["full", "two_rows", "odd"])
def test_host_pipeline_matches_oracle(name, rows, workspace):
    w = synth.WORKLOADS[name].with_rows(rows)
    x = w.generate()
    h_in = pinned_copy(x, w.dtype)
    h_out = torch.full((w.M, w.ld_out), float("nan"), dtype=h_in.dtype).pin_memory()
    es = w.elem_bytes
    pitch = -(-w.N * es // 16) * 16
    need = {"full": sr.softmax_rows_host_workspace_bytes(w.M, w.N, w.dtype),
            "two_rows": 2 * 2 * pitch, "odd": 7 * 2 * pitch + 48}[workspace]
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    sr.softmax_rows_host(h_in, h_out, w.M, w.N, w.ld_in, w.ld_out, w.dtype, ws, need)
    torch.cuda.current_stream().synchronize()
    out = gu.to_host(h_out, w.dtype)
    gu.check_rows(out, x, w.N, w.ld_in, w.dtype, "host %s ws=%s" % (name, workspace))


def test_host_pipeline_pageable_in_place_and_errors():
    w = synth.WORKLOADS["f32_4096x4096"].with_rows(33)
    x = w.generate()
    buf = torch.from_numpy(x.copy())  # pageable, used in place
    need = sr.softmax_rows_host_workspace_bytes(w.M, w.N, w.dtype)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    sr.softmax_rows_host(buf, buf, w.M, w.N, w.N, w.N, w.dtype, ws, need)
    torch.cuda.current_stream().synchronize()
    gu.check_rows(buf.numpy(), x, w.N, w.N, w.dtype, "host in place")
    L = sr.load()
    st = torch.cuda.current_stream().cuda_stream
    assert L.softmax_rows_host(buf.data_ptr(), buf.data_ptr(), w.M, w.N, w.N, w.N, w.dtype,
                               ws.data_ptr(), 16, st) == sr.SR_EINVAL  # workspace too small
    assert L.softmax_rows_host(buf.data_ptr(), buf.data_ptr(), w.M, w.N, w.N, w.N, w.dtype,
                               None, need, st) == sr.SR_EINVAL
    assert L.softmax_rows_host(buf.data_ptr(), buf.data_ptr(), 0, w.N, w.N, w.N, w.dtype,
                               None, 0, st) == sr.SR_OK
