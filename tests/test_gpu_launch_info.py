"""softmax_rows_last_launch: the registers, local (spill) bytes and launch
shape of the last kernel the calling thread launched, as the bench records
them. The launch shape must match the plan that ran."""
import pytest

import memory_bound_row_rows_gb300 as sr
import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _run(name, rows, plan=sr.SR_PLAN_AUTO):
    w = synth.WORKLOADS[name].with_rows(rows)
    xd = gu.to_device(w.generate(), w.dtype)
    y = torch.empty((w.M, w.ld_out), dtype=xd.dtype, device="cuda")
    sr.softmax_rows_ex(xd, y, w.M, w.N, w.ld_in, w.ld_out, w.dtype, plan)
    torch.cuda.synchronize()
    return sr.softmax_rows_last_launch()


def test_row_plan_launch_record():
    info = _run("f32_4096x4096", 40)
    assert info["registers"] > 0 and info["local_bytes"] >= 0
    assert info["grid"] == 40 and info["cluster"] == 1
    assert info["block"] in (64, 128, 256, 512)
    assert "block" in info["name"]


def test_wide_plan_launch_record():
    info = _run("bf16_1024x131072", 3)
    assert info["cluster"] >= 2 and info["grid"] == 3 * info["cluster"]
    assert "wide_rows_kernel" in info["name"] or "wide_staged_kernel" in info["name"]
    assert 0 < info["registers"] <= 255


def test_warp_plan_launch_record():
    info = _run("bf16_16384x1000_ld1024", 64)
    assert "warp" in info["name"] and info["cluster"] == 1


def test_split_records_its_kernel():
    w = synth.WIDE_FEW["f16_4x32769"]
    xd = gu.to_device(w.generate(), w.dtype)
    y = torch.empty((w.M, w.ld_out), dtype=xd.dtype, device="cuda")
    need = sr.softmax_rows_split_workspace_bytes(xd, y, w.M, w.N, w.ld_in, w.ld_out, w.dtype)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    sr.softmax_rows_split(xd, y, w.M, w.N, w.ld_in, w.ld_out, w.dtype, ws, need)
    torch.cuda.synchronize()
    info = sr.softmax_rows_last_launch()
    sh = sr.softmax_rows_split_shape(xd, y, w.M, w.N, w.ld_in, w.ld_out, w.dtype)
    assert "split_grid_kernel" in info["name"] and info["grid"] == sh["lanes"] * sh["parts"]
