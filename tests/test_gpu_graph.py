"""The entry points under CUDA graph capture: a few calls captured into one graph and
replayed give the same results as direct calls (checked against the oracle). The calls
allocate nothing and their per-device set-up (attributes, occupancy) is done by the
first, uncaptured call."""
import numpy as np
import pytest

import memory_bound_row_rows_gb300 as sr
import oracle
import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def device_rows(w, rows):
    x = w.generate() if rows is None else w.rows(0, rows)
    return x, gu.to_device(x, w.dtype)


@pytest.mark.parametrize("name,rows,plan", [
    ("f32_4096x4096", 40, sr.SR_PLAN_ROW),
    ("bf16_16384x1000_ld1024", 300, sr.SR_PLAN_WARP),
    ("bf16_1024x131072", 6, sr.SR_PLAN_WIDE),
    ("f16_causal_524288x2048", 300, sr.SR_PLAN_ONLINE),
    ("bf16_1024x131072", 6, sr.SR_PLAN_CLUSTER),
])
def test_softmax_in_a_graph(name, rows, plan):
    w = synth.WORKLOADS[name].with_rows(rows)
    x, xd = device_rows(w, None)
    ys = [torch.full((w.M, w.ld_out), float("nan"), dtype=gu.torch_dtype(w.dtype), device="cuda")
          for _ in range(3)]
    sr.softmax_rows_ex(xd, ys[0], w.M, w.N, w.ld_in, w.ld_out, w.dtype, plan)  # set-up, uncaptured
    torch.cuda.synchronize()
    for y in ys:
        y.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for y in ys:
            sr.softmax_rows_ex(xd, y, w.M, w.N, w.ld_in, w.ld_out, w.dtype, plan)
    torch.cuda.synchronize()
    assert all(torch.isnan(y).all() for y in ys), "capture executed the kernels"
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    for y in ys:
        gu.check_rows(gu.to_host(y, w.dtype), x, w.N, w.ld_in, w.dtype,
                      "%s plan %s in a graph" % (name, sr.PLAN_NAMES[plan]))
    assert sr.softmax_rows_last_device_error() == sr.SR_OK


@pytest.mark.parametrize("name,plan", [("f16_16384x4096", sr.SR_PLAN_ROW),
                                       ("f16_64x131072", sr.SR_PLAN_CLUSTER)])
def test_backward_and_rmsnorm_in_a_graph(name, plan):
    bw = synth.BACKWARD[name].with_rows(min(64, synth.BACKWARD[name].M))
    y, dy = bw.y_rows(0, bw.M), bw.dy_rows(0, bw.M)
    yd, gd = gu.to_device(y, bw.dtype), gu.to_device(dy, bw.dtype)
    dx = torch.empty((bw.M, bw.N), dtype=gu.torch_dtype(bw.dtype), device="cuda")
    rn = synth.RMSNORM[name].with_rows(min(64, synth.RMSNORM[name].M))
    x, r, wt = rn.x_rows(0, rn.M), rn.residual_rows(0, rn.M), rn.weight()
    xd, rd, wd = gu.to_device(x, rn.dtype), gu.to_device(r, rn.dtype), gu.to_device(wt, rn.dtype)
    yr = torch.empty((rn.M, rn.N), dtype=gu.torch_dtype(rn.dtype), device="cuda")

    def calls():
        sr.softmax_rows_backward_ex(yd, gd, dx, bw.M, bw.N, bw.ld, bw.ld, bw.N, bw.dtype, plan)
        sr.rmsnorm_residual_rows_ex(xd, rd, wd, yr, rn.M, rn.N, rn.ld, rn.ld, rn.N, rn.eps,
                                    rn.dtype, plan)

    calls()
    torch.cuda.synchronize()
    dx.fill_(float("nan"))
    yr.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        calls()
    g.replay()
    torch.cuda.synchronize()
    dec = lambda a, d, n: synth.storage_to_float64(np.ascontiguousarray(a[:, :n]), d)
    ref = oracle.load().softmax_backward(y.reshape(-1), dy.reshape(-1), bw.M, bw.N, bw.ld, bw.ld,
                                         bw.N, bw.dtype)
    got = dec(gu.to_host(dx, bw.dtype), bw.dtype, bw.N)
    want = dec(ref, bw.dtype, bw.N)
    assert np.allclose(got, want, rtol=2 ** -9, atol=1e-6)
    ref = oracle.load().rmsnorm_residual(x.reshape(-1), r.reshape(-1), wt, rn.M, rn.N, rn.ld, rn.ld,
                                         rn.N, float(np.float32(rn.eps)), rn.dtype)
    got = dec(gu.to_host(yr, rn.dtype), rn.dtype, rn.N)
    want = dec(ref, rn.dtype, rn.N)
    assert np.allclose(got, want, rtol=2 ** -9, atol=1e-6)
    assert sr.softmax_rows_last_device_error() == sr.SR_OK


def test_streamed_rows_in_a_graph():
    """The streamed WIDE kernel and the streamed row-pair CLUSTER kernel, captured."""
    M, N, dtype = 3, 262152, synth.BF16
    x = synth.generate(M, N, dtype=dtype, seed=33, p1=2.0)
    xd = gu.to_device(x, dtype)
    y = torch.empty((M, N), dtype=gu.torch_dtype(dtype), device="cuda")
    Mb, Nb = 4, 131080
    yb = synth.generate(Mb, Nb, dtype=synth.F16, seed=34, dist=synth.DIST_UNIFORM, p0=0.0,
                        p1=2.0 / Nb)
    gb = synth.generate(Mb, Nb, dtype=synth.F16, seed=35)
    ybd, gbd = gu.to_device(yb, synth.F16), gu.to_device(gb, synth.F16)
    dx = torch.empty((Mb, Nb), dtype=torch.float16, device="cuda")

    def calls():
        sr.softmax_rows(xd, y, M, N, N, N, dtype)
        sr.softmax_rows_backward(ybd, gbd, dx, Mb, Nb, Nb, Nb, Nb, synth.F16)

    calls()
    torch.cuda.synchronize()
    y.fill_(float("nan"))
    dx.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        calls()
    g.replay()
    torch.cuda.synchronize()
    gu.check_rows(gu.to_host(y, dtype), x, N, N, dtype, "streamed WIDE in a graph")
    ref = oracle.load().softmax_backward(yb.reshape(-1), gb.reshape(-1), Mb, Nb, Nb, Nb, Nb,
                                         synth.F16)
    dec = lambda a: synth.storage_to_float64(np.ascontiguousarray(a), synth.F16)
    assert np.allclose(dec(gu.to_host(dx, synth.F16)), dec(ref), rtol=2 ** -9, atol=1e-6)
    assert sr.softmax_rows_last_device_error() == sr.SR_OK


def test_host_pipeline_in_a_graph():
    """softmax_rows_host forks onto its own streams and joins back: capturable too."""
    w = synth.WORKLOADS["f32_4096x4096"].with_rows(64)
    x = w.generate()
    x_pin = torch.from_numpy(x).pin_memory()
    y_pin = torch.full((w.M, w.ld_out), float("nan")).pin_memory()
    need = sr.softmax_rows_host_workspace_bytes(w.M, w.N, w.dtype)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    sr.softmax_rows_host(x_pin, y_pin, w.M, w.N, w.ld_in, w.ld_out, w.dtype, ws, need)
    torch.cuda.synchronize()
    y_pin.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        sr.softmax_rows_host(x_pin, y_pin, w.M, w.N, w.ld_in, w.ld_out, w.dtype, ws, need)
    g.replay()
    torch.cuda.synchronize()
    gu.check_rows(y_pin.numpy(), x, w.N, w.ld_in, w.dtype, "host pipeline in a graph")


def test_staged_rows_in_a_graph():
    """The staged WIDE kernel (1 MiB rows, half of each slice in shared memory), captured."""
    M, N, dtype = 4, 524288, synth.BF16
    x = synth.generate(M, N, dtype=dtype, seed=36, p1=2.0)
    xd = gu.to_device(x, dtype)
    y = torch.empty((M, N), dtype=gu.torch_dtype(dtype), device="cuda")
    sr.softmax_rows(xd, y, M, N, N, N, dtype)
    torch.cuda.synchronize()
    assert "wide_staged_kernel" in sr.softmax_rows_last_launch()["name"]
    y.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        sr.softmax_rows(xd, y, M, N, N, N, dtype)
    g.replay()
    torch.cuda.synchronize()
    gu.check_rows(gu.to_host(y, dtype), x, N, N, dtype, "staged WIDE in a graph")
    assert sr.softmax_rows_last_device_error() == sr.SR_OK
