"""rmsnorm_residual_rows against the oracle.

The gate is derived from the arithmetic. h = dtype(x + r) is computed the
same way on both sides (an FP32 add rounded once to the dtype equals one
rounding of the exact sum for these formats), so h agrees exactly. The kernels
sum h^2 in FP32 in a tree of depth well under 128 (relative error below
2^-17), then divide, take an IEEE square root and reciprocal, and multiply
twice: the FP32 result is within 2^-16 of the exact value, relatively, before
the one rounding to the dtype. Elementwise:
    |gpu - oracle| <= 2^-16 * |oracle| + ulp_dtype(oracle).
"""
import numpy as np
import pytest

import memory_bound_row_rows_gb300 as sr
import oracle
import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

PLANS = [sr.SR_PLAN_AUTO, sr.SR_PLAN_ROW, sr.SR_PLAN_CLUSTER, sr.SR_PLAN_ONLINE]
MANT = {synth.F32: 23, synth.BF16: 7, synth.F16: 10}
MIN_EXP = {synth.F32: -126, synth.BF16: -126, synth.F16: -14}


def ulp(r, dtype):
    a = np.abs(r)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.exp2(np.maximum(e, MIN_EXP[dtype]) - MANT[dtype])


def rms_gate(gpu, ref, dtype, label):
    with np.errstate(invalid="ignore"):
        err = np.abs(gpu - ref)
        tol = 2.0 ** -16 * np.abs(ref) + ulp(ref, dtype)
    bad = (np.isnan(ref) != np.isnan(gpu)) | (np.isinf(ref) & ~(gpu == ref)) | \
          (np.isfinite(ref) & ~(err <= tol))
    assert not bad.any(), "%s: %d of %d outside the gate; worst err %.3g" % (
        label, int(bad.sum()), bad.size, float(np.nanmax(np.where(bad, err, 0))))


def run_case(x, r, w, M, N, ld_x, ld_r, ld_y, eps, dtype, plan, label):
    xd, rd, wd = gu.to_device(x, dtype), gu.to_device(r, dtype), gu.to_device(w, dtype)
    y = torch.full((max(M, 1), ld_y), float("nan"), dtype=gu.torch_dtype(dtype), device="cuda")
    st = sr.load().rmsnorm_residual_rows_ex(xd.data_ptr(), rd.data_ptr(), wd.data_ptr(),
                                            y.data_ptr(), M, N, ld_x, ld_r, ld_y, eps, dtype, plan,
                                            torch.cuda.current_stream().cuda_stream)
    if st == sr.SR_EPLAN:
        assert plan in (sr.SR_PLAN_ROW, sr.SR_PLAN_CLUSTER), label
        return False
    assert st == sr.SR_OK, "%s: status %d" % (label, st)
    torch.cuda.synchronize()
    out = gu.to_host(y, dtype)
    ref = oracle.load().rmsnorm_residual(x.reshape(-1), r.reshape(-1), w, M, N, ld_x, ld_r, N,
                                         float(np.float32(eps)), dtype)
    dec = lambda a: synth.storage_to_float64(np.ascontiguousarray(a[:, :N]), dtype)
    rms_gate(dec(out), dec(ref), dtype, label)
    if ld_y > N:
        pad = synth.storage_to_float64(np.ascontiguousarray(out[:, N:]), dtype)
        assert np.isnan(pad).all(), "%s: pad columns written" % label
    return True


@pytest.mark.parametrize("plan", PLANS, ids=lambda p: sr.PLAN_NAMES[p])
@pytest.mark.parametrize("name", sorted(synth.RMSNORM))
def test_shapes(name, plan):
    w = synth.RMSNORM[name]
    M = min(w.M, 600)
    run_case(w.x_rows(0, M), w.residual_rows(0, M), w.weight(), M, w.N, w.ld, w.ld, w.N, w.eps,
             w.dtype, plan, "%s/%s" % (name, sr.PLAN_NAMES[plan]))


@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16, synth.F16],
                         ids=lambda d: synth.DTYPE_NAMES[d])
@pytest.mark.parametrize("N", [1, 5, 8, 33, 256, 1000, 2056, 4097, 8200, 16392, 40000])
def test_widths_pitches_eps(dtype, N):
    M = 37
    for (ld_x, ld_r, ld_y), eps in (((N, N, N), 1e-6), ((N + 8, N + 16, N + 24), 0.0),
                                    ((N + 1, N, N + 3), 0.5)):
        # Spread magnitudes so that x + r rounds often.
        x = synth.generate(M, N, ld_x, dtype, seed=90 + N, p1=4.0)
        r = synth.generate(M, N, ld_r, dtype, seed=91 + N, p1=0.01)
        w = synth.generate(1, N, N, dtype, seed=92 + N, dist=synth.DIST_UNIFORM, p0=-1.0,
                           p1=2.0).reshape(-1)
        for plan in PLANS:
            run_case(x, r, w, M, N, ld_x, ld_r, ld_y, eps, dtype, plan,
                     "N=%d ld=%s eps=%g/%s" % (N, (ld_x, ld_r, ld_y), eps, sr.PLAN_NAMES[plan]))


def test_special_rows():
    dtype, M, N = synth.BF16, 5, 3000
    x = synth.generate(M, N, dtype=dtype, seed=95)
    r = synth.generate(M, N, dtype=dtype, seed=96)
    w = synth.generate(1, N, dtype=dtype, seed=97, dist=synth.DIST_UNIFORM, p0=0.5,
                       p1=1.5).reshape(-1)
    x[0, :] = 0
    r[0, :] = 0          # zero row: 0 with eps > 0
    x[1, 7] = 0x7FC0     # NaN in x: the whole row is NaN
    r[2, 11] = 0x7F80    # +inf in the residual: RMS infinite, finite entries 0, that one NaN
    x[3, :] = 0x3F80     # constant row of one (plus a residual) at large scale
    r[3, :] = 0x4700     # 32768
    for plan in PLANS:
        run_case(x, r, w, M, N, N, N, N, 1e-5, dtype, plan, "special/%s" % sr.PLAN_NAMES[plan])


def test_many_rows_and_tails():
    for M in (1, 3, 4, 5, 151, 153, 4099):
        for N, dtype in ((64, synth.F16), (96, synth.F32), (1024, synth.BF16)):
            x = synth.generate(M, N, dtype=dtype, seed=M)
            r = synth.generate(M, N, dtype=dtype, seed=M + 7)
            w = synth.generate(1, N, dtype=dtype, seed=M + 9, dist=synth.DIST_UNIFORM, p0=0.5,
                               p1=1.5).reshape(-1)
            for plan in PLANS:
                run_case(x, r, w, M, N, N, N, N, 1e-6, dtype, plan, "M=%d N=%d" % (M, N))


def test_torch_wrapper_against_torch_composition():
    """The wrapper against PyTorch's own FP32 composition (a second, independent
    reference): h = (x + r) rounded to fp16, y = h * rsqrt(mean(h^2) + eps) * w."""
    g = torch.Generator("cuda").manual_seed(5)
    x = torch.randn(256, 3072, device="cuda", generator=g).half()
    r = torch.randn(256, 3072, device="cuda", generator=g).half()
    w = (torch.rand(3072, device="cuda", generator=g) + 0.5).half()
    y = sr.rmsnorm_residual(x, r, w, eps=1e-6)
    h = (x.float() + r.float()).half().float()
    ref = (h * torch.rsqrt(h.pow(2).mean(dim=1, keepdim=True) + 1e-6)) * w.float()
    assert bool(((y.float() - ref).abs() <= 2.0 ** -10 * ref.abs() + 2.0 ** -14).all())


def test_empty_and_rejected():
    L = sr.load()
    s = torch.cuda.current_stream().cuda_stream
    a = torch.zeros(16, 16, device="cuda")
    b = torch.zeros(16, 16, device="cuda")
    w = torch.ones(16, device="cuda")
    assert L.rmsnorm_residual_rows(0, 0, 0, 0, 0, 16, 16, 16, 16, 1e-6, 0, s) == sr.SR_OK
    assert L.rmsnorm_residual_rows(a.data_ptr(), b.data_ptr(), w.data_ptr(), a.data_ptr(), 16, 16,
                                   16, 16, 16, 1e-6, 0, s) == sr.SR_EINVAL


@pytest.mark.parametrize("name", ["f16_16384x4096", "bf16_16384x4096", "f16_64x131072"])
def test_full_size_sampled_rows(name):
    w = synth.RMSNORM[name]
    x, r, wt = w.x_rows(0, w.M), w.residual_rows(0, w.M), w.weight()
    xd, rd, wd = gu.to_device(x, w.dtype), gu.to_device(r, w.dtype), gu.to_device(wt, w.dtype)
    y = torch.empty((w.M, w.N), dtype=gu.torch_dtype(w.dtype), device="cuda")
    assert sr.load().rmsnorm_residual_rows(xd.data_ptr(), rd.data_ptr(), wd.data_ptr(),
                                           y.data_ptr(), w.M, w.N, w.ld, w.ld, w.N, w.eps,
                                           w.dtype, torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    rows = sorted(set(np.random.default_rng(9).integers(0, w.M, size=48).tolist()) | {0, w.M - 1})
    out = gu.to_host(y[rows], w.dtype)
    ref = oracle.load().rmsnorm_residual(x[rows].reshape(-1), r[rows].reshape(-1), wt, len(rows),
                                         w.N, w.ld, w.ld, w.N, float(np.float32(w.eps)), w.dtype)
    dec = lambda a: synth.storage_to_float64(np.ascontiguousarray(a[:, :w.N]), w.dtype)
    rms_gate(dec(out), dec(ref), w.dtype, name)


@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16, synth.F16],
                         ids=lambda d: synth.DTYPE_NAMES[d])
@pytest.mark.parametrize("M", [9, 80])
def test_streamed_cluster_rows(dtype, M):
    """Aligned rows too wide for a cluster's registers: the streamed CLUSTER
    kernel reads x, the residual and the weights again in its second pass."""
    N = 131080
    x = synth.generate(M, N, N, dtype, seed=100 + M, p1=4.0)
    r = synth.generate(M, N, N, dtype, seed=101 + M, p1=0.01)
    w = synth.generate(1, N, N, dtype, seed=102 + M, dist=synth.DIST_UNIFORM, p0=-1.0,
                       p1=2.0).reshape(-1)
    for plan in (sr.SR_PLAN_AUTO, sr.SR_PLAN_CLUSTER):
        assert run_case(x, r, w, M, N, N, N, N, 1e-6, dtype, plan,
                        "streamed M=%d/%s" % (M, sr.PLAN_NAMES[plan]))
