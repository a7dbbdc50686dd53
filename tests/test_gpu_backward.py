"""softmax_rows_backward (dx = y * (dy - sum(y * dy))) against the oracle.

The gate is derived from the arithmetic. The kernels hold the dot product
d = sum_k y_k dy_k in FP32, summed in a tree of depth well under 128, so
|d_gpu - d| <= 2^-17 * S with S = sum_k |y_k dy_k|. Then
dx_j = y_j * (dy_j - d) in FP32 adds two roundings, and the cast to the
dtype one more. Elementwise:
    |gpu - oracle| <= |y_j| * (2^-17 * S + 2^-22 * |dy_j - d|)
                      + 2^-22 * |oracle| + 2 * ulp_dtype(oracle).
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
    e = np.maximum(e, MIN_EXP[dtype])
    return np.exp2(e - MANT[dtype])


def bwd_gate(gpu, ref, y, dy, dtype, label):
    """gpu, ref, y, dy: decoded float64 (M, N) arrays."""
    d = (y * dy).sum(axis=1, keepdims=True)
    S = np.abs(y * dy).sum(axis=1, keepdims=True)
    with np.errstate(invalid="ignore", over="ignore"):
        tol = (np.abs(y) * (2.0 ** -17 * S + 2.0 ** -22 * np.abs(dy - d))
               + 2.0 ** -22 * np.abs(ref) + 2 * ulp(ref, dtype))
        err = np.abs(gpu - ref)
    nan_r, nan_g = np.isnan(ref), np.isnan(gpu)
    inf_mismatch = np.isinf(ref) & ~(gpu == ref)
    bad = (nan_r != nan_g) | inf_mismatch | (np.isfinite(ref) & ~(err <= tol))
    assert not bad.any(), "%s: %d of %d outside the gate; worst err %.3g at tol %.3g" % (
        label, int(bad.sum()), bad.size, float(np.nanmax(np.where(bad, err, 0))),
        float(tol[bad].min()) if bad.any() else 0.0)


def run_bwd(yd, gd, M, N, ld_y, ld_dy, ld_dx, dtype, plan, fill=float("nan")):
    dx = torch.full((max(M, 1), ld_dx), fill, dtype=gu.torch_dtype(dtype), device="cuda")
    st = sr.load().softmax_rows_backward_ex(yd.data_ptr() if M else 0, gd.data_ptr() if M else 0,
                                           dx.data_ptr(), M, N, ld_y, ld_dy, ld_dx, dtype, plan,
                                           torch.cuda.current_stream().cuda_stream)
    return st, dx


def check_case(y, dy, M, N, ld_y, ld_dy, ld_dx, dtype, plan, label):
    """Run one plan on host inputs y (M x ld_y) and dy (M x ld_dy); gate it.
    Returns False when the plan cannot take the shape."""
    yd, gd = gu.to_device(y, dtype), gu.to_device(dy, dtype)
    st, dx = run_bwd(yd, gd, M, N, ld_y, ld_dy, ld_dx, dtype, plan)
    if st == sr.SR_EPLAN:
        assert plan != sr.SR_PLAN_AUTO and plan != sr.SR_PLAN_ONLINE, label
        return False
    assert st == sr.SR_OK, "%s: status %d" % (label, st)
    torch.cuda.synchronize()
    out = gu.to_host(dx, dtype)
    ref = oracle.load().softmax_backward(y.reshape(-1), dy.reshape(-1), M, N, ld_y, ld_dy, N,
                                         dtype)
    dec = lambda a, n=N: synth.storage_to_float64(np.ascontiguousarray(a[:, :n]), dtype)
    bwd_gate(dec(out), dec(ref), dec(y), dec(dy), dtype, label)
    # Pad columns keep their NaN fill: nothing is written past N.
    if ld_dx > N:
        pad = synth.storage_to_float64(np.ascontiguousarray(out[:, N:]), dtype)
        assert np.isnan(pad).all(), "%s: pad columns written" % label
    return True


@pytest.mark.parametrize("plan", PLANS, ids=lambda p: sr.PLAN_NAMES[p])
@pytest.mark.parametrize("name", sorted(synth.BACKWARD))
def test_training_shapes(name, plan):
    w = synth.BACKWARD[name]
    M = min(w.M, 600)  # a ragged subset of the taller shapes
    y, dy = w.y_rows(0, M), w.dy_rows(0, M)
    check_case(y, dy, M, w.N, w.ld, w.ld, w.N, w.dtype, plan, "%s/%s" % (name, sr.PLAN_NAMES[plan]))


@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16, synth.F16],
                         ids=lambda d: synth.DTYPE_NAMES[d])
def test_true_softmax_outputs(dtype):
    # y is the (oracle's) softmax of a logit row, dy a gradient: the intended use.
    M, N = 300, 3000
    x = synth.generate(M, N, dtype=dtype, seed=40, p1=2.0)
    y = oracle.softmax_rows(x.reshape(-1), M, N, N, N, dtype)
    dy = synth.generate(M, N, dtype=dtype, seed=41)
    for plan in PLANS:
        check_case(y, dy, M, N, N, N, N, dtype, plan, "softmax-y/%s" % sr.PLAN_NAMES[plan])


@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16, synth.F16],
                         ids=lambda d: synth.DTYPE_NAMES[d])
@pytest.mark.parametrize("N", [1, 7, 8, 31, 64, 129, 1000, 2047, 2056, 4104, 8200, 16392, 40000])
def test_widths_and_pitches(dtype, N):
    M = 37  # fewer rows than SMs, not a multiple of any rows-per-block
    for ld_y, ld_dy, ld_dx in ((N, N, N), (N + 8, N + 16, N + 24), (N + 1, N, N + 3)):
        y = synth.generate(M, N, ld_y, dtype, seed=50 + N, dist=synth.DIST_UNIFORM, p0=0.0,
                           p1=2.0 / N)
        dy = synth.generate(M, N, ld_dy, dtype, seed=60 + N)
        for plan in PLANS:
            check_case(y, dy, M, N, ld_y, ld_dy, ld_dx, dtype, plan,
                       "N=%d ld=%s/%s" % (N, (ld_y, ld_dy, ld_dx), sr.PLAN_NAMES[plan]))


def test_many_short_rows_and_tails():
    # Row counts around the rows-per-block of one-warp teams (4) and a
    # grid that walks several rows per block.
    for M in (1, 3, 4, 5, 151, 152, 153, 5001):
        for N, dtype in ((64, synth.F16), (100, synth.F32), (1024, synth.BF16)):
            y = synth.generate(M, N, dtype=dtype, seed=M, dist=synth.DIST_UNIFORM, p0=0.0, p1=0.02)
            dy = synth.generate(M, N, dtype=dtype, seed=M + 1)
            for plan in PLANS:
                check_case(y, dy, M, N, N, N, N, dtype, plan, "M=%d N=%d" % (M, N))


def test_special_values():
    dtype, M, N = synth.F32, 6, 2048
    y = synth.generate(M, N, dtype=dtype, seed=70, dist=synth.DIST_UNIFORM, p0=0.0, p1=0.001)
    dy = synth.generate(M, N, dtype=dtype, seed=71)
    y[0, :] = 0.0
    y[0, 17] = 1.0            # one-hot y: dx = 0 exactly
    dy[1, :] = 2.5            # constant dy with y summing to one: dx ~ 0
    y[1, :] = 1.0 / N
    dy[2, 5] = np.nan         # NaN in dy: the whole row is NaN
    y[3, 9] = np.inf          # inf in y: the dot product is infinite
    dy[4, :] = 0.0            # zero gradient: dx = 0
    y[5, :] = -y[5, :]        # negative y is taken as written
    for plan in PLANS:
        check_case(y, dy, M, N, N, N, N, dtype, plan, "special/%s" % sr.PLAN_NAMES[plan])


def test_empty_and_rejected():
    L = sr.load()
    s = torch.cuda.current_stream().cuda_stream
    a = torch.zeros(16, 16, device="cuda")
    b = torch.zeros(16, 16, device="cuda")
    assert L.softmax_rows_backward(0, 0, 0, 0, 16, 16, 16, 16, 0, s) == sr.SR_OK
    assert L.softmax_rows_backward(a.data_ptr(), b.data_ptr(), a.data_ptr(), 16, 16, 16, 16, 16,
                                   0, s) == sr.SR_EINVAL
    assert L.softmax_rows_backward(a.data_ptr(), b.data_ptr(), b.data_ptr(), 16, 16, 16, 16, 16,
                                   0, s) == sr.SR_EINVAL


def test_torch_wrapper_matches_autograd_shape():
    # The wrapper returns a fresh tensor with dx's shape; values gated above.
    x = torch.randn(64, 500, device="cuda", generator=torch.Generator("cuda").manual_seed(3))
    y = torch.softmax(x, dim=1)
    dy = torch.randn_like(y)
    dx = sr.softmax_backward(y, dy)
    assert dx.shape == y.shape and dx.dtype == y.dtype
    # Rows of a softmax backward sum to ~0 when y sums to one.
    assert float(dx.sum(dim=1).abs().max()) < 1e-5


@pytest.mark.parametrize("name", ["f16_16384x4096", "f32_4096x4096", "f16_64x131072"])
def test_full_size_sampled_rows(name):
    """The benchmark's launch on the whole matrix, checked on sampled rows."""
    w = synth.BACKWARD[name]
    y, dy = w.y_rows(0, w.M), w.dy_rows(0, w.M)
    yd, gd = gu.to_device(y, w.dtype), gu.to_device(dy, w.dtype)
    st, dx = run_bwd(yd, gd, w.M, w.N, w.ld, w.ld, w.N, w.dtype, sr.SR_PLAN_AUTO)
    assert st == sr.SR_OK
    torch.cuda.synchronize()
    rows = sorted(set(np.random.default_rng(7).integers(0, w.M, size=48).tolist()) | {0, w.M - 1})
    out = gu.to_host(dx[rows], w.dtype)
    ys, gs = y[rows], dy[rows]
    ref = oracle.load().softmax_backward(ys.reshape(-1), gs.reshape(-1), len(rows), w.N, w.ld,
                                         w.ld, w.N, w.dtype)
    dec = lambda a: synth.storage_to_float64(np.ascontiguousarray(a[:, :w.N]), w.dtype)
    bwd_gate(dec(out), dec(ref), dec(ys), dec(gs), w.dtype, name)


@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16, synth.F16],
                         ids=lambda d: synth.DTYPE_NAMES[d])
def test_offset_views(dtype):
    """Matrices that start k elements past a 16-byte boundary: with equal k
    for all three the rows are read as vectors after a short head; with
    different k element by element."""
    M, N = 40, 4096
    # One spare row, so that a view starting k elements in still holds M full rows.
    y = synth.generate(M + 1, N + 8, dtype=dtype, seed=80, dist=synth.DIST_UNIFORM, p0=0.0,
                       p1=2.0 / N)
    dy = synth.generate(M + 1, N + 8, dtype=dtype, seed=81)
    tdt = gu.torch_dtype(dtype)
    yd, gd = gu.to_device(y, dtype).reshape(-1), gu.to_device(dy, dtype).reshape(-1)
    for ky, kg, kx in ((1, 1, 1), (3, 3, 3), (1, 2, 3), (0, 5, 0)):
        if dtype == synth.F32 and max(ky, kg, kx) > 3:
            continue
        out = torch.full((M * (N + 8) + 8,), float("nan"), dtype=tdt, device="cuda")
        for plan in PLANS:
            st = sr.load().softmax_rows_backward_ex(
                yd[ky:].data_ptr(), gd[kg:].data_ptr(), out[kx:].data_ptr(), M, N, N + 8, N + 8,
                N + 8, dtype, plan, torch.cuda.current_stream().cuda_stream)
            if st == sr.SR_EPLAN:
                assert plan == sr.SR_PLAN_CLUSTER or plan == sr.SR_PLAN_ROW
                continue
            assert st == sr.SR_OK
            torch.cuda.synchronize()
            got = gu.to_host(out[kx:kx + M * (N + 8)].reshape(M, N + 8), dtype)
            ys = gu.to_host(yd[ky:ky + M * (N + 8)].reshape(M, N + 8), dtype)
            gs = gu.to_host(gd[kg:kg + M * (N + 8)].reshape(M, N + 8), dtype)
            ref = oracle.load().softmax_backward(ys.reshape(-1), gs.reshape(-1), M, N, N + 8,
                                                 N + 8, N, dtype)
            dec = lambda a: synth.storage_to_float64(np.ascontiguousarray(a[:, :N]), dtype)
            bwd_gate(dec(got), dec(ref), dec(ys), dec(gs), dtype,
                     "offsets %s/%s" % ((ky, kg, kx), sr.PLAN_NAMES[plan]))


@pytest.mark.parametrize("name", ["f16_64x131072", "f16_4x32769"])
def test_cluster_wait_expiry(name):
    """The CLUSTER plan's bounded waits: with the partials not sent every wait
    expires, the status is reported, nothing is written, and the context still
    runs a normal call afterwards."""
    w = synth.BACKWARD[name].with_rows(4)
    y, dy = w.y_rows(0, w.M), w.dy_rows(0, w.M)
    yd, gd = gu.to_device(y, w.dtype), gu.to_device(dy, w.dtype)
    dx = torch.full((w.M, w.N), float("nan"), dtype=gu.torch_dtype(w.dtype), device="cuda")
    assert sr.softmax_rows_last_device_error() == sr.SR_OK
    sr.softmax_rows_backward_test_expiry(yd, gd, dx, w.M, w.N, w.ld, w.ld, w.N, w.dtype,
                                         2_000_000)
    assert sr.softmax_rows_last_device_error() == sr.SR_EDEVICE_TIMEOUT
    assert torch.isnan(dx).all(), "an expired kernel wrote output"
    assert sr.softmax_rows_last_device_error() == sr.SR_OK
    check_case(y, dy, w.M, w.N, w.ld, w.ld, w.N, w.dtype, sr.SR_PLAN_CLUSTER, "after expiry")


@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16, synth.F16],
                         ids=lambda d: synth.DTYPE_NAMES[d])
@pytest.mark.parametrize("M", [9, 80])
def test_streamed_cluster_rows(dtype, M):
    """Aligned rows too wide for a cluster's registers: the streamed CLUSTER
    kernel (16-block clusters for 9 rows, 8-block clusters for 80)."""
    N = 131080
    for ld in (N, N + 8):
        y = synth.generate(M, N, ld, dtype, seed=M + ld, dist=synth.DIST_UNIFORM, p0=0.0,
                           p1=2.0 / N)
        dy = synth.generate(M, N, ld, dtype, seed=M + ld + 1)
        assert sr.softmax_rows_backward_plan(0x7F0000000000, 0x7F1000000000, 0x7F2000000000, M, N,
                                             ld, ld, ld, dtype, sr.SR_PLAN_AUTO,
                                             152) == sr.SR_PLAN_CLUSTER
        for plan in (sr.SR_PLAN_AUTO, sr.SR_PLAN_CLUSTER):
            assert check_case(y, dy, M, N, ld, ld, ld, dtype, plan,
                              "streamed M=%d ld=%d/%s" % (M, ld, sr.PLAN_NAMES[plan]))


def test_streamed_cluster_wait_expiry():
    M, N, dtype = 3, 131080, synth.BF16
    y = synth.generate(M, N, N, dtype, seed=5, dist=synth.DIST_UNIFORM, p0=0.0, p1=2.0 / N)
    dy = synth.generate(M, N, N, dtype, seed=6)
    yd, gd = gu.to_device(y, dtype), gu.to_device(dy, dtype)
    dx = torch.full((M, N), float("nan"), dtype=gu.torch_dtype(dtype), device="cuda")
    assert sr.softmax_rows_last_device_error() == sr.SR_OK
    sr.softmax_rows_backward_test_expiry(yd, gd, dx, M, N, N, N, N, dtype, 2_000_000)
    assert sr.softmax_rows_last_device_error() == sr.SR_EDEVICE_TIMEOUT
    assert torch.isnan(dx).all(), "an expired kernel wrote output"
    assert sr.softmax_rows_last_device_error() == sr.SR_OK
    check_case(y, dy, M, N, N, N, N, dtype, sr.SR_PLAN_CLUSTER, "streamed after expiry")
