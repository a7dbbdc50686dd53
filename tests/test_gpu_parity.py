"""CUDA path against the CPU oracle, element by element (GPU required).

Every call goes through the C ABI (the ctypes binding). Inputs come from the
seeded generator; outputs are pre-filled with NaN so a kernel that skips an
element cannot pass on stale values.
"""
import math

import numpy as np
import pytest

import memory_bound_row_rows_gb300 as sr
import oracle
import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

PLANS = [sr.SR_PLAN_AUTO, sr.SR_PLAN_WARP, sr.SR_PLAN_CTA, sr.SR_PLAN_CLUSTER, sr.SR_PLAN_ONLINE,
         sr.SR_PLAN_SMEM, sr.SR_PLAN_ROW, sr.SR_PLAN_WIDE]


def nan_filled(M, ld, dtype):
    return torch.full((M, ld), float("nan"), dtype=gu.torch_dtype(dtype), device="cuda")


def run_plan(x_dev, M, N, ld_in, ld_out, dtype, plan, out=None):
    y = nan_filled(M, ld_out, dtype) if out is None else out
    st = sr.load().softmax_rows_ex(x_dev.data_ptr(), y.data_ptr(), M, N, ld_in, ld_out, dtype,
                                   plan, torch.cuda.current_stream().cuda_stream)
    return st, y


def plan_applies(x_dev, y_dev, M, N, ld_in, ld_out, dtype, plan):
    return sr.softmax_rows_plan_check(x_dev, y_dev, M, N, ld_in, ld_out, dtype, plan) > 0


# ---- every workload's value law at oracle-friendly row counts, every plan ----

SMALL_CASES = [
    ("f32_1024x256", 0, 300),
    ("f32_4096x4096", 0, 70),
    ("bf16_16384x1000_ld1024", 0, 300),
    ("bf16_1024x131072", 0, 10),
    ("f16_causal_524288x2048", 0, 300),
    ("f16_causal_524288x2048", 1900, 300),  # crosses the causal period
]


@pytest.mark.parametrize("name,row0,rows", SMALL_CASES, ids=lambda v: str(v))
@pytest.mark.parametrize("plan", PLANS, ids=lambda p: sr.PLAN_NAMES[p])
def test_small_parity(name, row0, rows, plan):
    w = synth.WORKLOADS[name]
    x = w.rows(row0, rows)
    xd = gu.to_device(x, w.dtype)
    y = nan_filled(rows, w.ld_out, w.dtype)
    if not plan_applies(xd, y, rows, w.N, w.ld_in, w.ld_out, w.dtype, plan):
        st, _ = run_plan(xd, rows, w.N, w.ld_in, w.ld_out, w.dtype, plan, out=y)
        assert st == sr.SR_EPLAN
        assert torch.isnan(y).all(), "a rejected plan wrote to the output"
        return
    st, y = run_plan(xd, rows, w.N, w.ld_in, w.ld_out, w.dtype, plan, out=y)
    assert st == sr.SR_OK, sr.softmax_rows_strerror(st)
    torch.cuda.synchronize()
    gu.check_rows(gu.to_host(y, w.dtype), x, w.N, w.ld_in, w.dtype,
                  "%s[%d:+%d] plan %s" % (name, row0, rows, sr.PLAN_NAMES[plan]))
    assert sr.softmax_rows_last_device_error() == sr.SR_OK


# ---- full sizes, automatic plan (the benchmark's launch), sampled rows ----

FULL = ["f32_1024x256", "f32_4096x4096", "bf16_16384x1000_ld1024", "bf16_1024x131072",
        "f16_causal_524288x2048"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled(name):
    w = synth.WORKLOADS[name]
    x = w.generate()
    xd = gu.to_device(x, w.dtype)
    y = nan_filled(w.M, w.ld_out, w.dtype)
    st = sr.softmax_rows(xd, y, w.M, w.N, w.ld_in, w.ld_out, w.dtype)
    assert st == sr.SR_OK
    torch.cuda.synchronize()
    rng = np.random.default_rng(1234)
    sample = np.unique(np.concatenate([np.arange(min(64, w.M)), np.arange(max(0, w.M - 64), w.M),
                                       rng.integers(0, w.M, 128)]))
    ys = gu.to_host(y[torch.from_numpy(sample).to("cuda")], w.dtype)
    gu.check_rows(ys, x[sample], w.N, w.ld_in, w.dtype, "%s sampled" % name)
    # Properties of every row: finite, in [0, 1], sums to 1 within rounding,
    # exact zeros where the input is -inf.
    bound = {synth.F32: 2.0 ** -24, synth.BF16: 2.0 ** -9, synth.F16: 2.0 ** -11}[w.dtype]
    chunk = max(1, (1 << 26) // w.N)
    for r0 in range(0, w.M, chunk):
        yc = y[r0:r0 + chunk, :w.N].double()
        assert torch.isfinite(yc).all(), "%s: non-finite output near row %d" % (name, r0)
        assert (yc >= 0).all() and (yc <= 1).all()
        err = (yc.sum(dim=1) - 1).abs().max().item()
        assert err <= bound + 2.0 ** -20, "%s: row sum off by %g near row %d" % (name, err, r0)
        if w.causal_period:
            xc = xd[r0:r0 + chunk, :w.N]
            assert (y[r0:r0 + chunk, :w.N][torch.isneginf(xc)] == 0).all()
    assert sr.softmax_rows_last_device_error() == sr.SR_OK


@pytest.mark.parametrize("name,plan", [("bf16_1024x131072", sr.SR_PLAN_WIDE),
                                       ("bf16_1024x131072", sr.SR_PLAN_CLUSTER)])
def test_full_size_forced_wide_plans(name, plan):
    """Both wide-row plans on the whole wide workload, checked on sampled rows."""
    w = synth.WORKLOADS[name]
    x = w.generate()
    xd = gu.to_device(x, w.dtype)
    st, y = run_plan(xd, w.M, w.N, w.ld_in, w.ld_out, w.dtype, plan)
    assert st == sr.SR_OK
    torch.cuda.synchronize()
    sample = np.unique(np.concatenate([np.arange(8), np.arange(w.M - 8, w.M),
                                       np.random.default_rng(5).integers(0, w.M, 48)]))
    ys = gu.to_host(y[torch.from_numpy(sample).to("cuda")], w.dtype)
    gu.check_rows(ys, x[sample], w.N, w.ld_in, w.dtype, "%s plan %s" % (name, sr.PLAN_NAMES[plan]))
    assert sr.softmax_rows_last_device_error() == sr.SR_OK


@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16, synth.F16], ids=["f32", "bf16", "f16"])
@pytest.mark.parametrize("N,M", [(2049, 37), (4097, 64), (32769, 4), (40000, 3), (131071, 2)])
def test_wide_shifted_rows(dtype, N, M):
    """Odd widths with equal pitches, and views starting k elements past a
    16-byte boundary: the ROW and WIDE plans read them as shifted vectors."""
    vec = 4 if dtype == synth.F32 else 8
    x = synth.generate(M + 1, N, dtype=dtype, seed=N + M, p1=2.5)
    base = gu.to_device(x.reshape(-1), dtype)
    for k in (0, 1, vec - 1):
        xd = base[k:]
        yb = torch.full(((M + 1) * N,), float("nan"), dtype=gu.torch_dtype(dtype), device="cuda")
        yd = yb[k:]
        for plan in (sr.SR_PLAN_WIDE, sr.SR_PLAN_ROW, sr.SR_PLAN_AUTO):
            got = sr.softmax_rows_plan_check(xd, yd, M, N, N, N, dtype, plan)
            if plan == sr.SR_PLAN_ROW and got < 0:
                continue  # wider than one block
            assert got in (sr.SR_PLAN_WIDE, sr.SR_PLAN_ROW), (plan, got)
            yb.fill_(float("nan"))
            st = sr.load().softmax_rows_ex(xd.data_ptr(), yd.data_ptr(), M, N, N, N, dtype, plan,
                                           torch.cuda.current_stream().cuda_stream)
            assert st == sr.SR_OK
            torch.cuda.synchronize()
            got = gu.to_host(yd[:M * N].reshape(M, N), dtype)
            xs = gu.to_host(xd[:M * N].reshape(M, N), dtype)
            gu.check_rows(got, xs, N, N, dtype, "shifted N=%d k=%d" % (N, k))
            # Nothing written outside the M rows.
            assert torch.isnan(yb[:k]).all() and torch.isnan(yd[M * N:]).all()


# ---- edge shapes: widths around every plan boundary, odd row counts ----

EDGE_N = [1, 2, 3, 7, 31, 33, 127, 255, 1000, 2047, 2048, 2049, 4095, 4104, 8192, 8193, 16384,
          16392, 20480, 24576, 32769, 65536]


@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16, synth.F16], ids=["f32", "bf16", "f16"])
@pytest.mark.parametrize("N", EDGE_N)
def test_edge_shapes(dtype, N):
    for M in (1, 3, 157):
        if M * N > 4_000_000:
            continue
        x = synth.generate(M, N, dtype=dtype, seed=N * 7 + M, p1=3.0)
        xd = gu.to_device(x, dtype)
        for plan in PLANS:
            y = nan_filled(M, N, dtype)
            if not plan_applies(xd, y, M, N, N, N, dtype, plan):
                continue
            st, y = run_plan(xd, M, N, N, N, dtype, plan, out=y)
            assert st == sr.SR_OK
            torch.cuda.synchronize()
            gu.check_rows(gu.to_host(y, dtype), x, N, N, dtype,
                          "edge M=%d N=%d plan %s" % (M, N, sr.PLAN_NAMES[plan]))


@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16, synth.F16], ids=["f32", "bf16", "f16"])
@pytest.mark.parametrize("N", [100, 1000, 2048, 5000, 40000])
def test_misaligned_rows(dtype, N):
    """Rows not 16-byte aligned (one-element offsets, odd pitches) take the scalar plans."""
    M = 37
    ld_in, ld_out = N + 1, N + 3
    x = synth.generate(M, N, ld=ld_in, dtype=dtype, seed=N + 3, p1=2.0)
    base_in = gu.to_device(np.concatenate([x.reshape(-1)[:1], x.reshape(-1)]), dtype)
    xd = base_in[1:]  # one element past a 16-byte boundary
    yb = torch.full((M * ld_out + 1,), float("nan"), dtype=gu.torch_dtype(dtype), device="cuda")
    yd = yb[1:]
    for plan in PLANS:
        if not plan_applies(xd, yd, M, N, ld_in, ld_out, dtype, plan):
            assert plan in (sr.SR_PLAN_CTA, sr.SR_PLAN_CLUSTER, sr.SR_PLAN_WARP, sr.SR_PLAN_SMEM,
                            sr.SR_PLAN_ROW, sr.SR_PLAN_WIDE)
            continue
        yb.fill_(float("nan"))
        st = sr.load().softmax_rows_ex(xd.data_ptr(), yd.data_ptr(), M, N, ld_in, ld_out, dtype,
                                       plan, torch.cuda.current_stream().cuda_stream)
        assert st == sr.SR_OK
        torch.cuda.synchronize()
        out = gu.to_host(yd, dtype).reshape(M, ld_out)
        gu.check_rows(out, x, N, ld_in, dtype, "misaligned N=%d plan %s" % (N, sr.PLAN_NAMES[plan]))
        assert torch.isnan(yd.view(M, ld_out)[:, N:]).all(), "pad columns written"
        assert torch.isnan(yb[:1]).all()


# ---- rows whose answer is fixed by the definition ----

def special_rows(N, dtype):
    rows = []
    rows.append(np.full(N, -math.inf))                       # all -inf -> NaN
    r = np.linspace(-2, 2, N); r[N // 3] = math.nan; rows.append(r)   # NaN -> NaN row
    r = np.linspace(-2, 2, N); r[N // 2] = math.inf; rows.append(r)   # +inf -> NaN row
    rows.append(np.zeros(N))                                 # uniform -> 1/N
    r = np.full(N, -math.inf); r[[0, N // 2, N - 1]] = 3.0; rows.append(r)  # 3 tied maxima
    r = np.full(N, -math.inf); r[: max(1, N // 5)] = np.linspace(-1, 1, max(1, N // 5))
    rows.append(r)                                           # masked suffix (causal row)
    r = np.full(N, -math.inf); r[-1] = -7.0; rows.append(r)  # single finite entry -> 1
    r = np.linspace(-100, 100, N); rows.append(r)            # extreme logits
    from tests import pins
    return pins.to_grid(np.array(rows), dtype)


@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16, synth.F16], ids=["f32", "bf16", "f16"])
@pytest.mark.parametrize("N", [5, 1000, 4096, 16384, 40000])
def test_special_rows(dtype, N):
    from tests import pins
    vals = special_rows(N, dtype)
    M = vals.shape[0]
    x = pins.encode_exact(vals, dtype)
    xd = gu.to_device(x, dtype)
    for plan in PLANS:
        y = nan_filled(M, N, dtype)
        if not plan_applies(xd, y, M, N, N, N, dtype, plan):
            continue
        st, y = run_plan(xd, M, N, N, N, dtype, plan, out=y)
        assert st == sr.SR_OK
        torch.cuda.synchronize()
        out = gu.to_host(y, dtype)
        ref = gu.check_rows(out, x, N, N, dtype, "special N=%d plan %s" % (N, sr.PLAN_NAMES[plan]))
        g = synth.storage_to_float64(out, dtype)
        assert np.isnan(g[0]).all() and np.isnan(g[1]).all() and np.isnan(g[2]).all()
        # Uniform row: the FP32 reciprocal of N rounded once to the dtype; for
        # bf16/f16 that is the oracle's value unless rounding 1/N to binary32
        # first lands on a tie of the 16-bit format.
        want = {pins.to_grid([np.float32(1.0) / np.float32(N)], dtype)[0],
                synth.storage_to_float64(ref[3:4, :1], dtype)[0, 0]}
        assert set(np.unique(g[3])) <= want, (plan, np.unique(g[3]), want)
        assert np.all(g[4][vals[4] == -math.inf] == 0.0)
        assert np.all(g[5][vals[5] == -math.inf] == 0.0)
        assert g[6][-1] == 1.0 and np.all(g[6][:-1] == 0.0)


# ---- rows too wide for a cluster's registers: the streamed WIDE kernel ----

@pytest.mark.parametrize("dtype,M,N", [(synth.BF16, 3, 600008), (synth.F32, 2, 300000),
                                       (synth.F16, 9, 600000), (synth.BF16, 20, 1048576)],
                         ids=lambda v: str(v))
def test_streamed_wide_rows(dtype, M, N):
    from tests import pins
    x = synth.generate(M, N, dtype=dtype, seed=N + M, p1=3.0)
    sp = pins.encode_exact(special_rows(N, dtype), dtype)
    k = min(M, sp.shape[0])
    x[:k] = sp[:k]  # all -inf, a NaN, a +inf, uniform, tied maxima, ... as rows allow
    xd = gu.to_device(x, dtype)
    assert sr.softmax_rows_plan(xd, xd, M, N, N, N, dtype) == sr.SR_PLAN_WIDE
    st, y = run_plan(xd, M, N, N, N, dtype, sr.SR_PLAN_AUTO)
    assert st == sr.SR_OK
    torch.cuda.synchronize()
    out = gu.to_host(y, dtype)
    gu.check_rows(out, x, N, N, dtype, "streamed %dx%d" % (M, N))
    g = synth.storage_to_float64(out[:k], dtype)
    assert np.isnan(g[0]).all()
    if k > 2:
        assert np.isnan(g[1]).all() and np.isnan(g[2]).all()
    assert sr.softmax_rows_last_device_error() == sr.SR_OK


def test_streamed_wide_in_place():
    """in == out: every block finishes its first pass over a row before any block
    writes it (the pair exchange orders them), so the second pass still reads x."""
    M, N, dtype = 5, 300000, synth.F32
    x = synth.generate(M, N, dtype=dtype, seed=91, p1=3.0)
    buf = gu.to_device(x, dtype)
    st = sr.load().softmax_rows_ex(buf.data_ptr(), buf.data_ptr(), M, N, N, N, dtype,
                                   sr.SR_PLAN_WIDE, torch.cuda.current_stream().cuda_stream)
    assert st == sr.SR_OK
    torch.cuda.synchronize()
    gu.check_rows(gu.to_host(buf, dtype), x, N, N, dtype, "streamed in place")


def test_streamed_wide_wait_expiry():
    M, N, dtype = 3, 600008, synth.BF16
    x = synth.generate(M, N, dtype=dtype, seed=77, p1=2.0)
    xd = gu.to_device(x, dtype)
    y = nan_filled(M, N, dtype)
    assert sr.softmax_rows_last_device_error() == sr.SR_OK
    sr.softmax_rows_test_expiry(xd, y, M, N, N, N, dtype, sr.SR_PLAN_WIDE, 2_000_000)
    assert sr.softmax_rows_last_device_error() == sr.SR_EDEVICE_TIMEOUT
    assert torch.isnan(y).all(), "an expired kernel wrote output"
    sr.softmax_rows_ex(xd, y, M, N, N, N, dtype, sr.SR_PLAN_WIDE)
    torch.cuda.synchronize()
    gu.check_rows(gu.to_host(y, dtype), x, N, N, dtype, "streamed after expiry")
    assert sr.softmax_rows_last_device_error() == sr.SR_OK



# Streamed rows with enough rows for 8-block clusters take the bulk-copy ring
# kernel: 800 KB rows at 3 blocks/SM, 1.2 MB rows at 2 (their resident rows
# would not fit in half the L2 at 3), ragged chunks at the end of each slice.
@pytest.mark.parametrize("dtype,M,N", [(synth.F16, 96, 400000), (synth.BF16, 80, 600008),
                                       (synth.F32, 80, 300000), (synth.F32, 77, 262148)],
                         ids=lambda v: str(v))
def test_streamed_bulk_rows(dtype, M, N):
    from tests import pins
    x = synth.generate(M, N, dtype=dtype, seed=N + 3 * M, p1=3.0)
    sp = pins.encode_exact(special_rows(N, dtype), dtype)
    x[M - sp.shape[0]:] = sp  # special rows at the end, on the last clusters
    xd = gu.to_device(x, dtype)
    st, y = run_plan(xd, M, N, N, N, dtype, sr.SR_PLAN_AUTO)
    assert st == sr.SR_OK
    torch.cuda.synchronize()
    assert "wide_bulk_kernel" in sr.softmax_rows_last_launch()["name"]
    gu.check_rows(gu.to_host(y, dtype), x, N, N, dtype, "bulk streamed %dx%d" % (M, N))
    assert sr.softmax_rows_last_device_error() == sr.SR_OK


def test_streamed_bulk_in_place():
    M, N, dtype = 96, 400008, synth.BF16
    x = synth.generate(M, N, dtype=dtype, seed=93, p1=3.0)
    buf = gu.to_device(x, dtype)
    st = sr.load().softmax_rows_ex(buf.data_ptr(), buf.data_ptr(), M, N, N, N, dtype,
                                   sr.SR_PLAN_WIDE, torch.cuda.current_stream().cuda_stream)
    assert st == sr.SR_OK
    torch.cuda.synchronize()
    assert "wide_bulk_kernel" in sr.softmax_rows_last_launch()["name"]
    gu.check_rows(gu.to_host(buf, dtype), x, N, N, dtype, "bulk streamed in place")


def test_streamed_bulk_wait_expiry():
    M, N, dtype = 80, 600008, synth.BF16
    x = synth.generate(M, N, dtype=dtype, seed=79, p1=2.0)
    xd = gu.to_device(x, dtype)
    y = nan_filled(M, N, dtype)
    assert sr.softmax_rows_last_device_error() == sr.SR_OK
    sr.softmax_rows_test_expiry(xd, y, M, N, N, N, dtype, sr.SR_PLAN_WIDE, 2_000_000)
    assert sr.softmax_rows_last_device_error() == sr.SR_EDEVICE_TIMEOUT
    assert "wide_bulk_kernel" in sr.softmax_rows_last_launch()["name"]
    assert torch.isnan(y).all(), "an expired kernel wrote output"
    sr.softmax_rows_ex(xd, y, M, N, N, N, dtype, sr.SR_PLAN_WIDE)
    torch.cuda.synchronize()
    gu.check_rows(gu.to_host(y, dtype), x, N, N, dtype, "bulk streamed after expiry")
    assert sr.softmax_rows_last_device_error() == sr.SR_OK

# ---- many short rows: the WARP plan's shared-lane layouts ----

# Rows of at most 64 vectors with rows enough for 4 blocks per SM are taken by
# 8 lanes (<= 32 vectors) or 16 lanes (<= 64 vectors) each. The row counts are
# ragged, so the last warp holds row groups past M, and the widths leave lanes
# of a group without a vector. Special rows sit at both ends of the matrix.
@pytest.mark.parametrize("dtype,M,N", [(synth.BF16, 20003, 256), (synth.F32, 20003, 128),
                                       (synth.BF16, 20001, 40), (synth.F16, 9999, 512),
                                       (synth.F32, 9731, 200), (synth.F16, 300, 512)],
                         ids=lambda v: str(v))
def test_short_rows_shared_lanes(dtype, M, N):
    from tests import pins
    w = synth.Workload("short", dtype, M, N, N, N, 21, synth.DIST_NORMAL, 0.0, 1.0)
    x = w.generate()
    sp = pins.encode_exact(special_rows(N, dtype), dtype)
    k = sp.shape[0]
    x[:k] = sp
    x[M - k:] = sp
    xd = gu.to_device(x, dtype)
    for plan in (sr.SR_PLAN_AUTO, sr.SR_PLAN_WARP):
        assert sr.softmax_rows_plan(xd, xd, M, N, N, N, dtype) == sr.SR_PLAN_WARP
        st, y = run_plan(xd, M, N, N, N, dtype, plan)
        assert st == sr.SR_OK
        torch.cuda.synchronize()
        out = gu.to_host(y, dtype)
        gu.check_rows(out, x, N, N, dtype, "short rows %dx%d plan %s" % (M, N, sr.PLAN_NAMES[plan]))
        g = synth.storage_to_float64(out, dtype)
        assert np.isnan(g[0]).all() and np.isnan(g[M - k]).all()
        assert g[k - 2][-1] == 1.0 and g[M - 2][-1] == 1.0
    assert sr.softmax_rows_last_device_error() == sr.SR_OK


# ---- in place, canaries, streams, empty and rejected calls ----

@pytest.mark.parametrize("name", ["f32_4096x4096", "bf16_16384x1000_ld1024", "bf16_1024x131072",
                                  "f16_causal_524288x2048"])
def test_in_place(name):
    w = synth.WORKLOADS[name].with_rows(24)
    x = w.generate()
    for plan in PLANS:
        buf = gu.to_device(x, w.dtype)
        if not plan_applies(buf, buf, w.M, w.N, w.ld_in, w.ld_in, w.dtype, plan):
            continue
        st = sr.load().softmax_rows_ex(buf.data_ptr(), buf.data_ptr(), w.M, w.N, w.ld_in, w.ld_in,
                                       w.dtype, plan, torch.cuda.current_stream().cuda_stream)
        assert st == sr.SR_OK
        torch.cuda.synchronize()
        gu.check_rows(gu.to_host(buf, w.dtype), x, w.N, w.ld_in, w.dtype,
                      "in place %s plan %s" % (name, sr.PLAN_NAMES[plan]))


def test_guard_regions_untouched():
    """Bytes before and after the output and its pad columns stay bit-identical."""
    for name in FULL[:4]:
        w = synth.WORKLOADS[name].with_rows(33)
        x = w.generate()
        xd = gu.to_device(x, w.dtype)
        ld_out = w.N + 64
        guard = 4096
        total = guard + w.M * ld_out + guard
        big = torch.full((total,), 0.125, dtype=gu.torch_dtype(w.dtype), device="cuda")
        yd = big[guard:guard + w.M * ld_out]
        for plan in PLANS:
            if not plan_applies(xd, yd, w.M, w.N, w.ld_in, ld_out, w.dtype, plan):
                continue
            big.fill_(0.125)
            st = sr.load().softmax_rows_ex(xd.data_ptr(), yd.data_ptr(), w.M, w.N, w.ld_in, ld_out,
                                           w.dtype, plan, torch.cuda.current_stream().cuda_stream)
            assert st == sr.SR_OK
            torch.cuda.synchronize()
            assert (big[:guard] == 0.125).all() and (big[-guard:] == 0.125).all()
            assert (yd.view(w.M, ld_out)[:, w.N:] == 0.125).all()
            gu.check_rows(gu.to_host(yd, w.dtype).reshape(w.M, ld_out), x, w.N, w.ld_in, w.dtype,
                          "guard %s plan %s" % (name, sr.PLAN_NAMES[plan]))


def test_side_stream_and_empty_calls():
    w = synth.WORKLOADS["f32_4096x4096"].with_rows(50)
    x = w.generate()
    xd = gu.to_device(x, w.dtype)
    y = nan_filled(w.M, w.N, w.dtype)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        st = sr.load().softmax_rows(xd.data_ptr(), y.data_ptr(), w.M, w.N, w.N, w.N, w.dtype,
                                    s.cuda_stream)
    assert st == sr.SR_OK
    s.synchronize()
    gu.check_rows(gu.to_host(y, w.dtype), x, w.N, w.N, w.dtype, "side stream")
    y2 = nan_filled(4, 8, synth.F32)
    assert sr.load().softmax_rows(xd.data_ptr(), y2.data_ptr(), 0, 8, 8, 8, 0, None) == sr.SR_OK
    assert sr.load().softmax_rows(xd.data_ptr(), y2.data_ptr(), 4, 8, 4, 8, 0, None) == sr.SR_EINVAL
    assert sr.load().softmax_rows(xd.data_ptr(), y2.data_ptr(), 4, 8, 8, 8, 7, None) == sr.SR_EDTYPE
    torch.cuda.synchronize()
    assert torch.isnan(y2).all()


# ---- aligned rows of 1 MiB: the staged WIDE variant (16-block clusters, half of
# each block's slice in shared memory) ----

@pytest.mark.parametrize("dtype,M,N,csize", [(synth.BF16, 130, 524288, 16),
                                             (synth.F32, 77, 262144, 16),
                                             (synth.F16, 3, 524288, 16)],
                         ids=["bf16", "f32", "f16-few-rows"])
def test_wide_staged_rows(dtype, M, N, csize):
    x = synth.generate(M, N, dtype=dtype, seed=700 + M, p1=2.0)
    xd = gu.to_device(x, dtype)
    st, y = run_plan(xd, M, N, N, N, dtype, sr.SR_PLAN_AUTO)
    assert st == sr.SR_OK
    torch.cuda.synchronize()
    info = sr.softmax_rows_last_launch()
    assert "wide_staged_kernel" in info["name"] and info["cluster"] == csize
    gu.check_rows(gu.to_host(y, dtype), x, N, N, dtype, "staged WIDE")
    assert sr.softmax_rows_last_device_error() == sr.SR_OK


def test_wide_staged_in_place():
    """in == out: each block reads its whole slice (registers and shared memory)
    before the exchange and writes only its own slice after it."""
    M, N, dtype = 6, 524288, synth.BF16
    x = synth.generate(M, N, dtype=dtype, seed=93, p1=2.0)
    buf = gu.to_device(x, dtype)
    st = sr.load().softmax_rows_ex(buf.data_ptr(), buf.data_ptr(), M, N, N, N, dtype,
                                   sr.SR_PLAN_AUTO, torch.cuda.current_stream().cuda_stream)
    assert st == sr.SR_OK
    torch.cuda.synchronize()
    assert "wide_staged_kernel" in sr.softmax_rows_last_launch()["name"]
    gu.check_rows(gu.to_host(buf, dtype), x, N, N, dtype, "staged WIDE in place")


def test_wide_staged_wait_expiry():
    M, N, dtype = 8, 524288, synth.BF16
    x = synth.generate(M, N, dtype=dtype, seed=32)
    xd = gu.to_device(x, dtype)
    y = nan_filled(M, N, dtype)
    assert sr.softmax_rows_last_device_error() == sr.SR_OK
    sr.softmax_rows_test_expiry(xd, y, M, N, N, N, dtype, sr.SR_PLAN_WIDE, 2_000_000)
    assert sr.softmax_rows_last_device_error() == sr.SR_EDEVICE_TIMEOUT
    assert "wide_staged_kernel" in sr.softmax_rows_last_launch()["name"]
    assert torch.isnan(y).all(), "an expired kernel wrote output"
    st, y = run_plan(xd, M, N, N, N, dtype, sr.SR_PLAN_WIDE)
    assert st == sr.SR_OK
    torch.cuda.synchronize()
    gu.check_rows(gu.to_host(y, dtype), x, N, N, dtype, "after expiry")
    assert sr.softmax_rows_last_device_error() == sr.SR_OK


# ---- the bounded wait: an expiring wait reports an error, the context survives ----

@pytest.mark.parametrize("name,plan", [("f32_4096x4096", sr.SR_PLAN_CTA),
                                       ("bf16_1024x131072", sr.SR_PLAN_CLUSTER),
                                       ("bf16_1024x131072", sr.SR_PLAN_WIDE),
                                       ("f32_4096x4096", sr.SR_PLAN_SMEM),
                                       ("f16_causal_524288x2048", sr.SR_PLAN_SMEM)])
def test_bounded_wait_expiry(name, plan):
    w = synth.WORKLOADS[name].with_rows(5)
    x = w.generate()
    xd = gu.to_device(x, w.dtype)
    y = nan_filled(w.M, w.N, w.dtype)
    assert sr.softmax_rows_last_device_error() == sr.SR_OK
    sr.softmax_rows_test_expiry(xd, y, w.M, w.N, w.ld_in, w.ld_out, w.dtype, plan, 2_000_000)
    assert sr.softmax_rows_last_device_error() == sr.SR_EDEVICE_TIMEOUT
    assert torch.isnan(y).all(), "an expired kernel wrote output"
    assert sr.softmax_rows_last_device_error() == sr.SR_OK  # the word was cleared
    sr.softmax_rows_ex(xd, y, w.M, w.N, w.ld_in, w.ld_out, w.dtype, plan)
    torch.cuda.synchronize()
    gu.check_rows(gu.to_host(y, w.dtype), x, w.N, w.ld_in, w.dtype, "after expiry")
    assert sr.softmax_rows_last_device_error() == sr.SR_OK
