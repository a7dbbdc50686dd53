"""softmax_rows_masked (per-row lengths or a causal period) against the masked oracle.

Masked entries of every input hold NaN: a kernel that read one would produce
NaN where the oracle (which never reads them) has finite values.
"""
import numpy as np
import pytest

import memory_bound_row_rows_gb300 as sr
import oracle
import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

MASKED_PLANS = [sr.SR_PLAN_AUTO, sr.SR_PLAN_WARP, sr.SR_PLAN_ROW, sr.SR_PLAN_ONLINE]
NAN_BITS = {synth.F32: np.float32(np.nan), synth.BF16: np.uint16(0x7FC0),
            synth.F16: np.uint16(0x7E00)}


def poisoned(x, lens, N, dtype):
    x = x.copy()
    for i, L in enumerate(lens):
        x[i, max(0, min(int(L), N)):N] = NAN_BITS[dtype]
    return x


def check(out, x, M, N, ld_in, dtype, lens=None, period=0, label=""):
    ref = oracle.load().softmax_rows_masked(np.ascontiguousarray(x).reshape(-1), M, N, ld_in, N,
                                            dtype, lens=lens, causal_period=period,
                                            nthreads=synth.host_threads())
    g = synth.storage_to_float64(out[:, :N], dtype)
    r = synth.storage_to_float64(ref, dtype)
    ok, nbad, rep = gu.gate(g, r, dtype)
    assert ok, "%s: %d elements outside the gate (max %.3g)" % (label, nbad, rep["max_abs"])
    return r


def run_masked(xd, M, N, ld_in, ld_out, dtype, lens_d=None, period=0, plan=0):
    y = torch.full((M, ld_out), float("nan"), dtype=gu.torch_dtype(dtype), device="cuda")
    st = sr.load().softmax_rows_masked(xd.data_ptr(), y.data_ptr(), M, N, ld_in, ld_out, dtype,
                                       0 if lens_d is None else lens_d.data_ptr(), period, plan,
                                       torch.cuda.current_stream().cuda_stream)
    return st, y


@pytest.mark.parametrize("plan", MASKED_PLANS, ids=lambda p: sr.PLAN_NAMES[p])
def test_causal_rows_with_poisoned_mask(plan):
    w = synth.WORKLOADS["f16_causal_524288x2048"]
    row0, M = 1000, 2200
    x = w.rows(row0, M)  # causal -inf beyond each row's length
    lens = np.array([(row0 + i) % 2048 + 1 for i in range(M)], dtype=np.int32)
    xp = poisoned(x, lens, w.N, w.dtype)
    # The rows start at row0, so pass explicit lengths (the causal period counts from row 0).
    xd = gu.to_device(xp, w.dtype)
    ld = torch.from_numpy(lens).cuda()
    st, y = run_masked(xd, M, w.N, w.N, w.N, w.dtype, lens_d=ld, plan=plan)
    if st == sr.SR_EPLAN:
        assert plan == sr.SR_PLAN_WARP or plan == sr.SR_PLAN_ROW
        return
    assert st == sr.SR_OK
    torch.cuda.synchronize()
    out = gu.to_host(y, w.dtype)
    r = check(out, xp, M, w.N, w.N, w.dtype, lens=lens, label="causal poisoned")
    # Same as the plain softmax of the -inf-masked data.
    plain = oracle.softmax_rows(x.reshape(-1), M, w.N, w.N, w.N, w.dtype)
    assert np.array_equal(synth.storage_to_float64(plain, w.dtype), r)


def test_causal_period_from_row_zero():
    w = synth.WORKLOADS["f16_causal_524288x2048"]
    M = 4200
    x = w.rows(0, M)
    lens = np.array([i % 2048 + 1 for i in range(M)], dtype=np.int32)
    xp = poisoned(x, lens, w.N, w.dtype)
    xd = gu.to_device(xp, w.dtype)
    for plan in MASKED_PLANS:
        st, y = run_masked(xd, M, w.N, w.N, w.N, w.dtype, period=2048, plan=plan)
        assert st == sr.SR_OK
        torch.cuda.synchronize()
        check(gu.to_host(y, w.dtype), xp, M, w.N, w.N, w.dtype, period=2048,
              label="causal period plan %s" % sr.PLAN_NAMES[plan])


@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16, synth.F16], ids=["f32", "bf16", "f16"])
@pytest.mark.parametrize("N", [5, 100, 1000, 2048, 4096, 5000, 40000])
def test_random_lengths(dtype, N):
    rng = np.random.default_rng(N + 7 * dtype)
    M = 61
    x = synth.generate(M, N, dtype=dtype, seed=N * 3 + dtype, p1=3.0)
    lens = rng.integers(0, N + 10, size=M).astype(np.int32)
    lens[:4] = [0, 1, N, N + 100]
    xp = poisoned(x, lens, N, dtype)
    xd = gu.to_device(xp, dtype)
    ld = torch.from_numpy(lens).cuda()
    for plan in MASKED_PLANS:
        st, y = run_masked(xd, M, N, N, N, dtype, lens_d=ld, plan=plan)
        if st == sr.SR_EPLAN:
            continue
        assert st == sr.SR_OK
        torch.cuda.synchronize()
        out = gu.to_host(y, dtype)
        check(out, xp, M, N, N, dtype, lens=lens, label="lengths N=%d plan %s" % (
            N, sr.PLAN_NAMES[plan]))
        g = synth.storage_to_float64(out, dtype)
        assert np.all(np.isnan(g[0])), "a length-0 row is all -inf: NaN"
        assert g[1][0] == 1.0 and np.all(g[1][1:] == 0.0)


def test_masked_misaligned_and_errors():
    dtype, M, N = synth.BF16, 33, 3001
    x = synth.generate(M, N, ld=N + 1, dtype=dtype, seed=5, p1=2.0)
    lens = np.arange(M, dtype=np.int32) * 97
    xp = poisoned(x, lens, N, dtype)
    base = gu.to_device(np.concatenate([xp.reshape(-1)[:1], xp.reshape(-1)]), dtype)
    xd = base[1:]
    ld = torch.from_numpy(lens).cuda()
    st, y = run_masked(xd, M, N, N + 1, N, dtype, lens_d=ld)
    assert st == sr.SR_OK
    torch.cuda.synchronize()
    check(gu.to_host(y, dtype), xp, M, N, N + 1, dtype, lens=lens, label="misaligned")
    L = sr.load()
    s = torch.cuda.current_stream().cuda_stream
    assert L.softmax_rows_masked(xd.data_ptr(), y.data_ptr(), M, N, N + 1, N, dtype,
                                 ld.data_ptr(), 2048, 0, s) == sr.SR_EINVAL
    assert L.softmax_rows_masked(xd.data_ptr(), y.data_ptr(), M, N, N + 1, N, dtype,
                                 None, -1, 0, s) == sr.SR_EINVAL
    assert L.softmax_rows_masked(xd.data_ptr(), y.data_ptr(), M, N, N + 1, N, dtype,
                                 ld.data_ptr(), 0, sr.SR_PLAN_CLUSTER, s) == sr.SR_EPLAN


def test_full_causal_workload_masked_sampled():
    w = synth.WORKLOADS["f16_causal_524288x2048"]
    x = w.generate()
    xd = gu.to_device(x, w.dtype)
    st, y = run_masked(xd, w.M, w.N, w.N, w.N, w.dtype, period=2048)
    assert st == sr.SR_OK
    torch.cuda.synchronize()
    rng = np.random.default_rng(3)
    sample = np.unique(np.concatenate([np.arange(64), np.arange(w.M - 64, w.M),
                                       rng.integers(0, w.M, 128)]))
    ys = gu.to_host(y[torch.from_numpy(sample).cuda()], w.dtype)
    check(ys, x[sample], len(sample), w.N, w.N, w.dtype,
          lens=np.array([r % 2048 + 1 for r in sample], dtype=np.int32), label="full causal")
