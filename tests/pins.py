"""The pins that hold the oracle to the mathematics, not to itself.

Each ``check_*`` takes an ``oracle.Oracle`` (the real library, or a mutant
compiled by the mutation test) and raises AssertionError on a mismatch. What
each compares against:

* 60-digit ``decimal`` softmax with exact ``Fraction`` rounding (brute.py);
* closed forms: a constant row gives round(1/N); two entries give the
  logistic 1/(1+e^(b-a)); k tied maxima with the rest -inf give 1/k; a causal
  attention row q has exactly q+1 nonzeros; an all -inf, NaN or +inf row is
  NaN (the definition);
* invariants: rows sum to 1 within the dtype's rounding, outputs lie in
  [0, 1], the argmax is kept, a shift by a constant changes nothing (bit for
  bit on a dyadic grid), the pad columns are never read or written, and the
  thread count does not change the bits;
* numpy's own decoders for every f16 / bf16 bit pattern.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np

import synth
from tests import brute

F32, BF16, F16 = 0, 1, 2
DTYPES = (F32, BF16, F16)
UNIT_ROUNDOFF = {F32: 2.0 ** -24, BF16: 2.0 ** -9, F16: 2.0 ** -11}


# ---- encoding helpers (test side) --------------------------------------------

def encode_exact(values, dtype: int) -> np.ndarray:
    """Store values that are exactly representable in the dtype (asserted)."""
    v = np.asarray(values, dtype=np.float64)
    if dtype == F32:
        out = v.astype(np.float32)
        assert np.array_equal(out.astype(np.float64), v, equal_nan=True)
        return out
    if dtype == F16:
        h = v.astype(np.float16)
        assert np.array_equal(h.astype(np.float64), v, equal_nan=True)
        return h.view(np.uint16)
    f = v.astype(np.float32)
    assert np.array_equal(f.astype(np.float64), v, equal_nan=True)
    bits = f.view(np.uint32)
    assert np.all((bits & 0xFFFF) == 0) or np.all(np.isnan(v[(bits & 0xFFFF) != 0]))
    return (bits >> 16).astype(np.uint16)


def decode(a: np.ndarray, dtype: int) -> np.ndarray:
    return synth.storage_to_float64(np.asarray(a), dtype)


def to_grid(values, dtype: int) -> np.ndarray:
    """Round float64 values onto the dtype's grid (numpy's own conversions)."""
    v = np.asarray(values, dtype=np.float64)
    if dtype == F32:
        return v.astype(np.float32).astype(np.float64)
    if dtype == F16:
        return v.astype(np.float16).astype(np.float64)
    f = v.astype(np.float32)
    bits = f.view(np.uint32).astype(np.uint64)
    bits = (bits + 0x7FFF + ((bits >> 16) & 1)) >> 16 << 16
    return bits.astype(np.uint32).view(np.float32).astype(np.float64)


def run_rows(orc, rows_values, dtype: int) -> np.ndarray:
    """Oracle output (decoded to float64) for a list of equal-length rows."""
    x = encode_exact(np.asarray(rows_values, dtype=np.float64), dtype)
    M, N = x.shape
    return decode(orc.softmax_rows(x.reshape(-1), M, N, N, N, dtype), dtype)


def same(a, b) -> bool:
    return np.array_equal(np.asarray(a), np.asarray(b), equal_nan=True)


# ---- step 1 and step 5 alone ------------------------------------------------

def check_decode(orc):
    pats = np.arange(65536, dtype=np.uint16)
    got = orc.decode(pats, F16)
    with np.errstate(invalid="ignore"):  # NaN payloads warn on some platforms
        want = pats.view(np.float16).astype(np.float64)
    assert same(got, want), "f16 decode"
    got = orc.decode(pats, BF16)
    with np.errstate(invalid="ignore"):
        want = (pats.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert same(got, want), "bf16 decode"
    rng = np.random.default_rng(7)
    f = rng.integers(0, 2**32, 4096, dtype=np.uint64).astype(np.uint32).view(np.float32)
    with np.errstate(invalid="ignore"):
        want = f.astype(np.float64)
    assert same(orc.decode(f, F32), want), "f32 decode"


def cast_cases(dtype: int) -> np.ndarray:
    p, emin, emax = brute.FORMATS[dtype]
    one = [1.0, 0.0, -0.0, 0.5, 1.0 / 3.0, 2.0 / 3.0, 0.1, 1e-3, 1e-6, 1e-8]
    ulp1 = 2.0 ** (1 - p)
    ties = [1 + ulp1 / 2, 1 + 3 * ulp1 / 2, 0.75 + ulp1 / 4, 1 - ulp1 / 4]
    # Just above a tie once rounded to binary32: a cast through float would
    # land on the tie and round to even, the single rounding must go up.
    traps = [1 + ulp1 / 2 + 2.0 ** -40, 1 + 3 * ulp1 / 2 - 2.0 ** -40]
    tiny = 2.0 ** (emin - p + 1)  # smallest subnormal
    subn = [tiny, tiny / 2, tiny * 0.75, tiny * 1.5, tiny * 2.5, 2.0 ** emin * (1 - ulp1 / 4),
            2.0 ** emin * (1 - ulp1), 2.0 ** emin]
    big = 2.0 ** emax * (2 - ulp1)
    over = [big, big * (1 + ulp1 / 8), big * (1 + ulp1 / 4 + 1e-9), 2.0 ** (emax + 1) * 1.5]
    rng = np.random.default_rng(11 + dtype)
    rnd = list(rng.uniform(0, 1, 300)) + list(np.exp(rng.uniform(math.log(tiny), math.log(big), 300)))
    vals = one + ties + traps + subn + over + rnd
    vals = vals + [-v for v in vals] + [math.inf, -math.inf]
    return np.array(vals, dtype=np.float64)


def check_cast(orc):
    for dtype in DTYPES:
        v = cast_cases(dtype)
        got = decode(orc.cast(v, dtype), dtype)
        want = np.array([brute.round_exact(Fraction(x), dtype) if math.isfinite(x) else x
                         for x in v])
        bad = np.nonzero(~((got == want) | (np.isnan(got) & np.isnan(want))))[0]
        assert bad.size == 0, "cast dtype %d: %r -> %r, want %r" % (
            dtype, v[bad[:3]], got[bad[:3]], want[bad[:3]])
        assert np.isnan(decode(orc.cast(np.array([math.nan]), dtype), dtype)[0])


# ---- brute force ------------------------------------------------------------

def _brute_compare(orc, rows, dtype: int, label: str):
    rows = np.asarray(rows, dtype=np.float64)
    got = run_rows(orc, rows, dtype)
    x = encode_exact(rows, dtype)
    got64 = orc.softmax_rows_f64(x.reshape(-1), rows.shape[0], rows.shape[1], rows.shape[1], dtype)
    for i, row in enumerate(rows):
        want = brute.softmax_exact_cast(row, dtype)
        assert same(got[i], want), "%s dtype %d row %d: %r vs %r" % (label, dtype, i, got[i], want)
        w64 = brute.softmax_decimal_f64(row)
        fin = np.isfinite(w64)
        assert same(np.isnan(got64[i]), np.isnan(w64)), label
        assert np.allclose(got64[i][fin], w64[fin], rtol=1e-14, atol=0), (
            "%s f64 dtype %d row %d" % (label, dtype, i))


def check_brute_random(orc):
    for dtype in DTYPES:
        for N in (1, 2, 3, 5, 8, 13, 16):
            for seed, sigma in ((1, 1.0), (2, 3.0), (3, 10.0)):
                vals = synth.storage_to_float64(
                    synth.generate(4, N, dtype=dtype, seed=seed * 100 + N, p1=sigma), dtype)
                _brute_compare(orc, vals, dtype, "random N=%d" % N)


def check_brute_extremes(orc):
    for dtype in DTYPES:
        rows = [
            [100.0, -100.0, 99.0, 0.0, -0.5, 100.0, 37.0, -99.0],
            [10000.0, 9999.0 if dtype != BF16 else 9984.0, -10000.0, 0.0, 10000.0, 1.0, 2.0, 3.0],
            [-10000.0, -10000.0, -9984.0, -10000.0, -10000.0, -10000.0, -10000.0, -10000.0],
            [-math.inf, 2.0, -math.inf, -1.0, 0.25, -math.inf, -math.inf, 3.0],
            [-math.inf, -math.inf, -math.inf, -math.inf, -math.inf, -math.inf, -math.inf, -40.0],
            [1.0, 1.0, 1.0, 1.0, 1.0, 1.0, 1.0, 1.0],
        ]
        _brute_compare(orc, to_grid(rows, dtype), dtype, "extremes")


# ---- closed forms -------------------------------------------------------------

def check_uniform_rows(orc):
    for dtype in DTYPES:
        for N in (1, 2, 3, 7, 100, 1000, 4096, 5000):
            want = brute.round_exact(Fraction(1, N), dtype)
            for c in (0.0, -3.5, 100.0, -9984.0):
                got = run_rows(orc, np.full((1, N), c), dtype)
                assert np.all(got == want), "uniform dtype %d N=%d c=%g" % (dtype, N, c)


def check_two_entries(orc):
    import decimal
    for dtype in DTYPES:
        for a, b in ((0.0, 1.0), (2.5, -3.0), (10.0, 10.0), (-7.25, 0.5), (0.0, 20.0)):
            with decimal.localcontext(brute.CTX):
                d = decimal.Decimal(b) - decimal.Decimal(a)
                y0 = 1 / (1 + d.exp())
                y1 = 1 / (1 + (-d).exp())
            want = [brute.round_exact(Fraction(y0), dtype), brute.round_exact(Fraction(y1), dtype)]
            got = run_rows(orc, [[a, b]], dtype)[0]
            assert same(got, want), "two entries dtype %d (%g, %g): %r vs %r" % (dtype, a, b, got, want)


def check_tied_maxima(orc):
    for dtype in DTYPES:
        for k, N in ((1, 5), (2, 9), (3, 64), (5, 1000), (7, 4096)):
            row = np.full(N, -math.inf)
            idx = np.linspace(0, N - 1, k).astype(int)
            row[idx] = 1.5
            got = run_rows(orc, [row], dtype)[0]
            want = np.zeros(N)
            want[idx] = brute.round_exact(Fraction(1, k), dtype)
            assert same(got, want), "tied maxima dtype %d k=%d" % (dtype, k)


def check_causal_rows(orc):
    w = synth.WORKLOADS["f16_causal_524288x2048"]
    rows = [0, 1, 2, 5, 1000, 2046, 2047, 2048, 2049, 4095 + 2048]
    x = w.generate_rows(rows)
    got = decode(orc.softmax_rows(x.reshape(-1), len(rows), w.N, w.ld_in, w.N, w.dtype), w.dtype)
    for k, r in enumerate(rows):
        q = r % 2048
        assert np.all(got[k, q + 1:] == 0.0), "causal row %d: nonzero past q" % r
        assert np.all(got[k, :q + 1] > 0.0), "causal row %d: zero before q" % r
    assert got[0, 0] == 1.0 and np.all(got[0, 1:] == 0.0)


def check_nan_rows(orc):
    for dtype in DTYPES:
        rows = [[-math.inf] * 6,
                [0.0, math.nan, 1.0, 2.0, -1.0, 0.5],
                [0.0, 1.0, math.inf, 2.0, -1.0, 0.5],
                [math.nan] * 6]
        got = run_rows(orc, rows, dtype)
        assert np.all(np.isnan(got)), "NaN rows dtype %d: %r" % (dtype, got)
        ok = run_rows(orc, [[0.0, 1.0, -math.inf, 2.0, -1.0, 0.5]], dtype)
        assert np.all(np.isfinite(ok))


# ---- invariants ------------------------------------------------------------------

SMALL = {
    "f32_1024x256": 64,
    "f32_4096x4096": 33,
    "bf16_16384x1000_ld1024": 48,
    "bf16_1024x131072": 3,
    "f16_causal_524288x2048": 40,
}


def _small_cases():
    for name, rows in SMALL.items():
        yield synth.WORKLOADS[name].with_rows(rows)


def check_row_sums_and_range(orc):
    for w in _small_cases():
        x = w.generate()
        y = decode(orc.softmax_rows(x.reshape(-1), w.M, w.N, w.ld_in, w.ld_out, w.dtype,
                                    nthreads=4), w.dtype)[:, :w.N]
        assert np.all(y >= 0.0) and np.all(y <= 1.0), w.name
        bound = UNIT_ROUNDOFF[w.dtype] + 2.0 ** -20
        err = np.abs(y.sum(axis=1) - 1.0)
        assert np.all(err <= bound), "%s: row sum off by %g" % (w.name, err.max())
        xv = synth.storage_to_float64(x[:, :w.N], w.dtype)
        am = np.argmax(xv, axis=1)
        assert np.all(y[np.arange(w.M), am] == y.max(axis=1)), "%s: argmax moved" % w.name


def check_shift_invariance(orc):
    rng = np.random.default_rng(5)
    for dtype in DTYPES:
        for N in (3, 17, 256, 1000):
            base = rng.integers(-32, 33, size=(4, N)) / 4.0  # multiples of 1/4 in [-8, 8]
            a = run_rows(orc, base, dtype)
            for c in (16.0, -16.0, 0.25):
                b = run_rows(orc, base + c, dtype)
                assert same(a, b), "shift dtype %d N=%d c=%g" % (dtype, N, c)


def check_strides(orc):
    w = synth.WORKLOADS["bf16_16384x1000_ld1024"].with_rows(20)
    x = w.generate()  # pitch 1024, columns 1000.. are NaN
    assert np.all(np.isnan(synth.storage_to_float64(x[:, w.N:], w.dtype)))
    dense = np.ascontiguousarray(x[:, :w.N])
    ref = orc.softmax_rows(dense.reshape(-1), w.M, w.N, w.N, w.N, w.dtype)
    sentinel = np.full((w.M, 1040), 0x7BCD, dtype=np.uint16)
    out = orc.softmax_rows(x.reshape(-1), w.M, w.N, w.ld_in, 1040, w.dtype, out=sentinel)
    assert same(out[:, :w.N], ref), "strided input changed the result"
    assert np.all(out[:, w.N:] == 0x7BCD), "output pad columns were written"
    assert np.all(np.isfinite(decode(out[:, :w.N], w.dtype)))


def check_thread_independence(orc):
    w = synth.WORKLOADS["f32_4096x4096"].with_rows(37)
    x = w.generate()
    a = orc.softmax_rows(x.reshape(-1), w.M, w.N, w.ld_in, w.ld_out, w.dtype, nthreads=1)
    b = orc.softmax_rows(x.reshape(-1), w.M, w.N, w.ld_in, w.ld_out, w.dtype, nthreads=5)
    assert same(a, b)


# ---- masked softmax (valid lengths, causal rows) ------------------------------

def check_masked_brute(orc):
    rng = np.random.default_rng(21)
    for dtype in DTYPES:
        for N in (1, 3, 8, 13):
            M = 6
            vals = to_grid(rng.normal(0, 3, size=(M, N)), dtype)
            lens = np.array([0, 1, N, N + 5, -2, max(1, N // 2)], dtype=np.int32)
            # Masked entries hold poison: they must never be read.
            poisoned = vals.copy()
            for i, L in enumerate(lens):
                poisoned[i, max(0, min(L, N)):] = math.nan
            x = encode_exact(poisoned, dtype)
            got = decode(orc.softmax_rows_masked(x.reshape(-1), M, N, N, N, dtype, lens=lens), dtype)
            for i, L in enumerate(lens):
                L = max(0, min(int(L), N))
                if L == 0:
                    assert np.all(np.isnan(got[i])), "masked row of length 0 must be NaN"
                    continue
                want = np.zeros(N)
                want[:L] = brute.softmax_exact_cast(vals[i, :L], dtype)
                assert same(got[i], want), "masked brute dtype %d N=%d L=%d: %r vs %r" % (
                    dtype, N, L, got[i], want)


def check_masked_causal(orc):
    for dtype in DTYPES:
        P, N, M = 5, 7, 12
        x = encode_exact(np.zeros((M, N)), dtype)  # constant rows: 1/L on the first L entries
        got = decode(orc.softmax_rows_masked(x.reshape(-1), M, N, N, N, dtype, causal_period=P),
                     dtype)
        for i in range(M):
            L = min(N, i % P + 1)
            want = np.zeros(N)
            want[:L] = brute.round_exact(Fraction(1, L), dtype)
            assert same(got[i], want), "causal dtype %d row %d" % (dtype, i)
        # The causal generator's rows: masking by period equals the data's own -inf mask.
        w = synth.WORKLOADS["f16_causal_524288x2048"]
        rows = w.generate_rows([0, 5, 2047, 2048, 4000])
        lens = np.array([r % 2048 + 1 for r in (0, 5, 2047, 2048, 4000)], dtype=np.int32)
        a = orc.softmax_rows_masked(rows.reshape(-1), 5, w.N, w.N, w.N, w.dtype, lens=lens)
        vals = decode(rows, w.dtype)
        for k in range(5):
            L = int(lens[k])
            assert np.all(decode(a[k, L:], w.dtype) == 0.0)
            assert same(decode(a[k, :L], w.dtype), brute.softmax_exact_cast(vals[k, :L], w.dtype)) \
                if L <= 16 else np.allclose(decode(a[k, :L], w.dtype).sum(), 1.0, atol=2e-3)


# ---- softmax backward -------------------------------------------------------------

def _bwd_decimal(y, dy):
    import decimal
    with decimal.localcontext(brute.CTX):
        Y = [decimal.Decimal(float(v)) for v in y]
        G = [decimal.Decimal(float(v)) for v in dy]
        dot = sum(a * b for a, b in zip(Y, G))
        return [a * (b - dot) for a, b in zip(Y, G)]


def check_backward_brute(orc):
    rng = np.random.default_rng(31)
    for dtype in DTYPES:
        for N in (1, 2, 5, 13):
            M = 4
            y = to_grid(rng.uniform(0, 1, size=(M, N)), dtype)
            dy = to_grid(rng.normal(0, 2, size=(M, N)), dtype)
            got = decode(orc.softmax_backward(encode_exact(y, dtype), encode_exact(dy, dtype),
                                              M, N, N, N, N, dtype), dtype)
            for i in range(M):
                want = [brute.round_exact(Fraction(v), dtype) for v in _bwd_decimal(y[i], dy[i])]
                assert same(got[i], want), "backward brute dtype %d N=%d" % (dtype, N)


def check_backward_is_softmax_vjp(orc):
    """dx equals the vector-Jacobian product of softmax, by central differences
    of the 60-digit softmax: dx_k = d/dt [softmax(x + t e_k) . dy] at t = 0."""
    import decimal
    rng = np.random.default_rng(32)
    for N in (2, 3, 6):
        x = rng.normal(0, 1.5, size=N)
        dy = rng.normal(0, 1, size=N)
        y = np.array([float(v) for v in brute.softmax_decimal(x)])
        got = orc.softmax_backward(y.astype(np.float32), dy.astype(np.float32), 1, N, N, N, N,
                                   F32).astype(np.float64)[0]
        with decimal.localcontext(brute.CTX):
            h = decimal.Decimal("1e-25")
            G = [decimal.Decimal(float(v)) for v in dy.astype(np.float32)]
            for k in range(N):
                def f(t):
                    xs = [decimal.Decimal(float(v)) for v in x]
                    xs[k] += t
                    m = max(xs)
                    e = [(v - m).exp() for v in xs]
                    s = sum(e)
                    return sum((a / s) * g for a, g in zip(e, G))
                fd = float((f(h) - f(-h)) / (2 * h))
                # y and dy were rounded to f32 before the oracle saw them.
                assert abs(got[k] - fd) <= 2e-6 * (1 + abs(fd)), "vjp N=%d k=%d: %g vs %g" % (
                    N, k, got[k], fd)


def check_backward_closed_forms(orc):
    for dtype in DTYPES:
        N = 9
        y = np.zeros((3, N))
        y[0, 4] = 1.0                       # one-hot y: dx = 0 whatever dy is
        y[1, :] = 0.0                       # zero y: dx = 0
        y[2, :3] = [0.25, 0.25, 0.5]        # dy = constant c: dx_j = c*y_j*(1 - sum y) = 0
        dy = np.array([np.linspace(-3, 3, N), np.linspace(1, 2, N), np.full(N, 1.5)])
        got = decode(orc.softmax_backward(encode_exact(to_grid(y, dtype), dtype),
                                          encode_exact(to_grid(dy, dtype), dtype),
                                          3, N, N, N, N, dtype), dtype)
        assert np.all(got == 0.0), "backward closed forms dtype %d: %r" % (dtype, got)
        # Row sums of dx vanish when y sums to one (exactly representable y).
        y2 = np.array([[0.5, 0.25, 0.125, 0.125]])
        dy2 = np.array([[1.0, -2.0, 0.5, 4.0]])
        d = decode(orc.softmax_backward(encode_exact(y2, dtype), encode_exact(dy2, dtype), 1, 4, 4, 4,
                                        4, dtype), dtype)
        assert abs(d.sum()) <= 4 * UNIT_ROUNDOFF[dtype] * np.abs(d).max()


# ---- residual RMSNorm -------------------------------------------------------------

def _rms_brute(x, r, w, eps, dtype):
    """60-digit RMSNorm of one row: h = dtype(exact x + r), y = dtype(h w / sqrt(mean h^2 + eps))."""
    import decimal
    h = [brute.round_exact(Fraction(float(a)) + Fraction(float(b)), dtype) for a, b in zip(x, r)]
    with decimal.localcontext(brute.CTX):
        H = [decimal.Decimal(v) for v in h]
        ms = sum(v * v for v in H) / len(H)
        rms = (ms + decimal.Decimal(float(eps))).sqrt()
        out = []
        for v, wj in zip(H, w):
            q = v * decimal.Decimal(float(wj)) / rms if rms != 0 else decimal.Decimal("NaN")
            out.append(math.nan if q.is_nan() else brute.round_exact(Fraction(q), dtype))
    return np.array(out)


def _rms(orc, x, r, w, eps, dtype):
    M, N = x.shape
    return decode(orc.rmsnorm_residual(encode_exact(x, dtype), encode_exact(r, dtype),
                                       encode_exact(w, dtype), M, N, N, N, N, eps, dtype), dtype)


def check_rmsnorm_brute(orc):
    rng = np.random.default_rng(41)
    for dtype in DTYPES:
        for N in (1, 3, 8, 17):
            M = 3
            # Magnitudes spread over several binades so that x + r often needs rounding.
            x = to_grid(rng.normal(0, 1, size=(M, N)) * 2.0 ** rng.integers(-6, 7, size=(M, N)),
                        dtype)
            r = to_grid(rng.normal(0, 1, size=(M, N)) * 2.0 ** rng.integers(-6, 7, size=(M, N)),
                        dtype)
            w = to_grid(rng.uniform(0.5, 1.5, size=N), dtype)
            for eps in (0.0, 1e-6, 0.25):
                got = _rms(orc, x, r, w, eps, dtype)
                for i in range(M):
                    want = _rms_brute(x[i], r[i], w, eps, dtype)
                    assert same(got[i], want), "rmsnorm brute dtype %d N=%d eps=%g" % (dtype, N, eps)


def check_rmsnorm_closed_forms(orc):
    for dtype in DTYPES:
        w = np.array([1.0, 2.0, 0.5, -1.0, 0.75, 1.5])
        N = w.size
        # A constant row of c (c = x + r exactly), eps = 0: h / rms = sign(c), so y = sign(c) w.
        x = np.array([[3.0] * N, [-0.375] * N, [96.0] * N])
        r = np.array([[1.0] * N, [-0.125] * N, [32.0] * N])
        y = _rms(orc, to_grid(x, dtype), to_grid(r, dtype), to_grid(w, dtype), 0.0, dtype)
        assert np.array_equal(y, np.sign(x + r) * w), "rmsnorm constant rows dtype %d" % dtype
        # Alternating +-c: mean square c^2 again.
        x2 = np.array([[2.0, -2.0] * (N // 2)])
        y2 = _rms(orc, to_grid(x2, dtype), np.zeros_like(x2), to_grid(w, dtype), 0.0, dtype)
        assert np.array_equal(y2[0], np.sign(x2[0]) * w)
        # N = 1: y = w h / sqrt(h^2 + eps); with h = 3, eps = 16: y = 3/5 w.
        y3 = _rms(orc, np.array([[1.0]]), np.array([[2.0]]), np.array([5.0]), 16.0, dtype)
        assert y3[0, 0] == brute.round_exact(Fraction(3), dtype)
        # Zero row: 0/0 with eps = 0, zeros with eps > 0.
        z = np.zeros((1, 4))
        assert np.isnan(_rms(orc, z, z, np.ones(4), 0.0, dtype)).all()
        assert (_rms(orc, z, z, np.ones(4), 1e-6, dtype) == 0.0).all()


def check_rmsnorm_invariants(orc):
    rng = np.random.default_rng(42)
    for dtype in DTYPES:
        M, N = 4, 64
        x = to_grid(rng.normal(0, 1, size=(M, N)), dtype)
        r = to_grid(rng.normal(0, 1, size=(M, N)), dtype)
        w1 = np.ones(N)
        y = _rms(orc, x, r, w1, 0.0, dtype)
        # Unit weight, eps = 0: each output row has mean square one (up to the casts).
        ms = (y * y).mean(axis=1)
        assert np.all(np.abs(ms - 1.0) <= 4 * UNIT_ROUNDOFF[dtype]), (dtype, ms)
        # Scaling x and r by a power of two leaves y unchanged (eps = 0).
        y4 = _rms(orc, x * 4.0, r * 4.0, w1, 0.0, dtype)
        assert np.array_equal(y, y4)
        # Doubling the weight doubles y exactly; a zero residual gives RMSNorm of x.
        w = to_grid(rng.uniform(0.5, 1.5, size=N), dtype)
        assert np.array_equal(_rms(orc, x, r, 2 * w, 1e-5, dtype),
                              2 * _rms(orc, x, r, w, 1e-5, dtype))
        assert np.array_equal(_rms(orc, x, np.zeros_like(x), w, 1e-5, dtype),
                              _rms(orc, np.zeros_like(x), x, w, 1e-5, dtype))


ALL_CHECKS = [
    check_decode, check_cast, check_brute_random, check_brute_extremes, check_uniform_rows,
    check_two_entries, check_tied_maxima, check_causal_rows, check_nan_rows,
    check_row_sums_and_range, check_shift_invariance, check_strides, check_thread_independence,
    check_masked_brute, check_masked_causal,
    check_backward_brute, check_backward_is_softmax_vjp, check_backward_closed_forms,
    check_rmsnorm_brute, check_rmsnorm_closed_forms, check_rmsnorm_invariants,
]
