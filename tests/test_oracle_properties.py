"""Randomised checks of the oracle against brute force (no GPU).

Hypothesis draws small rows of values on each dtype's grid, mixed with -inf,
+inf, NaN and large logits. It compares the oracle's cast result with the exact
softmax computed by tests/brute.py (Python decimal, rounded by exact rational
arithmetic). These add breadth to the fixed cases in tests/pins.py.
"""
import math

import numpy as np
import pytest

import oracle
import synth
from tests import brute, pins

hypothesis = pytest.importorskip("hypothesis")
st = hypothesis.strategies

SPECIAL = [-math.inf, math.inf, math.nan, 100.0, -100.0, 0.0, 88.5, -103.25]


@st.composite
def rows(draw):
    dtype = draw(st.sampled_from([synth.F32, synth.BF16, synth.F16]))
    M = draw(st.integers(1, 3))
    N = draw(st.integers(1, 12))
    finite = st.floats(-60.0, 60.0, allow_nan=False, allow_infinity=False)
    value = st.one_of(finite, finite, finite, st.sampled_from(SPECIAL))
    vals = draw(st.lists(st.lists(value, min_size=N, max_size=N), min_size=M, max_size=M))
    return dtype, pins.to_grid(np.array(vals, dtype=np.float64), dtype)


@hypothesis.settings(max_examples=150, deadline=None, derandomize=True)
@hypothesis.given(rows())
def test_oracle_matches_exact_softmax(case):
    dtype, vals = case
    M, N = vals.shape
    x = pins.encode_exact(vals, dtype)
    got = synth.storage_to_float64(
        oracle.load().softmax_rows(np.ascontiguousarray(x).reshape(-1), M, N, N, N, dtype), dtype)
    for i in range(M):
        want = brute.softmax_exact_cast(vals[i], dtype)
        assert pins.same(got[i], want), (dtype, vals[i], got[i], want)
        fin = np.isfinite(got[i])
        # The definition's invariants, where the row is finite.
        if fin.all():
            assert (got[i] >= 0).all() and (got[i] <= 1).all()
            u = {synth.F32: 2.0 ** -24, synth.BF16: 2.0 ** -9, synth.F16: 2.0 ** -11}[dtype]
            assert abs(got[i].sum() - 1.0) <= N * u + 2.0 ** -20


@st.composite
def pair_rows(draw):
    dtype = draw(st.sampled_from([synth.F32, synth.BF16, synth.F16]))
    M = draw(st.integers(1, 3))
    N = draw(st.integers(1, 12))
    a = draw(st.lists(st.lists(st.floats(0.0, 1.0), min_size=N, max_size=N), min_size=M,
                      max_size=M))
    b = draw(st.lists(st.lists(st.floats(-8.0, 8.0), min_size=N, max_size=N), min_size=M,
                      max_size=M))
    return dtype, pins.to_grid(np.array(a), dtype), pins.to_grid(np.array(b), dtype)


@hypothesis.settings(max_examples=80, deadline=None, derandomize=True)
@hypothesis.given(pair_rows())
def test_backward_oracle_within_its_fp64_bound(case):
    """The oracle forms dx_j = y_j (dy_j - d) in FP64 before its one cast, so where
    dy_j and d cancel its FP64 value can differ from the exact one by up to
    e_j = |y_j| (|dy_j| + sum_k |y_k dy_k|) (N + 2) 2^-53 (found by this test: y =
    [1, 0.5], dy = [1, 2^-52] gives exactly -2^-53 but 0 in FP64). The cast result
    must lie between the casts of exact - e_j and exact + e_j; away from such
    cancellation the two coincide and the result is the exactly rounded one."""
    from fractions import Fraction
    dtype, y, dy = case
    M, N = y.shape
    got = pins.decode(oracle.load().softmax_backward(pins.encode_exact(y, dtype),
                                                     pins.encode_exact(dy, dtype),
                                                     M, N, N, N, N, dtype), dtype)
    for i in range(M):
        exact = [Fraction(v) for v in pins._bwd_decimal(y[i], dy[i])]
        S = sum(abs(Fraction(a) * Fraction(b)) for a, b in zip(y[i], dy[i]))
        for j in range(N):
            e = abs(Fraction(y[i][j])) * (abs(Fraction(dy[i][j])) + S) * (N + 2) / 2 ** 53
            lo = brute.round_exact(exact[j] - e, dtype)
            hi = brute.round_exact(exact[j] + e, dtype)
            assert lo <= got[i][j] <= hi, (dtype, y[i], dy[i], j, got[i][j], lo, hi)


@hypothesis.settings(max_examples=80, deadline=None, derandomize=True)
@hypothesis.given(pair_rows(), st.sampled_from([0.0, 1e-6, 0.25]))
def test_rmsnorm_oracle_matches_exact(case, eps):
    dtype, x, r = case
    M, N = x.shape
    w = pins.to_grid(np.linspace(0.5, 1.5, N), dtype)
    got = pins._rms(oracle.load(), x, r, w, eps, dtype)
    for i in range(M):
        assert pins.same(got[i], pins._rms_brute(x[i], r[i], w, eps, dtype)), (dtype, x[i], r[i])


@hypothesis.settings(max_examples=100, deadline=None, derandomize=True)
@hypothesis.given(rows(), st.data())
def test_masked_oracle_matches_exact_prefix(case, data):
    """Masked rows equal the exact softmax of the row with its masked entries set to
    -inf, whatever the masked entries hold: exact zeros past L, and NaN everywhere
    when no valid entry is finite (L = 0, or a valid prefix of -inf only; found by
    this test: [-inf | 0] with L = 1 is [NaN, NaN])."""
    dtype, vals = case
    M, N = vals.shape
    lens = np.array(data.draw(st.lists(st.integers(-2, N + 3), min_size=M, max_size=M)),
                    dtype=np.int32)
    poisoned = vals.copy()
    for i, L in enumerate(lens):
        poisoned[i, max(0, min(int(L), N)):] = math.nan  # never read
    x = pins.encode_exact(poisoned, dtype)
    got = pins.decode(oracle.load().softmax_rows_masked(x.reshape(-1), M, N, N, N, dtype,
                                                        lens=lens), dtype)
    for i, L in enumerate(lens):
        L = max(0, min(int(L), N))
        filled = vals[i].copy()
        filled[L:] = -math.inf
        want = brute.softmax_exact_cast(filled, dtype)
        assert pins.same(got[i], want), (dtype, vals[i], L, got[i], want)
