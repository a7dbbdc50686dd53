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
