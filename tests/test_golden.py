"""The oracle reproduces the bits frozen in tests/golden/oracle_fixtures.json.

The fixtures were written by tests/golden/make_golden.py from the oracle itself (the
source pages print no worked example with values); the oracle is pinned independently
by tests/pins.py. This test catches a change of the oracle's results across machines,
compilers or edits: any difference, in any bit, fails (NaNs match NaNs of either sign).
"""
import json
import os

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
FIXTURES = json.load(open(os.path.join(HERE, "golden", "oracle_fixtures.json")))["cases"]


def arr(bits, dtype):
    if dtype == 0:
        return np.array(bits, dtype=np.uint32).view(np.float32)
    return np.array(bits, dtype=np.uint16)


def bits(a):
    a = np.ascontiguousarray(a)
    return a.view(np.uint32 if a.dtype == np.float32 else np.uint16).reshape(-1).tolist()


def is_nan(b, dtype):
    """NaN bit patterns (of any sign and payload) of f32, bf16 or f16."""
    b = np.array(b, dtype=np.uint64)
    if dtype == 0:
        return ((b & 0x7F800000) == 0x7F800000) & ((b & 0x007FFFFF) != 0)
    if dtype == 1:
        return ((b & 0x7F80) == 0x7F80) & ((b & 0x007F) != 0)
    return ((b & 0x7C00) == 0x7C00) & ((b & 0x03FF) != 0)


def same(got_bits, want_bits, dtype):
    """Equal bits, except that a NaN matches any NaN: IEEE 754 leaves the sign of a
    generated NaN open (x86-64 produces 0/0 with the sign bit set, aarch64 without)."""
    g, w = np.array(got_bits, dtype=np.uint64), np.array(want_bits, dtype=np.uint64)
    gn, wn = is_nan(g, dtype), is_nan(w, dtype)
    return bool(np.array_equal(gn, wn) and np.array_equal(g[~gn], w[~wn]))


@pytest.mark.parametrize("k", range(len(FIXTURES)),
                         ids=["%s-%d-%d" % (c["op"], c["dtype"], c["N"]) for c in FIXTURES])
def test_oracle_matches_fixture(k):
    c = FIXTURES[k]
    orc = oracle.load()
    d, M, N = c["dtype"], c["M"], c["N"]
    if c["op"] == "softmax":
        got = orc.softmax_rows(arr(c["x"], d), M, N, N, N, d)
        want = c["y"]
    elif c["op"] == "softmax_masked":
        got = orc.softmax_rows_masked(arr(c["x"], d), M, N, N, N, d, lens=np.array(c["lens"]))
        want = c["y"]
    elif c["op"] == "softmax_backward":
        got = orc.softmax_backward(arr(c["y"], d), arr(c["dy"], d), M, N, N, N, N, d)
        want = c["dx"]
    else:
        got = orc.rmsnorm_residual(arr(c["x"], d), arr(c["r"], d), arr(c["w"], d), M, N, N, N, N,
                                   c["eps"], d)
        want = c["y"]
    assert same(bits(got), want, d)
