"""The oracle reproduces the bits frozen in tests/golden/oracle_fixtures.json.

The fixtures were written by tests/golden/make_golden.py from the oracle itself (the
source pages print no worked example with values); the oracle is pinned independently
by tests/pins.py. This test catches a change of the oracle's results across machines,
compilers or edits: any difference, in any bit, fails.
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
    assert bits(got) == want
