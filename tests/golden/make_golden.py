#!/usr/bin/env python3
"""Write tests/golden/oracle_fixtures.json: small inputs and the oracle's outputs, as
exact bit patterns (hex), for the softmax, the masked softmax, the softmax backward and
the residual RMSNorm in f32, bf16 and f16.

The source pages print no worked example with values, so these fixtures come from the
oracle alone (this script calls nothing but oracle/ and synth/). The oracle itself is
pinned by the brute-force, closed-form and invariant checks of tests/pins.py; the
fixtures freeze its bits, so that a rebuild on another machine or compiler (the oracle
is built on x86-64 and on aarch64) is checked against the same numbers.

    python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import synth  # noqa: E402

DTYPES = (synth.F32, synth.BF16, synth.F16)


def hexs(a):
    a = np.ascontiguousarray(a)
    return a.view(np.uint32 if a.dtype == np.float32 else np.uint16).reshape(-1).tolist()


def case_inputs(dtype, M, N, seed, **kw):
    return synth.generate(M, N, dtype=dtype, seed=seed, **kw)


def main():
    orc = oracle.load()
    cases = []
    for dtype in DTYPES:
        for N, M, p1 in ((1, 2, 1.0), (7, 3, 2.0), (33, 2, 4.0), (129, 2, 1.0)):
            x = case_inputs(dtype, M, N, 100 + N, p1=p1)
            y = orc.softmax_rows(x.reshape(-1), M, N, N, N, dtype)
            cases.append({"op": "softmax", "dtype": dtype, "M": M, "N": N,
                          "x": hexs(x), "y": hexs(y)})
        N, M = 40, 4
        x = case_inputs(dtype, M, N, 200, p1=3.0)
        lens = [0, 1, 17, 40]
        y = orc.softmax_rows_masked(x.reshape(-1), M, N, N, N, dtype, lens=np.array(lens))
        cases.append({"op": "softmax_masked", "dtype": dtype, "M": M, "N": N, "lens": lens,
                      "x": hexs(x), "y": hexs(y)})
        N, M = 24, 3
        yv = case_inputs(dtype, M, N, 300, dist=synth.DIST_UNIFORM, p0=0.0, p1=2.0 / N)
        dy = case_inputs(dtype, M, N, 301)
        dx = orc.softmax_backward(yv.reshape(-1), dy.reshape(-1), M, N, N, N, N, dtype)
        cases.append({"op": "softmax_backward", "dtype": dtype, "M": M, "N": N,
                      "y": hexs(yv), "dy": hexs(dy), "dx": hexs(dx)})
        xr = case_inputs(dtype, M, N, 400, p1=2.0)
        rr = case_inputs(dtype, M, N, 401, p1=0.5)
        wr = case_inputs(dtype, 1, N, 402, dist=synth.DIST_UNIFORM, p0=0.5, p1=1.5).reshape(-1)
        eps = float(np.float32(1e-6))
        yr = orc.rmsnorm_residual(xr.reshape(-1), rr.reshape(-1), wr, M, N, N, N, N, eps, dtype)
        cases.append({"op": "rmsnorm_residual", "dtype": dtype, "M": M, "N": N, "eps": eps,
                      "x": hexs(xr), "r": hexs(rr), "w": hexs(wr), "y": hexs(yr)})
    out = {"about": "Oracle regression fixtures written by tests/golden/make_golden.py "
                    "(oracle only); bit patterns of f32 (uint32) or bf16/f16 (uint16).",
           "cases": cases}
    with open(os.path.join(HERE, "oracle_fixtures.json"), "w") as f:
        json.dump(out, f, separators=(",", ":"))
        f.write("\n")


if __name__ == "__main__":
    main()
