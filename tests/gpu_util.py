"""Helpers for the GPU parity tests: device copies, the parity gate, diagnostics."""
from __future__ import annotations

import numpy as np

import oracle
import synth

# Parity gate |gpu - oracle| <= atol + rtol*|oracle|, elementwise; NaN where
# the oracle is NaN. FP32 at 1e-6; bf16/f16 at 0.004 (the Warpline README's
# K2 softmax tolerance, Protocol and correctness).
TOL = {synth.F32: (1e-6, 1e-6), synth.BF16: (4e-3, 4e-3), synth.F16: (4e-3, 4e-3)}

_TORCH_DTYPE = None


def torch_dtype(dtype):
    import torch
    return {synth.F32: torch.float32, synth.BF16: torch.bfloat16, synth.F16: torch.float16}[dtype]


def to_device(a: np.ndarray, dtype: int, device="cuda"):
    """Host storage array (float32 or uint16 bits) -> CUDA tensor of the dtype."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype != synth.F32:
        t = t.view(torch.int16).view(torch_dtype(dtype))
    return t.to(device)


def to_host(t, dtype: int) -> np.ndarray:
    import torch
    c = t.detach().cpu().contiguous()
    if dtype == synth.F32:
        return c.numpy()
    return c.view(torch.int16).numpy().view(np.uint16)


def gate(gpu: np.ndarray, ref: np.ndarray, dtype: int):
    """Return (ok, n_bad, max_abs_err, report dict) for decoded float64 arrays."""
    atol, rtol = TOL[dtype]
    nan_r, nan_g = np.isnan(ref), np.isnan(gpu)
    fin = ~nan_r
    err = np.abs(gpu - ref)
    bad = (nan_r != nan_g) | (fin & ~(err <= atol + rtol * np.abs(ref)))
    rep = {"max_abs": float(np.nanmax(np.where(fin, err, 0.0))) if err.size else 0.0}
    return (not bad.any()), int(bad.sum()), rep


def ulp_distance(gpu_bits: np.ndarray, ref_bits: np.ndarray, dtype: int) -> np.ndarray:
    """|bit distance| between non-negative finite values of the same dtype."""
    if dtype == synth.F32:
        g = gpu_bits.view(np.int32).astype(np.int64)
        r = ref_bits.view(np.int32).astype(np.int64)
    else:
        g = gpu_bits.astype(np.int64)
        r = ref_bits.astype(np.int64)
    return np.abs(g - r)


def check_rows(gpu_rows: np.ndarray, x_rows: np.ndarray, N: int, ld_in: int, dtype: int,
               label: str, max_ulp_16bit: int = 1):
    """Gate GPU output rows (storage, >= N columns) against the oracle on x_rows."""
    M = x_rows.shape[0]
    ref = oracle.softmax_rows(np.ascontiguousarray(x_rows).reshape(-1), M, N, ld_in, N, dtype,
                              nthreads=synth.host_threads())
    g = synth.storage_to_float64(gpu_rows[:, :N], dtype)
    r = synth.storage_to_float64(ref, dtype)
    ok, nbad, rep = gate(g, r, dtype)
    assert ok, "%s: %d of %d elements outside the gate (max abs %.3g)" % (
        label, nbad, g.size, rep["max_abs"])
    if dtype != synth.F32 and max_ulp_16bit is not None:
        # Stricter diagnostic: FP32 compute is far more accurate than one
        # bf16/f16 step, so results are the correctly rounded value or its
        # neighbour. bf16 results in the subnormal range may flush to zero.
        fin = np.isfinite(r) & (r >= (2.0 ** -126 if dtype == synth.BF16 else 0.0))
        d = ulp_distance(np.ascontiguousarray(gpu_rows[:, :N]), ref, dtype)[fin]
        assert d.size == 0 or d.max() <= max_ulp_16bit, "%s: %d ulp off" % (label, int(d.max()))
    return ref
