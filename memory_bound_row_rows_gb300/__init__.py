"""Python binding of the softmax_rows C ABI (include/softmax_rows.h).

Argument marshalling only: every step of the softmax runs in the CUDA kernels
of ``lib/libsoftmax_rows.so``. The functions keep the C names and arguments;
pointers may be given as integers or as tensors (their ``data_ptr()``), and a
stream as a ``torch.cuda.Stream``, a raw handle, or None for torch's current
stream. There is no CPU fallback: if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "SR_F32", "SR_BF16", "SR_F16", "SR_OK", "SR_EINVAL", "SR_EDTYPE", "SR_ECUDA",
    "SR_EDEVICE_TIMEOUT", "SR_EPLAN", "SR_EBOUNDS", "SR_BUILD_BOUNDS_CHECK", "SR_PLAN_AUTO", "SR_PLAN_WARP", "SR_PLAN_CTA",
    "SR_PLAN_CLUSTER", "SR_PLAN_ONLINE", "SR_PLAN_SMEM", "SR_PLAN_ROW", "SR_PLAN_WIDE",
    "PLAN_NAMES", "SoftmaxRowsError", "load", "lib_path", "open_library",
    "softmax_rows", "softmax_rows_ex", "softmax_rows_plan", "softmax_rows_plan_check",
    "softmax_rows_last_device_error", "softmax_rows_test_expiry", "softmax_rows_strerror",
    "softmax_rows_version", "softmax_rows_host", "softmax_rows_host_workspace_bytes",
    "softmax_rows_split", "softmax_rows_split_workspace_bytes", "softmax_rows_split_noalloc",
    "softmax_rows_split_shape", "softmax_rows_split_test_expiry",
    "softmax_rows_host_mapped",
    "softmax_rows_masked", "softmax_rows_backward", "softmax_rows_backward_ex",
    "softmax_rows_backward_plan", "softmax_rows_backward_test_expiry", "rmsnorm_residual_rows", "rmsnorm_residual_rows_ex",
    "rmsnorm_residual_rows_plan", "softmax_rows_wide_shape", "softmax_rows_last_launch", "softmax_rows_copy_ceiling", "softmax_rows_copy_ceiling2",
    "softmax", "softmax_backward", "rmsnorm_residual",
    "dtype_code",
]

SR_F32, SR_BF16, SR_F16 = 0, 1, 2
SR_OK, SR_EINVAL, SR_EDTYPE, SR_ECUDA, SR_EDEVICE_TIMEOUT, SR_EPLAN = 0, 1, 2, 3, 4, 5
SR_EBOUNDS = 6
SR_BUILD_BOUNDS_CHECK = 1
SR_PLAN_AUTO, SR_PLAN_WARP, SR_PLAN_CTA, SR_PLAN_CLUSTER, SR_PLAN_ONLINE = 0, 1, 2, 3, 4
SR_PLAN_SMEM, SR_PLAN_ROW, SR_PLAN_WIDE = 5, 6, 7
PLAN_NAMES = {SR_PLAN_AUTO: "auto", SR_PLAN_WARP: "warp", SR_PLAN_CTA: "cta",
              SR_PLAN_CLUSTER: "cluster", SR_PLAN_ONLINE: "online", SR_PLAN_SMEM: "smem",
              SR_PLAN_ROW: "row", SR_PLAN_WIDE: "wide"}

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "lib", "libsoftmax_rows.so")
_lib = None


class SoftmaxRowsError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s: %s (status %d)" % (where, softmax_rows_strerror(status), status))


def lib_path() -> str:
    return os.environ.get("SOFTMAX_ROWS_LIB", _LIB_PATH)


def load():
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    if _lib is None:
        _lib = open_library(lib_path())
    return _lib


def open_library(path: str):
    """A ctypes handle on a build of the library at ``path`` with every entry
    point's signature declared (the product build, or the bounds-checking one)."""
    if not os.path.exists(path):
        raise RuntimeError(
            "softmax_rows CUDA library not found at %s; build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'`" % path)
    lib = ctypes.CDLL(path)
    vp, i64, c_int, u64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint64
    f32 = ctypes.c_float
    sig = {
        "softmax_rows": [vp, vp, i64, i64, i64, i64, c_int, vp],
        "softmax_rows_ex": [vp, vp, i64, i64, i64, i64, c_int, c_int, vp],
        "softmax_rows_plan": [vp, vp, i64, i64, i64, i64, c_int],
        "softmax_rows_plan_check": [vp, vp, i64, i64, i64, i64, c_int, c_int],
        "softmax_rows_last_device_error": [vp],
        "softmax_rows_test_expiry": [vp, vp, i64, i64, i64, i64, c_int, c_int, u64, vp],
        "softmax_rows_strerror": [c_int],
        "softmax_rows_host": [vp, vp, i64, i64, i64, i64, c_int, vp, i64, vp],
        "softmax_rows_host_workspace_bytes": [i64, i64, c_int],
        "softmax_rows_host_mapped": [vp, vp, i64, i64, i64, i64, c_int, vp],
        "softmax_rows_split": [vp, vp, i64, i64, i64, i64, c_int, vp, i64, vp],
        "softmax_rows_split_workspace_bytes": [vp, vp, i64, i64, i64, i64, c_int],
        "softmax_rows_split_noalloc": [vp, vp, i64, i64, i64, i64, c_int, vp],
        "softmax_rows_split_shape": [vp, vp, i64, i64, i64, i64, c_int, c_int, i64, vp],
        "softmax_rows_split_test_expiry": [vp, vp, i64, i64, i64, i64, c_int, vp, i64, u64, vp],
        "softmax_rows_masked": [vp, vp, i64, i64, i64, i64, c_int, vp, i64, c_int, vp],
        "softmax_rows_backward": [vp, vp, vp, i64, i64, i64, i64, i64, c_int, vp],
        "softmax_rows_backward_ex": [vp, vp, vp, i64, i64, i64, i64, i64, c_int, c_int, vp],
        "softmax_rows_backward_plan": [vp, vp, vp, i64, i64, i64, i64, i64, c_int, c_int, c_int],
        "softmax_rows_backward_test_expiry": [vp, vp, vp, i64, i64, i64, i64, i64, c_int, u64, vp],
        "rmsnorm_residual_rows": [vp, vp, vp, vp, i64, i64, i64, i64, i64, f32, c_int, vp],
        "rmsnorm_residual_rows_ex": [vp, vp, vp, vp, i64, i64, i64, i64, i64, f32, c_int, c_int,
                                     vp],
        "rmsnorm_residual_rows_plan": [vp, vp, vp, vp, i64, i64, i64, i64, i64, f32, c_int, c_int,
                                       c_int],
        "softmax_rows_version": [],
        "softmax_rows_wide_shape": [i64, i64, c_int, c_int, vp, vp, vp, vp],
        "softmax_rows_last_launch": [vp],
        "softmax_rows_build_flags": [],
        "softmax_rows_copy_ceiling": [vp, vp, i64, i64, i64, i64, vp],
        "softmax_rows_copy_ceiling2": [vp, vp, vp, i64, i64, i64, i64, i64, vp],
        "softmax_rows_bounds_address": [],
        "softmax_rows_test_bounds_shrink": [i64],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = {"softmax_rows_strerror": ctypes.c_char_p,
                      "softmax_rows_host_workspace_bytes": i64,
                      "softmax_rows_split_workspace_bytes": i64,
                      "softmax_rows_bounds_address": u64}.get(name, c_int)
    return lib


def _ptr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return int(x.data_ptr())
    raise TypeError("expected a pointer (int) or a tensor, got %r" % type(x))


def _stream(s) -> int:
    if s is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream) if torch.cuda.is_available() else 0
    if isinstance(s, int):
        return s
    if hasattr(s, "cuda_stream"):
        return int(s.cuda_stream)
    raise TypeError("expected a CUDA stream, a handle or None, got %r" % type(s))


def _check(status: int, where: str) -> int:
    if status != SR_OK:
        raise SoftmaxRowsError(status, where)
    return status


def softmax_rows(in_, out, M, N, ld_in, ld_out, dtype, stream=None) -> int:
    return _check(load().softmax_rows(_ptr(in_), _ptr(out), M, N, ld_in, ld_out, dtype,
                                      _stream(stream)), "softmax_rows")


def softmax_rows_ex(in_, out, M, N, ld_in, ld_out, dtype, plan, stream=None) -> int:
    return _check(load().softmax_rows_ex(_ptr(in_), _ptr(out), M, N, ld_in, ld_out, dtype, plan,
                                         _stream(stream)), "softmax_rows_ex")


def softmax_rows_plan(in_, out, M, N, ld_in, ld_out, dtype) -> int:
    """The plan softmax_rows would run (> 0), or a negative status."""
    return int(load().softmax_rows_plan(_ptr(in_), _ptr(out), M, N, ld_in, ld_out, dtype))


def softmax_rows_wide_shape(M, N, dtype, sm_count) -> dict:
    """How the WIDE plan runs M rows of N elements on `sm_count` SMs (host logic):
    {"csize", "kv", "slice", "streamed"}; raises on bad arguments."""
    csize, kv, streamed = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    slice_ = ctypes.c_int64()
    st = load().softmax_rows_wide_shape(M, N, dtype, sm_count, ctypes.byref(csize),
                                        ctypes.byref(kv), ctypes.byref(slice_),
                                        ctypes.byref(streamed))
    if st != 0:
        raise SoftmaxRowsError(-st, "softmax_rows_wide_shape")
    return {"csize": csize.value, "kv": kv.value, "slice": slice_.value,
            "streamed": bool(streamed.value)}


def softmax_rows_plan_check(in_, out, M, N, ld_in, ld_out, dtype, plan) -> int:
    return int(load().softmax_rows_plan_check(_ptr(in_), _ptr(out), M, N, ld_in, ld_out, dtype,
                                              plan))


def softmax_rows_last_device_error(stream=None) -> int:
    """Status of the device error word (SR_OK or SR_EDEVICE_TIMEOUT); clears it."""
    return int(load().softmax_rows_last_device_error(_stream(stream)))


def softmax_rows_test_expiry(in_, out, M, N, ld_in, ld_out, dtype, plan, timeout_ns,
                             stream=None) -> int:
    return _check(load().softmax_rows_test_expiry(_ptr(in_), _ptr(out), M, N, ld_in, ld_out,
                                                  dtype, plan, timeout_ns, _stream(stream)),
                  "softmax_rows_test_expiry")


def softmax_rows_host(h_in, h_out, M, N, ld_in, ld_out, dtype, d_work, work_bytes,
                      stream=None) -> int:
    """Host-memory variant: h_in/h_out are host pointers (page-locked for overlap)."""
    return _check(load().softmax_rows_host(_ptr(h_in), _ptr(h_out), M, N, ld_in, ld_out, dtype,
                                           _ptr(d_work), work_bytes, _stream(stream)),
                  "softmax_rows_host")


def softmax_rows_host_mapped(h_in, h_out, M, N, ld_in, ld_out, dtype, stream=None) -> int:
    """Zero-copy variant: the kernel reads and writes mapped page-locked host memory."""
    return _check(load().softmax_rows_host_mapped(_ptr(h_in), _ptr(h_out), M, N, ld_in, ld_out,
                                                  dtype, _stream(stream)),
                  "softmax_rows_host_mapped")


def softmax_rows_masked(in_, out, M, N, ld_in, ld_out, dtype, lengths=None, causal_period=0,
                        plan=SR_PLAN_AUTO, stream=None) -> int:
    """Masked softmax; `lengths` is a device int32 array of M valid lengths (or None)."""
    return _check(load().softmax_rows_masked(_ptr(in_), _ptr(out), M, N, ld_in, ld_out, dtype,
                                             _ptr(lengths), causal_period, plan, _stream(stream)),
                  "softmax_rows_masked")


def softmax_rows_backward(y, dy, dx, M, N, ld_y, ld_dy, ld_dx, dtype, stream=None) -> int:
    """dx = y * (dy - sum(y * dy)) per row; y, dy, dx are device matrices."""
    return _check(load().softmax_rows_backward(_ptr(y), _ptr(dy), _ptr(dx), M, N, ld_y, ld_dy,
                                               ld_dx, dtype, _stream(stream)),
                  "softmax_rows_backward")


def softmax_rows_backward_ex(y, dy, dx, M, N, ld_y, ld_dy, ld_dx, dtype, plan,
                             stream=None) -> int:
    return _check(load().softmax_rows_backward_ex(_ptr(y), _ptr(dy), _ptr(dx), M, N, ld_y, ld_dy,
                                                  ld_dx, dtype, plan, _stream(stream)),
                  "softmax_rows_backward_ex")


def softmax_rows_backward_test_expiry(y, dy, dx, M, N, ld_y, ld_dy, ld_dx, dtype, timeout_ns,
                                      stream=None) -> int:
    """Test hook: the CLUSTER plan with its partials not sent (every wait expires)."""
    return _check(load().softmax_rows_backward_test_expiry(_ptr(y), _ptr(dy), _ptr(dx), M, N,
                                                           ld_y, ld_dy, ld_dx, dtype, timeout_ns,
                                                           _stream(stream)),
                  "softmax_rows_backward_test_expiry")


def softmax_rows_backward_plan(y, dy, dx, M, N, ld_y, ld_dy, ld_dx, dtype, plan=SR_PLAN_AUTO,
                               sm_count=0) -> int:
    """The plan the backward would run (> 0), or a negative status (host logic)."""
    return int(load().softmax_rows_backward_plan(_ptr(y), _ptr(dy), _ptr(dx), M, N, ld_y, ld_dy,
                                                 ld_dx, dtype, plan, sm_count))


def rmsnorm_residual_rows(x, residual, weight, y, M, N, ld_x, ld_r, ld_y, eps, dtype,
                          stream=None) -> int:
    """y = dtype(h * w / sqrt(mean(h^2) + eps)), h = dtype(x + residual); device pointers."""
    return _check(load().rmsnorm_residual_rows(_ptr(x), _ptr(residual), _ptr(weight), _ptr(y), M,
                                               N, ld_x, ld_r, ld_y, eps, dtype, _stream(stream)),
                  "rmsnorm_residual_rows")


def rmsnorm_residual_rows_ex(x, residual, weight, y, M, N, ld_x, ld_r, ld_y, eps, dtype, plan,
                             stream=None) -> int:
    return _check(load().rmsnorm_residual_rows_ex(_ptr(x), _ptr(residual), _ptr(weight), _ptr(y),
                                                  M, N, ld_x, ld_r, ld_y, eps, dtype, plan,
                                                  _stream(stream)),
                  "rmsnorm_residual_rows_ex")


def rmsnorm_residual_rows_plan(x, residual, weight, y, M, N, ld_x, ld_r, ld_y, eps, dtype,
                               plan=SR_PLAN_AUTO, sm_count=0) -> int:
    return int(load().rmsnorm_residual_rows_plan(_ptr(x), _ptr(residual), _ptr(weight), _ptr(y),
                                                 M, N, ld_x, ld_r, ld_y, eps, dtype, plan,
                                                 sm_count))


class _SplitShape(ctypes.Structure):
    _fields_ = [("lanes", ctypes.c_int), ("parts", ctypes.c_int),
                ("part_units", ctypes.c_int64), ("unit_elems", ctypes.c_int)]


def softmax_rows_split_shape(in_, out, M, N, ld_in, ld_out, dtype, max_blocks=0,
                             l2_bytes=0) -> dict:
    """How the split plan cuts a problem (host logic when max_blocks and l2_bytes
    are given): {"lanes", "parts", "part_units", "unit_elems"}; raises on bad
    arguments."""
    sh = _SplitShape()
    _check(load().softmax_rows_split_shape(_ptr(in_), _ptr(out), M, N, ld_in, ld_out, dtype,
                                           max_blocks, l2_bytes, ctypes.byref(sh)),
           "softmax_rows_split_shape")
    return {"lanes": sh.lanes, "parts": sh.parts, "part_units": sh.part_units,
            "unit_elems": sh.unit_elems}


def softmax_rows_split_test_expiry(in_, out, M, N, ld_in, ld_out, dtype, workspace,
                                   workspace_bytes, timeout_ns, stream=None) -> int:
    return int(load().softmax_rows_split_test_expiry(_ptr(in_), _ptr(out), M, N, ld_in, ld_out,
                                                     dtype, _ptr(workspace), workspace_bytes,
                                                     timeout_ns, _stream(stream)))


def softmax_rows_split(in_, out, M, N, ld_in, ld_out, dtype, workspace, workspace_bytes,
                       stream=None) -> int:
    """Split plan for wide rows (one cooperative kernel); `workspace` is a device buffer."""
    return _check(load().softmax_rows_split(_ptr(in_), _ptr(out), M, N, ld_in, ld_out, dtype,
                                            _ptr(workspace), workspace_bytes, _stream(stream)),
                  "softmax_rows_split")


def softmax_rows_split_noalloc(in_, out, M, N, ld_in, ld_out, dtype, stream=None) -> int:
    """Split plan with the library's built-in scratch: allocates nothing (see the C header)."""
    return _check(load().softmax_rows_split_noalloc(_ptr(in_), _ptr(out), M, N, ld_in, ld_out,
                                                    dtype, _stream(stream)),
                  "softmax_rows_split_noalloc")


def softmax_rows_split_workspace_bytes(in_, out, M, N, ld_in, ld_out, dtype) -> int:
    return int(load().softmax_rows_split_workspace_bytes(_ptr(in_), _ptr(out), M, N, ld_in,
                                                         ld_out, dtype))


def softmax_rows_host_workspace_bytes(M, N, dtype) -> int:
    return int(load().softmax_rows_host_workspace_bytes(M, N, dtype))


def softmax_rows_strerror(status: int) -> str:
    try:
        return load().softmax_rows_strerror(status).decode()
    except RuntimeError:
        return "status %d" % status


def softmax_rows_copy_ceiling2(a, b, out, M, row_bytes, ld_a_bytes, ld_b_bytes, ld_out_bytes,
                               stream=None) -> int:
    return _check(load().softmax_rows_copy_ceiling2(_ptr(a), _ptr(b), _ptr(out), M, row_bytes,
                                                    ld_a_bytes, ld_b_bytes, ld_out_bytes,
                                                    _stream(stream)),
                  "softmax_rows_copy_ceiling2")


def softmax_rows_copy_ceiling(in_, out, M, row_bytes, ld_in_bytes, ld_out_bytes,
                              stream=None) -> int:
    return _check(load().softmax_rows_copy_ceiling(_ptr(in_), _ptr(out), M, row_bytes,
                                                   ld_in_bytes, ld_out_bytes, _stream(stream)),
                  "softmax_rows_copy_ceiling")


def softmax_rows_version() -> int:
    return int(load().softmax_rows_version())


class LaunchInfo(ctypes.Structure):
    """Mirror of sr_launch_info."""
    _fields_ = [("registers", ctypes.c_int), ("local_bytes", ctypes.c_int),
                ("static_smem_bytes", ctypes.c_int), ("dynamic_smem_bytes", ctypes.c_int),
                ("grid", ctypes.c_int), ("block", ctypes.c_int), ("cluster", ctypes.c_int),
                ("name", ctypes.c_char * 256)]


def softmax_rows_last_launch() -> dict:
    """The calling thread's last kernel launch through the library, as a dict
    (registers, local_bytes, static_smem_bytes, dynamic_smem_bytes, grid, block,
    cluster, name)."""
    info = LaunchInfo()
    _check(load().softmax_rows_last_launch(ctypes.byref(info)), "softmax_rows_last_launch")
    d = {name: getattr(info, name) for name, _ in LaunchInfo._fields_}
    d["name"] = info.name.decode(errors="replace")
    return d


def dtype_code(torch_dtype) -> int:
    import torch
    codes = {torch.float32: SR_F32, torch.bfloat16: SR_BF16, torch.float16: SR_F16}
    if torch_dtype not in codes:
        raise TypeError("softmax_rows supports float32, bfloat16 and float16, not %s" % torch_dtype)
    return codes[torch_dtype]


def softmax(x, out=None, plan: int = SR_PLAN_AUTO, stream=None):
    """Row softmax of a 2-D CUDA tensor with unit column stride (any row stride).

    ``out`` (optional) is a CUDA tensor of the same shape and dtype with unit
    column stride; a new contiguous tensor is returned otherwise.
    """
    import torch
    if x.dim() != 2 or x.stride(1) != 1 or not x.is_cuda:
        raise ValueError("expected a 2-D CUDA tensor with unit column stride")
    M, N = x.shape
    if out is None:
        out = torch.empty((M, N), dtype=x.dtype, device=x.device)
    if out.shape != x.shape or out.dtype != x.dtype or out.stride(1) != 1:
        raise ValueError("out must match x in shape and dtype, with unit column stride")
    ld_in = x.stride(0) if M > 1 else N
    ld_out = out.stride(0) if M > 1 else N
    softmax_rows_ex(x, out, M, N, ld_in, ld_out, dtype_code(x.dtype), plan, stream)
    return out


def softmax_backward(y, dy, dx=None, plan: int = SR_PLAN_AUTO, stream=None):
    """Softmax backward of 2-D CUDA tensors with unit column stride.

    ``y`` is the softmax output and ``dy`` the gradient of the loss with
    respect to it; returns dx (a new contiguous tensor unless ``dx`` is given).
    """
    import torch
    for name, t in (("y", y), ("dy", dy)):
        if t.dim() != 2 or t.stride(1) != 1 or not t.is_cuda:
            raise ValueError("%s: expected a 2-D CUDA tensor with unit column stride" % name)
    if dy.shape != y.shape or dy.dtype != y.dtype:
        raise ValueError("y and dy must have the same shape and dtype")
    M, N = y.shape
    if dx is None:
        dx = torch.empty((M, N), dtype=y.dtype, device=y.device)
    if dx.shape != y.shape or dx.dtype != y.dtype or dx.stride(1) != 1:
        raise ValueError("dx must match y in shape and dtype, with unit column stride")
    ld = lambda t: t.stride(0) if M > 1 else N
    softmax_rows_backward_ex(y, dy, dx, M, N, ld(y), ld(dy), ld(dx), dtype_code(y.dtype), plan,
                             stream)
    return dx


def rmsnorm_residual(x, residual, weight, eps: float = 1e-6, y=None, plan: int = SR_PLAN_AUTO,
                     stream=None):
    """Residual RMSNorm of 2-D CUDA tensors with unit column stride; weight is 1-D."""
    import torch
    for name, t in (("x", x), ("residual", residual)):
        if t.dim() != 2 or t.stride(1) != 1 or not t.is_cuda:
            raise ValueError("%s: expected a 2-D CUDA tensor with unit column stride" % name)
    if residual.shape != x.shape or residual.dtype != x.dtype:
        raise ValueError("x and residual must have the same shape and dtype")
    M, N = x.shape
    if weight.dim() != 1 or weight.shape[0] != N or weight.dtype != x.dtype or \
            not weight.is_contiguous():
        raise ValueError("weight must be a contiguous vector of N elements of x's dtype")
    if y is None:
        y = torch.empty((M, N), dtype=x.dtype, device=x.device)
    if y.shape != x.shape or y.dtype != x.dtype or y.stride(1) != 1:
        raise ValueError("y must match x in shape and dtype, with unit column stride")
    ld = lambda t: t.stride(0) if M > 1 else N
    rmsnorm_residual_rows_ex(x, residual, weight, y, M, N, ld(x), ld(residual), ld(y), eps,
                             dtype_code(x.dtype), plan, stream)
    return y
