"""Build the CUDA library in-tree: nvcc, sm_103a only, translation units in parallel.

Produces ``memory_bound_row_rows_gb300/lib/libsoftmax_rows.so`` (statically
linked CUDA runtime, C ABI declared in ``include/softmax_rows.h``). A stamp of
the sources and flags skips the rebuild when nothing changed.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIBDIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIBDIR, "libsoftmax_rows.so")
# The bounds-checking debug build: every kernel checks its global accesses
# against the call's matrices (SR_BOUNDS_CHECK); relocatable device code lets
# the checks in every translation unit reach the one device error word.
CHECK_LIB = os.path.join(LIBDIR, "libsoftmax_rows_check.so")
CHECK_FLAGS = ["-DSR_BOUNDS_CHECK=1", "-rdc=true"]
HEADER = os.path.join(ROOT, "include", "softmax_rows.h")

UNITS = ["api.cu", "warp_rows.cu", "tma_rows.cu", "online_rows.cu", "smem_rows.cu",
         "block_rows.cu", "host_stream.cu",
         "split_rows.cu", "backward_rows.cu", "rmsnorm_rows.cu", "wide_rows.cu", "copy_rows.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden", "-Xptxas", "-v"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build softmax_rows")


def _stamp(extra_flags) -> str:
    h = hashlib.sha256()
    for name in sorted(os.listdir(CSRC)):
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode() + f.read())
    with open(HEADER, "rb") as f:
        h.update(f.read())
    h.update(" ".join(ARCH + NVCC_FLAGS + list(extra_flags)).encode())
    return h.hexdigest()


# Sources each plan's kernel is built from (besides the shared headers).
PLAN_SOURCES = {
    "row": ["block_rows.cu", "packed.cuh"], "warp": ["warp_rows.cu", "packed.cuh"], "cta": ["tma_rows.cu"],
    "cluster": ["tma_rows.cu"], "smem": ["smem_rows.cu"], "online": ["online_rows.cu"],
    "split": ["split_rows.cu", "split.h"], "wide": ["wide_rows.cu", "wide.h", "packed.cuh", "l2prefetch.cuh"],
    "backward": ["backward_rows.cu", "rowpair.cuh", "rowpair.h"],
    "rmsnorm": ["rmsnorm_rows.cu", "rowpair.cuh", "rowpair.h"],
    "copy": ["copy_rows.cu"],
}
SHARED_SOURCES = ["device.cuh", "internal.h"]


def source_hash(files=None) -> str:
    """Hash of kernel sources and build flags, tying profiler counters to a build.

    ``files`` (names under csrc/) limits it to one kernel's sources plus the
    shared device headers; None hashes every source.
    """
    if files is None:
        return _stamp([])[:16]
    h = hashlib.sha256()
    for name in sorted(set(files) | set(SHARED_SOURCES)):
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode() + f.read())
    h.update(" ".join(ARCH + NVCC_FLAGS).encode())
    return h.hexdigest()[:16]


def build(force: bool = False, extra_flags=(), out: str | None = None, verbose: bool = False,
          jobs: int | None = None) -> str:
    out = out or LIB
    os.makedirs(os.path.dirname(out), exist_ok=True)
    stamp_path = out + ".stamp"
    stamp = _stamp(extra_flags)
    if not force and os.path.exists(out) and os.path.exists(stamp_path):
        with open(stamp_path) as f:
            if f.read().strip() == stamp:
                return out
    objdir = out + ".obj"
    os.makedirs(objdir, exist_ok=True)
    cc = nvcc()

    def compile_unit(unit):
        obj = os.path.join(objdir, unit + ".o")
        cmd = [cc, *ARCH, *NVCC_FLAGS, *extra_flags, "-I", os.path.join(ROOT, "include"),
               "-c", os.path.join(CSRC, unit), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed on %s:\n%s\n%s" % (unit, r.stdout, r.stderr))
        with open(obj + ".ptxas.log", "w") as f:
            f.write(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=jobs or len(UNITS)) as ex:
        objs = list(ex.map(compile_unit, UNITS))
    tmp = out + ".tmp%d" % os.getpid()
    link_flags = [f for f in extra_flags if f.startswith("-rdc")]
    cmd = [cc, *ARCH, *link_flags, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc link failed:\n%s\n%s" % (r.stdout, r.stderr))
    os.replace(tmp, out)
    with open(stamp_path, "w") as f:
        f.write(stamp)
    if verbose:
        print("built", out)
    return out


def build_checked(force: bool = False, verbose: bool = False, jobs: int | None = None) -> str:
    """The bounds-checking debug build (same entry points, lib/libsoftmax_rows_check.so)."""
    return build(force=force, extra_flags=CHECK_FLAGS, out=CHECK_LIB, verbose=verbose, jobs=jobs)


if __name__ == "__main__":
    build(force=True, verbose=True)
