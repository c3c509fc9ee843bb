"""Builds libamk.so in-tree: the persistent decode kernel for sm_103a, the
planner and the C ABI.  Translation units compile in parallel; the CUDA
runtime is linked statically so the library loads wherever the driver does.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJ = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libamk.so")

SOURCES = ["amk_kernel.cu", "amk_api.cpp", "amk_plan.cpp", "amk_noalloc.cu", "amk_unfused.cu"]
HEADERS = ["amk_internal.h", "amk_launch.h", "amk_plan_impl.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """AMK_TRACE=1 in the environment builds the tuning variant whose kernel
    carries the per-task timing code (schedule option ``trace``);
    AMK_L2_PREFETCH=1 the one with the loader's L2 prefetch (schedule option
    ``l2_prefetch_kb``)."""
    os.makedirs(OBJ, exist_ok=True)
    hdrs = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, h)
                                                       for h in ("amk.h", "amk_plan.h", "amk_unfused.h")]
    flags = list(extra_flags)
    if os.environ.get("AMK_TRACE", "0") not in ("", "0"):
        flags.append("-DAMK_TRACE_CODE=1")
    if os.environ.get("AMK_L2_PREFETCH", "0") not in ("", "0"):
        flags.append("-DAMK_L2_PREFETCH_CODE=1")
    stamp = os.path.join(OBJ, "flags.txt")
    prev = open(stamp).read() if os.path.exists(stamp) else None
    if prev != " ".join(flags):
        # objects of other flags may be left behind: rebuild everything, and
        # keep no stamp until the whole build has succeeded
        force = True
        if prev is not None:
            os.remove(stamp)
    common = ["-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC] + flags
    procs, objs = [], []
    for src in SOURCES:
        path = os.path.join(CSRC, src)
        obj = os.path.join(OBJ, src + ".o")
        objs.append(obj)
        if force or _stale(obj, [path] + hdrs):
            cmd = [nvcc()] + common + ARCH + ["-c", path, "-o", obj + ".tmp"]
            if src.endswith(".cu"):
                cmd += ["-lineinfo", "-Xptxas", "-v"] if verbose else ["-lineinfo"]
            procs.append((subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT), obj, cmd))
    failed = []
    for p, obj, cmd in procs:
        out, _ = p.communicate()
        if verbose or p.returncode:
            sys.stderr.write(out.decode(errors="replace"))
        if p.returncode:
            failed.append(" ".join(cmd))
        else:
            os.replace(obj + ".tmp", obj)
    if failed:
        raise RuntimeError("compilation failed:\n" + "\n".join(failed))
    if force or _stale(LIB, objs):
        tmp = LIB + ".%d.tmp" % os.getpid()
        subprocess.check_call([nvcc()] + ARCH + ["-shared", "-o", tmp] + objs + ["-cudart", "static"])
        os.replace(tmp, LIB)
    with open(stamp, "w") as f:
        f.write(" ".join(flags))
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
