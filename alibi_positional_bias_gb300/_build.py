"""In-tree build of the CUDA library (sm_103a) with nvcc.

Each translation unit in ``csrc/`` is compiled in parallel, then linked into
``_build/libalibi_gb300.so`` (static CUDA runtime, no driver-library link: the
TMA encoder is fetched through the runtime's driver entry-point query).

``build(checks=True)`` compiles the same sources with ``-DALIBI_CHECKS`` into
``_build/libalibi_gb300_checks.so``: the debug-checks library, whose kernels test
every TMA coordinate, TMEM address and shared-memory operand before use and
record a failure in the device status word (``csrc/checks.h``). It is built on
demand (its test builds it), not by the default build.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libalibi_gb300.so")
BUILD_CHECKS = os.path.join(BUILD, "checks")
LIB_CHECKS = os.path.join(BUILD, "libalibi_gb300_checks.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
          f"-I{INCLUDE}", f"-I{CSRC}"]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")
    return exe


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _headers() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh"))
                  + glob.glob(os.path.join(INCLUDE, "*.h")))


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False, checks: bool = False) -> str:
    """Compile and link the library if any source or header changed. Returns the .so path."""
    odir, lib = (BUILD_CHECKS, LIB_CHECKS) if checks else (BUILD, LIB)
    os.makedirs(odir, exist_ok=True)
    srcs = sources()
    hdrs = _headers()
    objs = [os.path.join(odir, os.path.basename(s)[:-3] + ".o") for s in srcs]
    todo = [(s, o) for s, o in zip(srcs, objs) if force or _stale(o, [s] + hdrs)]
    exe = nvcc()

    def compile_one(so):
        s, o = so
        cmd = [exe, *ARCH, *CFLAGS, *(["-DALIBI_CHECKS"] if checks else []), "-c", s, "-o", o + ".tmp"]
        if ptxas_info:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {os.path.basename(s)}:\n{r.stderr}")
        os.replace(o + ".tmp", o)
        return r.stderr

    if todo:
        with cf.ThreadPoolExecutor(max_workers=max(1, min(len(todo), os.cpu_count() or 1))) as ex:
            for log in ex.map(compile_one, todo):
                if verbose and log:
                    print(log)
    if force or todo or _stale(lib, objs):
        tmp = lib + f".{os.getpid()}.tmp"
        r = subprocess.run([exe, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr}")
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv,
                checks="--checks" in sys.argv))
