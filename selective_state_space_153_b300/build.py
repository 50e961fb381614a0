"""Build the CUDA library libssm_scan.so in-tree (sm_103a only).

    python -m selective_state_space_153_b300.build [--force]

Every kernel family is its own translation unit (csrc/k_*.cu, plus the host logic in
csrc/ssm_api.cu), compiled as relocatable device code in parallel and linked into one shared
library (the device status word is defined once, in ssm_api.cu).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libssm_scan.so")
OBJ = os.path.join(PKG, "_build")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# Host symbols are hidden (only what include/ssm_scan.h declares is exported) and template
# statics are not "unique" symbols, so that two builds of the library loaded into one process
# (the normal and the checked build) share no state.
NVCC_FLAGS = ["-O3", "-std=c++17", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC,-fvisibility=hidden,-fno-gnu-unique",
              "--expt-relaxed-constexpr"]


def sources():
    return sorted(f for f in os.listdir(CSRC) if f.endswith(".cu"))


def _nvcc() -> str:
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(home, "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _deps():
    return [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "ssm_scan.h"),
                                                                 os.path.abspath(__file__)]


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(f) > t for f in deps)


def build(force: bool = False, verbose: bool = False, extra=(), lib: str = LIB, objdir: str = OBJ,
          jobs: int = 0) -> str:
    """Compile every csrc/*.cu (in parallel) and link ``lib``. ``extra``: additional nvcc
    flags (e.g. ``-DSSM_CHECK``; a build with extra flags should name its own ``lib`` and
    ``objdir``)."""
    deps = _deps()
    if not force and not _stale(lib, deps):
        return lib
    os.makedirs(objdir, exist_ok=True)
    nvcc = _nvcc()
    objs = []

    def compile_one(src):
        obj = os.path.join(objdir, src[:-3] + ".o")
        cmd = [nvcc, *NVCC_FLAGS, *extra, "-dc", "-I", INCLUDE, "-I", CSRC, "-o", obj + ".tmp",
               os.path.join(CSRC, src)]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src} ({r.returncode}):\n{r.stderr[-8000:]}")
        os.replace(obj + ".tmp", obj)
        return obj

    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=jobs or min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-Xcompiler", "-fPIC", "-o", tmp, *objs]
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed ({r.returncode}):\n{r.stderr[-8000:]}")
    os.replace(tmp, lib)
    return lib


CHECK_LIB = os.path.join(PKG, "libssm_scan_check.so")


def build_checked(force: bool = False, verbose: bool = False) -> str:
    """The checked build (-DSSM_CHECK): bounds checks on every global and shared-memory access
    of the scan and state-update kernels, NaN-poisoned shared memory. For tests."""
    return build(force=force, verbose=verbose, extra=("-DSSM_CHECK",), lib=CHECK_LIB,
                 objdir=os.path.join(OBJ, "check"))


PROBE_SRC = os.path.join(PKG, "probe", "ex2_rate.cu")
PROBE_LIB = os.path.join(PKG, "libssm_probe.so")


def build_probe(force: bool = False, verbose: bool = False) -> str:
    """The ex2-throughput probe the benchmark's roofline uses (not part of the scan library)."""
    if not force and not _stale(PROBE_LIB, [PROBE_SRC, os.path.abspath(__file__)]):
        return PROBE_LIB
    cmd = [_nvcc(), *NVCC_FLAGS, "-shared", "-o", PROBE_LIB + ".tmp", PROBE_SRC]
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on the probe ({r.returncode}):\n{r.stderr[-8000:]}")
    os.replace(PROBE_LIB + ".tmp", PROBE_LIB)
    return PROBE_LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
    print(build_probe(force="--force" in sys.argv, verbose=True))
    print(build_checked(force="--force" in sys.argv, verbose=True))
