"""Builds libswiglu_mlp.so (release) and libswiglu_mlp_debug.so (the same
sources with -DSWIGLU_DEBUG: device index checks) in place with nvcc for
sm_103a (GB300).  The two compile in parallel."""
from __future__ import annotations

import glob
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
SO = os.path.join(HERE, "libswiglu_mlp.so")
SO_DEBUG = os.path.join(HERE, "libswiglu_mlp_debug.so")
SOURCES = ["swiglu_mlp.cu"]

NVCC_FLAGS = [
    "-std=c++17", "-O3", "-lineinfo",
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-Xcompiler", "-fPIC", "-shared",
]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _stale(so: str) -> bool:
    if not os.path.exists(so):
        return True
    t = os.path.getmtime(so)
    deps = [os.path.join(CSRC, f) for f in SOURCES]
    deps += glob.glob(os.path.join(CSRC, "*.cuh"))
    deps.append(os.path.join(ROOT, "include", "swiglu_mlp.h"))
    deps.append(os.path.abspath(__file__))
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile whichever of the two libraries is missing or out of date;
    returns the release library's path."""
    jobs = []
    for so, extra in ((SO, []), (SO_DEBUG, ["-DSWIGLU_DEBUG"])):
        if not force and not _stale(so):
            continue
        tmp = so + ".%d.tmp" % os.getpid()
        cmd = [_nvcc(), *NVCC_FLAGS, *extra, "-o", tmp] + [os.path.join(CSRC, f) for f in SOURCES]
        if verbose:
            print(" ".join(cmd))
        jobs.append((subprocess.Popen(cmd), tmp, so, cmd))
    failed = None
    for proc, tmp, so, cmd in jobs:
        if proc.wait() != 0:
            failed = failed or subprocess.CalledProcessError(proc.returncode, cmd)
        else:
            os.replace(tmp, so)
    if failed is not None:
        raise failed
    return SO


if __name__ == "__main__":
    print(build(force=True, verbose=True))
