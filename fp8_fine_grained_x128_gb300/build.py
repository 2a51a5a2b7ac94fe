"""Build the CUDA library libfp8fg.so in-tree for sm_103a (GB300).

Every translation unit under csrc/ is compiled by nvcc in parallel with
``-gencode arch=compute_103a,code=sm_103a`` (IEEE division and denormals kept:
no fast-math), then linked into ``fp8_fine_grained_x128_gb300/libfp8fg.so``.
ptxas register / spill reports are written to ``_build/ptxas.log``.

``--debug`` builds the index-checked variant ``libfp8fg_debug.so`` instead
(objects in ``_build_debug/``): the same sources compiled with
``-DFP8FG_DEBUG``, in which every kernel store checks its index against the
extent of the buffer it writes and records FP8_ERR_BOUNDS on a miss.  The
binding loads it when FP8FG_DEBUG=1 is set in the environment.

    python -m fp8_fine_grained_x128_gb300.build [--force] [--debug]
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libfp8fg.so")
BUILD_DEBUG = os.path.join(HERE, "_build_debug")
LIB_DEBUG = os.path.join(HERE, "libfp8fg_debug.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
              "--expt-relaxed-constexpr", "-I", INCLUDE]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA library cannot be built")


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    return [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "fp8fg.h")]


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, build_dir: str, extra: list) -> tuple[str, str]:
    obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
    p = subprocess.run(cmd, capture_output=True, text=True)
    if p.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{p.stdout}\n{p.stderr}")
    return obj, p.stderr


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    build_dir, lib = (BUILD_DEBUG, LIB_DEBUG) if debug else (BUILD, LIB)
    extra = ["-DFP8FG_DEBUG"] if debug else []
    os.makedirs(build_dir, exist_ok=True)
    deps = _deps()
    if not force and not _stale(lib, deps):
        return lib
    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 1)) as ex:
        results = list(ex.map(lambda src: _compile(src, build_dir, extra), srcs))
    with open(os.path.join(build_dir, "ptxas.log"), "w") as f:
        for (obj, log) in results:
            f.write(f"==== {os.path.basename(obj)}\n{log}\n")
    tmp = lib + f".{os.getpid()}.tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-Xcompiler", "-fPIC", "-o", tmp, *[o for o, _ in results]]
    p = subprocess.run(cmd, capture_output=True, text=True)
    if p.returncode != 0:
        raise RuntimeError(f"link failed:\n{p.stdout}\n{p.stderr}")
    os.replace(tmp, lib)
    if verbose:
        print(f"built {lib}")
    return lib


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, debug="--debug" in sys.argv)
