"""In-tree build of ``libqgemv.so`` for sm_103a with nvcc (no cmake).

Each translation unit compiles in its own nvcc process, in parallel, then the
objects are linked into one shared library under ``_build/``.

``build(debug=True)`` (``python -m block_quantized_gemv_quantize_gb300.build
--debug``) makes the bounds-checking library ``_build/debug/libqgemv.so``
instead: the same sources with ``-DQGEMV_BOUNDS_CHECK``, whose kernels check
the indexes of their computed accesses and record failures in the library's
status page (read by ``qgemv_take_bounds_errors``) instead of faulting.  The
binding loads it when the environment has ``QGEMV_BOUNDS_CHECK=1``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libqgemv.so")
BUILD_DEBUG = os.path.join(BUILD, "debug")
LIB_DEBUG = os.path.join(BUILD_DEBUG, "libqgemv.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-Xptxas", "-warn-spills"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps() -> list[str]:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cuh"))]
    files.append(os.path.join(INCLUDE, "qgemv.h"))
    return files


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None,
          debug: bool = False) -> str:
    """Compile every CUDA source and link libqgemv.so (the bounds-checking
    one under _build/debug with debug=True); returns its path."""
    lib, bdir = (LIB_DEBUG, BUILD_DEBUG) if debug else (LIB, BUILD)
    if not force and up_to_date(lib):
        return lib
    os.makedirs(bdir, exist_ok=True)
    nvcc = _nvcc()
    flags = ARCH + NVCC_FLAGS + ["-I", INCLUDE] + (["-DQGEMV_BOUNDS_CHECK"] if debug else []) + (extra_flags or [])

    def compile_one(src: str) -> str:
        obj = os.path.join(bdir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    srcs = sources()
    with ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib + f".tmp{os.getpid()}"
    r = subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-lcudart"], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys

    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug="--debug" in sys.argv))
