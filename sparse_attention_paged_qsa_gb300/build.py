"""Build libqsa.so (the CUDA kernels and the C ABI) in-tree for sm_103a with nvcc.

Also builds libqsa_testhooks.so: the decode compiled with -DQSA_TEST_HOOKS, whose
one extra export lets the GPU tests stall a pipeline stage to drive the bounded
waits. The shipped libqsa.so carries no test hook. The translation units compile
in parallel, one nvcc process each.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
SOURCES = [os.path.join(CSRC, f) for f in ("qsa_decode.cu", "qsa_kv_write.cu", "qsa_topk.cu")]
HEADERS = [os.path.join(ROOT, "include", "qsa.h")]
LIB = os.path.join(PKG, "libqsa.so")
TEST_LIB = os.path.join(PKG, "libqsa_testhooks.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libqsa.so")


def _stale(out: str, inputs) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(f) > t for f in inputs)


def needs_build() -> bool:
    return _stale(LIB, SOURCES + HEADERS) or _stale(TEST_LIB, SOURCES[:1] + HEADERS)


def _flags(verbose: bool):
    f = [*ARCH, "-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC",
         "-I", os.path.join(ROOT, "include")]
    return f + (["-Xptxas=-v"] if verbose else [])


def build_library(force: bool = False, verbose: bool = False) -> str:
    """Compile every CUDA source into libqsa.so (and the decode into
    libqsa_testhooks.so) next to this file; returns the libqsa.so path."""
    if not force and not needs_build():
        return LIB
    tag = f".tmp{os.getpid()}"
    objs = [os.path.join(PKG, os.path.basename(s) + tag + ".o") for s in SOURCES]
    test_obj = os.path.join(PKG, "qsa_decode_testhooks" + tag + ".o")
    jobs = [[nvcc(), *_flags(verbose), "-c", s, "-o", o] for s, o in zip(SOURCES, objs)]
    jobs.append([nvcc(), *_flags(False), "-DQSA_TEST_HOOKS", "-c", SOURCES[0], "-o", test_obj])
    try:
        with ThreadPoolExecutor(len(jobs)) as ex:
            for r in ex.map(lambda c: subprocess.run(c), jobs):
                if r.returncode != 0:
                    raise subprocess.CalledProcessError(r.returncode, r.args)
        for out, inputs in ((LIB, objs), (TEST_LIB, [test_obj])):
            tmp = out + tag
            subprocess.run([nvcc(), *ARCH, "-shared", "-cudart", "shared", *inputs, "-o", tmp],
                           check=True)
            os.replace(tmp, out)
    finally:
        for o in objs + [test_obj]:
            if os.path.exists(o):
                os.remove(o)
    return LIB


if __name__ == "__main__":
    print(build_library(force=True, verbose=True))
