"""Compile the CUDA library in-tree for sm_103a: csrc/*.cu -> lib/libddtree.so.

Each translation unit is compiled in parallel with nvcc and linked into one
shared object with the CUDA runtime linked statically, so the library needs
nothing at run time but the driver.  Objects are rebuilt only when a source or
header is newer than them.

build(variant="testhooks") compiles the same sources with test-only hooks into
lib/libddtree_testhooks.so: short bounded-wait limits, a switch that makes the
prefix kernel skip the loads of one pipeline step (so a wait runs out and the
kernel reports DDT_STATUS_TIMEOUT), and counters of the lazy O rescales and of
the units rerun with 20-bit score exchange.  Only tests load it.
"""
from __future__ import annotations

import concurrent.futures
import glob
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "lib", "libddtree.so")
VARIANTS = {
    "release": (BUILD, LIB, ()),
    "testhooks": (os.path.join(HERE, "_build_testhooks"), os.path.join(HERE, "lib", "libddtree_testhooks.so"),
                  ("-DDDT_TEST_HOOKS", "-DDDT_WAIT_LIMIT=(1u<<14)", "-DDDT_DRAIN_LIMIT=(1u<<12)")),
}
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC = os.environ.get("NVCC", "nvcc")
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "-I", os.path.join(ROOT, "include")]


def _headers():
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(ROOT, "include", "*.h"))


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src, build_dir, defines=(), extra=()):
    obj = os.path.join(build_dir, os.path.basename(src).replace(".cu", ".o"))
    if _stale(obj, [src, *_headers()]) or extra:
        cmd = [NVCC, *ARCH, *FLAGS, *defines, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj


def build(verbose_ptxas: bool = False, variant: str = "release") -> str:
    """Build lib/libddtree.so (or the test-hooks variant); returns its path."""
    build_dir, lib, defines = VARIANTS[variant]
    os.makedirs(build_dir, exist_ok=True)
    os.makedirs(os.path.dirname(lib), exist_ok=True)
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    extra = ("-Xptxas", "-v") if verbose_ptxas else ()
    with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, min(len(sources), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(lambda s: _compile(s, build_dir, defines, extra), sources))
    if _stale(lib, objs):
        cmd = [NVCC, *ARCH, "-shared", "-o", lib, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    return lib


if __name__ == "__main__":
    import sys
    print(build(variant=sys.argv[1] if len(sys.argv) > 1 else "release"))
