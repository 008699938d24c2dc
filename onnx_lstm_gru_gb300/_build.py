"""Build the CUDA library librk.so in-tree for sm_103a with nvcc.

One nvcc process per translation unit, run in parallel, then one shared-object
link.  Objects are rebuilt when any source or header is newer than them.
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
LIB = os.path.join(BUILD, "librk.so")
# measurement aid of the benchmark (float32 FMA peak), its own shared object
PROBE_SRC = os.path.join(PKG, "probe", "fma_peak.cu")
PROBE_LIB = os.path.join(BUILD, "libfmapeak.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
          "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build librk.so")
    return cand


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))


def _headers():
    return glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


def build(force: bool = False, jobs: int | None = None, verbose: bool = False) -> str:
    """Compile every translation unit under csrc/ and link _build/librk.so."""
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    hdr_time = max([os.path.getmtime(h) for h in _headers()] + [0.0])
    srcs = sources()
    todo = []
    objs = []
    for src in srcs:
        obj = os.path.join(BUILD, os.path.basename(src) + ".o")
        objs.append(obj)
        if force or not os.path.exists(obj) or os.path.getmtime(obj) < max(os.path.getmtime(src), hdr_time):
            todo.append((src, obj))

    def compile_one(item):
        src, obj = item
        tmp = obj + f".{os.getpid()}.tmp"
        cmd = [nvcc, *ARCH, *CFLAGS, "-c", src, "-o", tmp]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stderr}")
        os.replace(tmp, obj)
        return r.stderr

    if todo:
        n = jobs or min(len(todo), max(1, os.cpu_count() or 1))
        with cf.ThreadPoolExecutor(max_workers=n) as ex:
            for log in ex.map(compile_one, todo):
                if verbose and log:
                    print(log)
    lib_time = os.path.getmtime(LIB) if os.path.exists(LIB) else -1.0
    if todo or lib_time < max(os.path.getmtime(o) for o in objs):
        tmp = LIB + f".{os.getpid()}.tmp"
        cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link of librk.so failed:\n{r.stderr}")
        os.replace(tmp, LIB)
    if not os.path.exists(PROBE_LIB) or os.path.getmtime(PROBE_LIB) < os.path.getmtime(PROBE_SRC):
        tmp = PROBE_LIB + f".{os.getpid()}.tmp"
        cmd = [nvcc, *ARCH, *CFLAGS, "-shared", PROBE_SRC, "-o", tmp]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"build of libfmapeak.so failed:\n{r.stderr}")
        os.replace(tmp, PROBE_LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
