"""Build the CUDA library in-tree: ``_build/libfa_gb300.so`` (sm_103a only).

Each translation unit compiles in its own nvcc process (in parallel), then
one nvcc call links the shared library.  No CMake, no torch extension
machinery: the library exports the plain C ABI of ``include/fa.h``.

The same call builds the debug library ``_build/libfa_gb300_debug.so``: the
release objects with the attention kernels' units recompiled with ``FA_DEBUG``
(device index checks and the fault knobs of ``include/fa_debug.h``).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libfa_gb300.so")
DEBUG_LIB_PATH = os.path.join(BUILD_DIR, "libfa_gb300_debug.so")
# recompiled with FA_DEBUG for the debug library
DEBUG_SOURCES = ["fa_fwd_sm103.cu", "fa_fwd256_sm103.cu", "fa_bwd_sm103.cu", "fa_bwd256_sm103.cu",
                 "fa_decode_sm103.cu"]
SOURCES = ["fa_api.cu", "fa_fwd_sm103.cu", "fa_fwd256_sm103.cu", "fa_bwd_sm103.cu",
           "fa_bwd256_sm103.cu", "fa_decode_sm103.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _inputs_mtime() -> float:
    paths = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    inc = os.path.join(ROOT, "include")
    paths += [os.path.join(inc, f) for f in os.listdir(inc)]
    paths.append(os.path.abspath(__file__))
    return max(os.path.getmtime(p) for p in paths)


def build_library(force: bool = False, verbose_ptxas: bool = False) -> str:
    os.makedirs(BUILD_DIR, exist_ok=True)
    if not force:
        newest = _inputs_mtime()
        if all(os.path.exists(p) and os.path.getmtime(p) >= newest
               for p in (LIB_PATH, DEBUG_LIB_PATH)):
            return LIB_PATH
    nvcc = nvcc_path()
    common = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-I", os.path.join(ROOT, "include")]
    if verbose_ptxas:
        common += ["-Xptxas", "-v"]

    def compile_one(job):
        src, debug = job
        obj = os.path.join(BUILD_DIR, src.replace(".cu", "_debug.o" if debug else ".o"))
        cmd = [nvcc] + common + (["-DFA_DEBUG"] if debug else [])
        cmd += ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return src, debug, obj, r.stdout + r.stderr

    jobs = [(s, False) for s in SOURCES] + [(s, True) for s in DEBUG_SOURCES]
    with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        results = list(ex.map(compile_one, jobs))
    if verbose_ptxas:
        for src, debug, _, log in results:
            print(f"== {src}{' (FA_DEBUG)' if debug else ''}\n{log}")
    release = {src: obj for src, debug, obj, _ in results if not debug}
    debug_objs = {src: obj for src, debug, obj, _ in results if debug}

    def link(objs, path):
        tmp = path + f".tmp{os.getpid()}"
        cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, path)

    link([release[s] for s in SOURCES], LIB_PATH)
    link([debug_objs.get(s, release[s]) for s in SOURCES], DEBUG_LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    import sys
    print(build_library(force=True, verbose_ptxas="-v" in sys.argv))
