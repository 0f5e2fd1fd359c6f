"""Build libringattn.so in-tree: nvcc for sm_103a only, translation units in parallel.

Output: ``context_exact_attention_gb300/libringattn.so`` (git-ignored).  The CUDA
runtime is linked statically and the driver is reached through the runtime's
entry-point query, so the library loads on a machine without a GPU driver.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libringattn.so")
# the debug build: same sources with every computed global index checked (-DRA_DEBUG_BOUNDS)
BUILD_DEBUG = os.path.join(PKG, "_build_debug")
LIB_DEBUG = os.path.join(PKG, "libringattn_debug.so")
SOURCES = ["api.cu", "attn_bf16_sm103.cu", "attn_bwd_sm103.cu", "attn_f32.cu", "merge.cu",
           "ulysses.cu", "host_pipeline.cu", "bwd_noalloc.cu", "varlen_schedule.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I" + INCLUDE, "-I" + CSRC]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libringattn.so")


def _inputs():
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    deps.append(os.path.join(INCLUDE, "ring_attn.h"))
    deps.append(os.path.abspath(__file__))
    return deps


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
          debug_bounds: bool = False) -> str:
    """Compile libringattn.so, or with debug_bounds=True libringattn_debug.so (every
    computed global index checked against its tensor's extent; see ra_check.cuh)."""
    out_lib, out_dir = (LIB_DEBUG, BUILD_DEBUG) if debug_bounds else (LIB, BUILD)
    if not force and up_to_date(out_lib):
        return out_lib
    nvcc = _nvcc()
    os.makedirs(out_dir, exist_ok=True)
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    if debug_bounds:
        extra.append("-DRA_DEBUG_BOUNDS")

    def compile_one(src):
        obj = os.path.join(out_dir, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose or ptxas_info:
            print(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = out_lib + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", *objs, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out_lib)
    return out_lib


if __name__ == "__main__":
    import sys

    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv,
                debug_bounds="--debug-bounds" in sys.argv))
