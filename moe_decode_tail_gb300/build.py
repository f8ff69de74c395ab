"""Build the CUDA library libmoetail.so in-tree (sm_103a only).

Each translation unit compiles in parallel with nvcc, then the objects link
into one shared library whose only exported symbols are the C ABI of
include/moe_tail.h.  The CUDA runtime is linked statically, so the library
needs only the driver at run time.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libmoetail.so")
TRACE_LIB = os.path.join(BUILD, "libmoetail_trace.so")  # the same kernels with the per-CTA trace
FLOOR_LIB = os.path.join(BUILD, "libmoetail_floor.so")  # latency-floor kernels (measurement only)
SOURCES = ["finalize.cu", "decode_gemm.cu", "moe_tail_api.cu", "noalloc.cu"]
FLOOR_SOURCES = ["floor.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + [
    "-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr",
    "-Xcompiler", "-fPIC,-fvisibility=hidden,-O2",
    "-I", os.path.join(ROOT, "include"),
]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmoetail.so")
    return exe


def _inputs(sources=SOURCES) -> list[str]:
    files = [os.path.join(CSRC, s) for s in sources]
    files += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    files.append(os.path.join(ROOT, "include", "moe_tail.h"))
    files.append(os.path.join(ROOT, "include", "moe_tail_trace.h"))
    files.append(os.path.join(ROOT, "include", "moe_tail_floor.h"))
    return files


def up_to_date(lib: str = LIB, sources=SOURCES) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _inputs(sources))


def build(force: bool = False, verbose: bool = False, ptxas_v: bool = False, trace: bool = False,
          floor: bool = False) -> str:
    """Build libmoetail.so, or with trace=True libmoetail_trace.so (the same
    kernels recording a per-CTA timeline; see include/moe_tail_trace.h), or
    with floor=True libmoetail_floor.so (the latency-floor kernels of
    include/moe_tail_floor.h, used by bench.py only)."""
    lib = FLOOR_LIB if floor else TRACE_LIB if trace else LIB
    sources = FLOOR_SOURCES if floor else SOURCES
    if not force and up_to_date(lib, sources):
        return lib
    os.makedirs(BUILD, exist_ok=True)
    exe = nvcc()
    tag = f".{os.getpid()}"

    def compile_one(src: str) -> str:
        obj = os.path.join(BUILD, src.replace(".cu", tag + (".trace" if trace else "") + ".o"))
        cmd = [exe, *NVCC_FLAGS, *(["-DMOE_TAIL_TRACE"] if trace else []), "-c", os.path.join(CSRC, src), "-o", obj]
        if ptxas_v:
            cmd += ["-Xptxas", "-v"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose or ptxas_v:
            sys.stderr.write(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(sources)) as pool:
        objs = list(pool.map(compile_one, sources))
    tmp = lib + tag
    r = subprocess.run([exe, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    for o in objs:
        os.remove(o)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_v="-v" in sys.argv, trace="--trace" in sys.argv,
                floor="--floor" in sys.argv))
