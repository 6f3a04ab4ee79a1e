"""Compile the CUDA sources under csrc/ into the in-tree shared library libgla.so.

Only sm_103a code is generated (one -gencode).  The translation units are
compiled in parallel and linked with the static CUDA runtime, so the library
depends on nothing but the driver at run time.
"""
from __future__ import annotations

import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libgla.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

SOURCES = ["gla_api.cu", "gla_simt.cu", "gla_decode.cu", "gla_tc.cu", "gla_short.cu", "gla_delta.cu", "gla_bwd.cu",
           "gla_bwd_tc.cu", "gla_delta_tc.cu"]
HEADERS = ["gla_internal.h", "gla_ptx.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-Xptxas", "-v"] + ARCH


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=None) -> str:
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    hdrs = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, "gla.h")]
    flags = NVCC_FLAGS + list(extra_flags or [])
    objs = []
    jobs = []
    for src in SOURCES:
        sp = os.path.join(CSRC, src)
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        objs.append(obj)
        if force or _stale(obj, [sp] + hdrs):
            jobs.append((sp, obj))

    def compile_one(job):
        sp, obj = job
        cmd = [nvcc] + flags + ["-I", INCLUDE, "-c", sp, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {os.path.basename(sp)}:\n{r.stderr}")
        return os.path.basename(sp), r.stderr

    if jobs:
        with ThreadPoolExecutor(max_workers=len(jobs)) as ex:
            for name, log in ex.map(compile_one, jobs):
                if verbose:
                    print(f"--- {name}\n{log}")
    if force or jobs or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True))
