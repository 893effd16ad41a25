"""Build libcdg.so (the sm_103a dgrad library) in-tree with nvcc.

    python -m implicit_gemm_dgrad_gb300.build [--force]

Seven translation units compiled in parallel (the dgrad and wgrad host APIs,
the plain, per-channel-sum and activation variants of the dgrad kernels, the
other dgrad kernels, the wgrad kernels), then linked
into a shared library next to this file.  The CUDA runtime is linked
statically; the driver API is reached through cudaGetDriverEntryPointByVersion.
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
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(HERE, "libcdg.so")
BUILD_DIR = os.path.join(HERE, "_build")
SOURCES = ["cdg_api.cu", "cwg_api.cu", "dgrad_sm103.cu", "dgrad_plain_sm103.cu", "dgrad_ext_sm103.cu",
           "dgrad_act_sm103.cu", "wgrad_sm103.cu"]
HEADERS = ["cdg_params.h", "cwg_params.h", "ptx.cuh", "wait.cuh", "dgrad_device.cuh", "dgrad_variant.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES + HEADERS]
    files.append(os.path.join(INCLUDE, "cdg.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD_DIR, exist_ok=True)
    common = [nvcc(), "-O3", "-std=c++17", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC",
              "-I", INCLUDE, "-I", CSRC, *extra_flags]
    if verbose:
        common += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(BUILD_DIR, os.path.splitext(src)[0] + ".o")
        cmd = common + ["-c", os.path.join(CSRC, src), "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, res

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    for src, _, res in results:
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
        if verbose and (res.stdout or res.stderr):
            sys.stderr.write(res.stdout + res.stderr)
    tmp = LIB + f".tmp{os.getpid()}"
    link = [nvcc(), *ARCH, "-shared", "-o", tmp] + [obj for _, obj, _ in results]
    res = subprocess.run(link, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB)
