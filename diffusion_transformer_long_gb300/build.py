"""Builds libditattn.so in-tree for sm_103a with nvcc (no cmake, no setuptools).

The translation units compile in parallel, then link into one shared library
that depends on the shared CUDA runtime (libcudart.so.13), so the library and
PyTorch share one runtime instance in a process.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(PKG, "libditattn.so")
SOURCES = ["attn_fwd.cu", "attn_fwd_short.cu", "lse_merge.cu", "layout_copy.cu", "noalloc.cu", "ditattn_api.cu"]
HEADERS = ["attn_kernel.cuh", "attn_host.cuh", "merge_math.cuh", "sm103_ptx.cuh", "launch.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def cuda_home() -> str:
    home = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH")
    if home and os.path.exists(os.path.join(home, "bin", "nvcc")):
        return home
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return "/usr/local/cuda"


def _newest_input() -> float:
    files = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    files.append(os.path.join(PKG, "..", "include", "ditattn.h"))
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile (if stale) and return the path of libditattn.so."""
    if not force and os.path.exists(LIB_PATH) and os.path.getmtime(LIB_PATH) >= _newest_input():
        return LIB_PATH
    home = cuda_home()
    nvcc = os.path.join(home, "bin", "nvcc")
    os.makedirs(BUILD_DIR, exist_ok=True)
    common = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                     "-cudart", "shared", "-I", CSRC, "-I", os.path.join(PKG, "..", "include")]
    if verbose:
        common += ["-Xptxas", "-v"]

    def compile_one(src: str) -> tuple[str, str]:
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        r = subprocess.run([nvcc, *common, "-c", os.path.join(CSRC, src), "-o", obj],
                           capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    libdir = os.path.join(home, "lib64")
    r = subprocess.run([nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp,
                        *[o for o, _ in results], "-Xlinker", f"-rpath,{libdir}"],
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
