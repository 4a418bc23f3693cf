"""Build libkvc8.so in-tree with nvcc for sm_103a (GB300).

Each .cu file compiles to an object in parallel; the objects link into
``dequant_kvc8_store_gb300/_build/libkvc8.so`` with the CUDA runtime linked
statically.  No fast-math: the kernels rely on IEEE division, multiplication
and round-to-nearest-even conversions being exact.
"""
from __future__ import annotations

import fcntl
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(OUT_DIR, "libkvc8.so")
SOURCES = ["kvc8_api.cu", "kvc8_store.cu", "kvc8_gather.cu", "kvc8_noalloc.cu", "kvc8_bf16.cu",
           "kvc8_attention.cu"]
HEADERS = [os.path.join(CSRC, "kvc8_internal.cuh"), os.path.join(INCLUDE, "kvc8.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libkvc8")


def _stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    deps = [os.path.join(CSRC, s) for s in SOURCES] + HEADERS + [os.path.abspath(__file__)]
    return any(os.path.getmtime(p) > t for p in deps)


def build(force: bool = False, verbose: bool = False, csrc: str = CSRC, out_dir: str = OUT_DIR) -> str:
    """Compile (if stale) and return the path of libkvc8.so (csrc / out_dir: a
    source tree and output folder other than the package's own)."""
    lib_path = os.path.join(out_dir, "libkvc8.so")
    if not force and csrc == CSRC and not _stale():
        return LIB_PATH
    os.makedirs(out_dir, exist_ok=True)
    # one build at a time per output folder (parallel test workers may all
    # find the library stale); the first one builds, the others reuse it
    with open(os.path.join(out_dir, ".lock"), "w") as lock:
        fcntl.flock(lock, fcntl.LOCK_EX)
        if not force and csrc == CSRC and not _stale():
            return LIB_PATH
        return _build_locked(csrc, out_dir, lib_path, verbose)


def _build_locked(csrc: str, out_dir: str, lib_path: str, verbose: bool) -> str:
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(out_dir, os.path.splitext(src)[0] + ".o")
        cmd = [cc, *ARCH, *NVCC_FLAGS, "-I", csrc, "-c", os.path.join(csrc, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
