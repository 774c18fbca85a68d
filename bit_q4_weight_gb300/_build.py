"""Build libjllm_q4k.so (the C-ABI CUDA library) in-tree with nvcc for sm_103a.

Each .cu file is compiled to an object in parallel, then linked into one
shared library with the CUDA runtime linked statically, so the library needs
nothing but the NVIDIA driver at run time.
"""
from __future__ import annotations

import concurrent.futures as cf
import fcntl
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libjllm_q4k.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
          "-I", os.path.join(ROOT, "include")]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libjllm_q4k.so")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _newest_input() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(ROOT, "include", "jllm_q4k.h")]
    return max(os.path.getmtime(f) for f in files)


def _up_to_date(lib: str) -> bool:
    return os.path.exists(lib) and os.path.getmtime(lib) >= _newest_input()


def build(force: bool = False, verbose: bool = False, extra: list[str] | None = None, variant: str = "") -> str:
    """Compile the library if it is missing or older than its sources; return its path.
    Processes that build at the same time (the ranks of one job) take turns on a lock
    file, and a process that waited finds the library already built.

    variant: a named build with extra compiler flags (`extra`), kept apart from the
    shipped library (its objects in _build_<variant>/, the library in
    libjllm_q4k_<variant>.so); the tests use one with -DJLLM_FAULT_INJECTION."""
    lib = LIB if not variant else os.path.join(PKG, f"libjllm_q4k_{variant}.so")
    bdir = BUILD if not variant else os.path.join(PKG, f"_build_{variant}")
    if not force and _up_to_date(lib):
        return lib
    os.makedirs(bdir, exist_ok=True)
    with open(os.path.join(bdir, ".lock"), "w") as lock:
        fcntl.flock(lock, fcntl.LOCK_EX)
        if not force and _up_to_date(lib):
            return lib
        return _build_locked(verbose, extra, lib, bdir)


def _build_locked(verbose: bool, extra: list[str] | None, lib: str, bdir: str) -> str:
    nvcc = _nvcc()
    flags = ARCH + CFLAGS + (extra or [])

    def compile_one(src: str) -> str:
        obj = os.path.join(bdir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *flags, "-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{res.stdout}\n{res.stderr}")
        if verbose and res.stderr:
            print(res.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp = lib + f".tmp{os.getpid()}"
    res = subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, lib)
    return lib


def build_microbench() -> str:
    """Compile microbench/tc_rates.cu (tensor-core rate measurements, not part of the library)
    into its own shared object; return its path."""
    src = os.path.join(PKG, "microbench", "tc_rates.cu")
    lib = os.path.join(PKG, "microbench", "libjllm_microbench.so")
    if os.path.exists(lib) and os.path.getmtime(lib) >= max(os.path.getmtime(src), _newest_input()):
        return lib
    tmp = lib + f".tmp{os.getpid()}"
    res = subprocess.run([_nvcc(), *ARCH, *CFLAGS, "-shared", src, "-o", tmp], capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys

    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
