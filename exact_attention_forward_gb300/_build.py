"""Compile the CUDA library (sm_103a) in-tree with nvcc.

One translation unit per kernel instance plus the host API, compiled in
parallel, linked into ``_fa_gb300.so`` next to this file (cudart linked
statically; the driver API is reached through cudaGetDriverEntryPoint, so the
library has no load-time dependency on libcuda).
"""
from __future__ import annotations

import concurrent.futures as cf
import fcntl
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(HERE, "_fa_gb300.so")
# throughput probes of the ex2 unit and the tensor pipe (measurement only; not the product path)
MB_SRC = os.path.join(CSRC, "microbench", "fa_microbench.cu")
MB_LIB = os.path.join(HERE, "_fa_microbench.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["fa_api.cu", "fa_fwd_bf16_d64.cu", "fa_fwd_bf16_d128.cu", "fa_fwd_e4m3_d128.cu",
           "fa_fwd_pair_bf16_d128.cu", "fa_static_ws.cu", "fa_append_kv.cu"]


def _nvcc():
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return cand


def _deps():
    return [os.path.join(CSRC, f) for f in os.listdir(CSRC)
            if os.path.isfile(os.path.join(CSRC, f))] + [os.path.join(ROOT, "include", "fa.h")]


def build_microbench(force: bool = False) -> str:
    """Build _fa_microbench.so (one translation unit) next to the main library."""
    deps = [MB_SRC, os.path.join(CSRC, "sm103_ptx.cuh"),
            os.path.join(ROOT, "include", "fa_microbench.h")]
    if (not force and os.path.exists(MB_LIB)
            and os.path.getmtime(MB_LIB) >= max(os.path.getmtime(d) for d in deps)):
        return MB_LIB
    os.makedirs(BUILD, exist_ok=True)
    with open(os.path.join(BUILD, ".lock_mb"), "w") as lock:
        fcntl.flock(lock, fcntl.LOCK_EX)
        tmp = MB_LIB + f".tmp{os.getpid()}"
        cmd = [_nvcc()] + ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                                  "-Xcompiler", "-fvisibility=hidden", "-I",
                                  os.path.join(ROOT, "include"), "-shared", MB_SRC, "-o", tmp]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {MB_SRC}:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, MB_LIB)
    return MB_LIB


def build(force: bool = False, verbose: bool = False, extra_flags=(), lib_path: str = LIB,
          build_dir: str = BUILD) -> str:
    """Build the library; `extra_flags` / `lib_path` / `build_dir` make a variant build
    (e.g. a compile-time option) elsewhere without touching the default library.
    Concurrent callers (parallel test workers) serialise on a lock file in build_dir."""
    def fresh():
        return (os.path.exists(lib_path)
                and os.path.getmtime(lib_path) >= max(os.path.getmtime(d) for d in _deps()))

    if not force and fresh():
        return lib_path
    os.makedirs(build_dir, exist_ok=True)
    with open(os.path.join(build_dir, ".lock"), "w") as lock:
        fcntl.flock(lock, fcntl.LOCK_EX)
        if not force and fresh():  # another process built it meanwhile
            return lib_path
        return _build_locked(verbose, extra_flags, lib_path, build_dir)


def _build_locked(verbose, extra_flags, lib_path, build_dir) -> str:
    nvcc = _nvcc()
    common = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-Xcompiler", "-fvisibility=hidden",
                     "-I", os.path.join(ROOT, "include"), "-I", CSRC] + list(extra_flags)
    if verbose:
        common += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc] + common + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose:
        for _, log in results:
            print(log)
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    import sys
    print(build(force=True, verbose="-v" in sys.argv))
