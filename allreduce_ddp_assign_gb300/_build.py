"""Build libddpbucket.so in-tree with nvcc (sm_103a only).

Each translation unit compiles in its own nvcc process (in parallel), then one
link with the shared CUDA runtime so the library and PyTorch use the same
runtime instance.  Rebuilds only when a source or the header is newer than the
library.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUTDIR = os.path.join(PKG, "_lib")
LIB = os.path.join(OUTDIR, "libddpbucket.so")
SOURCES = ["kernels.cu", "stream_ring.cu", "stream_fused.cu", "stream_fused_wire.cu", "stream_pack.cu", "bitmap.cu",
           "powersgd.cu", "reducer.cpp", "assign.cpp", "plan.cpp", "timeline.cpp", "status.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libddpbucket")
    return path


def _inputs() -> list[str]:
    files = [os.path.join(CSRC, s) for s in SOURCES] + [os.path.join(CSRC, "common.h"),
                                                        os.path.join(CSRC, "device_common.cuh"),
                                                        os.path.join(CSRC, "stream_impl.cuh"),
                                                        os.path.join(INCLUDE, "ddp_bucket.h")]
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False, extra: tuple = (), out: str | None = None) -> str:
    """Compile and link; `extra` adds nvcc flags (e.g. -D tunables) and `out` names
    another library path (the objects then go beside it)."""
    lib = out or LIB
    if not force and not extra and out is None and up_to_date():
        return LIB
    outdir = os.path.dirname(lib)
    os.makedirs(outdir, exist_ok=True)
    cc = nvcc()
    common = ["-std=c++17", "-O3", "-I", INCLUDE, "-Xcompiler", "-fPIC", "--cudart", "shared", *extra]

    def compile_one(src: str) -> str:
        obj = os.path.join(outdir, os.path.basename(src) + ".o")
        cmd = [cc, *common, "-c", os.path.join(CSRC, src), "-o", obj]
        if src.endswith(".cu"):
            cmd[1:1] = [*ARCH, "-lineinfo"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout, r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [cc, "-shared", *ARCH, "--cudart", "shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force=True, verbose=True))
