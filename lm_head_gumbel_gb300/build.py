"""Build the CUDA library ``libfs.so`` in-tree with nvcc, for sm_103a only."""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIBRARY = os.path.join(PKG, "libfs.so")
SOURCES = [os.path.join(CSRC, "fs_sample.cu"), os.path.join(CSRC, "fs_merge.cu")]
DEPENDS = SOURCES + [os.path.join(CSRC, f) for f in ("fs_kernels.cuh", "fs_ptx.cuh",
                                                    "fs_noise.cuh")] + [
    os.path.join(INCLUDE, "fs_sample.h")]

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfs.so")
    return cand


def command(output: str = LIBRARY, extra=()) -> list:
    return [nvcc_path(), *ARCH_FLAGS, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
            "-shared", f"-I{INCLUDE}", *extra, "-o", output, *SOURCES]


def up_to_date(output: str = LIBRARY) -> bool:
    if not os.path.exists(output):
        return False
    t = os.path.getmtime(output)
    return all(os.path.getmtime(f) <= t for f in DEPENDS)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libfs.so unless it is newer than every source it depends on."""
    if not force and up_to_date():
        return LIBRARY
    tmp = LIBRARY + f".tmp{os.getpid()}"
    cmd = command(tmp, ["-Xptxas", "-v"] if verbose else [])
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"libfs.so build failed:\n{' '.join(cmd)}\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, LIBRARY)
    if verbose:
        print(res.stderr)
    return LIBRARY


if __name__ == "__main__":
    print(build(force=True, verbose=True))
