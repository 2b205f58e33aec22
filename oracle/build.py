"""Compile the CPU oracle (``fs_oracle.c``) into a shared library.

Test infrastructure: building the checker is not using it.  The library is
written to ``oracle/_build/`` (git-ignored).  ``gcc`` with OpenMP is used when
available; without ``-fopenmp`` support the oracle still builds and runs on one
thread.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "fs_oracle.c")
BUILD_DIR = os.path.join(HERE, "_build")
LIBRARY = os.path.join(BUILD_DIR, "libfs_oracle.so")


def compile_source(source: str, output: str, openmp: bool = True) -> None:
    """Compile one oracle source file into ``output`` (a shared library).

    IEEE semantics are kept (no fast-math), so sums run in index order."""
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        raise RuntimeError("no C compiler (gcc/cc) found to build the oracle")
    os.makedirs(os.path.dirname(output), exist_ok=True)
    base = [cc, "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
            "-ffp-contract=off"]
    tmp = output + f".tmp{os.getpid()}"
    cmd = base + (["-fopenmp"] if openmp else []) + [source, "-o", tmp, "-lm"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0 and openmp:
        cmd = base + [source, "-o", tmp, "-lm"]
        res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"oracle build failed:\n{' '.join(cmd)}\n{res.stderr}")
    os.replace(tmp, output)


def build(force: bool = False) -> str:
    """Build ``libfs_oracle.so`` if missing or older than its source."""
    if (force or not os.path.exists(LIBRARY)
            or os.path.getmtime(LIBRARY) < os.path.getmtime(SOURCE)):
        compile_source(SOURCE, LIBRARY)
    return LIBRARY


def build_variant(source_text: str, name: str, directory: str | None = None) -> str:
    """Compile a modified copy of the oracle source (used by the tests that
    plant a mistake in the oracle to show that the pins catch it)."""
    directory = directory or tempfile.mkdtemp(prefix="fs_oracle_variant_")
    src = os.path.join(directory, f"{name}.c")
    with open(src, "w") as f:
        f.write(source_text)
    out = os.path.join(directory, f"lib{name}.so")
    compile_source(src, out)
    return out


if __name__ == "__main__":
    print(build(force=True))
