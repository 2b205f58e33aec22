"""The C ABI from a C program: tests/c_abi_example.c is compiled with gcc
against include/fs_sample.h and libfs.so (no Python on its side), and run on
the GPU; without a GPU it is only compiled and linked."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_abi_example.c")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def build_example(out_dir):
    from lm_head_gumbel_gb300 import build as libbuild
    try:
        lib = libbuild.build()
    except RuntimeError as e:  # no nvcc on this machine
        pytest.skip(str(e))
    if not shutil.which("gcc"):
        pytest.skip("gcc missing")
    libdir = os.path.dirname(lib)
    exe = os.path.join(str(out_dir), "c_abi_example")
    cmd = ["gcc", "-std=c99", "-O1", "-Wall", "-Werror", f"-I{ROOT}/include",
           f"-I{CUDA}/include", SRC, "-o", exe, f"-L{libdir}", "-lfs",
           f"-L{CUDA}/lib64", "-lcudart", f"-Wl,-rpath,{libdir}:{CUDA}/lib64", "-lm"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    return exe


def test_c_example_compiles_and_links(tmp_path):
    assert os.path.exists(build_example(tmp_path))


@pytest.mark.gpu
def test_c_example_runs(tmp_path):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    exe = build_example(tmp_path)
    res = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert res.returncode == 0, res.stdout + res.stderr
    assert res.stdout.strip() == "ok"
