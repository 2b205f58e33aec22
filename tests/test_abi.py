"""The C ABI without a GPU: the library loads, exports every function that
include/fs_sample.h declares, and rejects bad arguments on the host before
any device work (these calls return before touching CUDA)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fs_sample.h")


@pytest.fixture(scope="module")
def lib():
    from lm_head_gumbel_gb300 import build as libbuild
    try:
        libbuild.build()
    except RuntimeError as e:  # no nvcc on this machine
        pytest.skip(str(e))
    import lm_head_gumbel_gb300 as fs
    return fs.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fs_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_entry_points():
    names = declared_functions()
    for want in ("fs_sample", "fs_workspace_size", "fs_num_tiles", "fs_status_string",
                 "fs_gumbel_noise", "fs_last_device_error", "fs_group_merge", "fs_online_merge",
                 "fs_sample_noalloc", "fs_wait_timeout_selftest", "fs_sample_topk",
                 "fs_topk_workspace_size", "fs_sample_host"):
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_exports_are_c_symbols():
    """No C++ mangling on the entry points (checked with nm on the .so)."""
    import shutil
    import subprocess
    from lm_head_gumbel_gb300 import LIB_PATH
    if not shutil.which("nm") or not os.path.exists(LIB_PATH):
        pytest.skip("nm or library missing")
    out = subprocess.run(["nm", "-D", "--defined-only", LIB_PATH], capture_output=True,
                         text=True).stdout
    syms = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in declared_functions():
        assert name in syms, name


def test_host_helpers(lib):
    import lm_head_gumbel_gb300 as fs
    assert fs.fs_num_tiles(1) == 1
    assert fs.fs_num_tiles(128) == 1
    assert fs.fs_num_tiles(129) == 2
    assert fs.fs_num_tiles(151936) == 1187
    assert fs.fs_num_tiles(0) == 0
    assert fs.fs_workspace_size(4, 4096) == 512
    assert fs.fs_workspace_size(3, 129) == 512
    assert fs.fs_workspace_size(512, 151936) == 256 + 512 * 8
    assert fs.fs_workspace_size(65535, 151936) == ((256 + 65535 * 8 + 255) // 256) * 256
    assert fs.fs_workspace_size(0, 10) == 0
    for code, name in ((0, "FS_OK"), (1, "FS_ERR_INVALID_ARG"), (2, "FS_ERR_UNSUPPORTED"),
                       (3, "FS_ERR_CUDA"), (4, "FS_ERR_DEVICE_TIMEOUT"), (5, "FS_ERR_WORKSPACE")):
        assert fs.fs_status_string(code) == name
    assert fs.fs_status_string(99) == "FS_ERR_UNKNOWN"


def _args(**kw):
    import lm_head_gumbel_gb300 as fs
    base = dict(H=0x10000, W=0x20000, out_idx=0x30000, B=4, d=256, V=4096, ldh=256, ldw=256,
                out_tile_max=0x40000, out_tile_idx=0x50000)
    base.update(kw)
    return fs.FsSampleArgs(**base)


@pytest.mark.parametrize("kw,want", [
    (dict(H=None), 1), (dict(W=None), 1), (dict(out_idx=None, out_tile_max=None), 1),
    (dict(B=0), 1), (dict(B=65536), 1), (dict(d=0), 1), (dict(V=0), 1), (dict(V=2**31), 1),
    (dict(ldh=255), 1), (dict(ldh=260), 1), (dict(ldw=128), 1),
    (dict(H=0x10002), 1), (dict(W=0x20008), 1), (dict(out_idx=0x30004), 1),
    (dict(out_tile_idx=None), 1), (dict(out_tile_max=None), 1),
    (dict(vocab_mask=0x60000, mask_ld=127), 1),
    (dict(out_tile_lse=0x80000, out_tile_max=None, out_tile_idx=None), 1),
    (dict(vocab_offset=-4), 1), (dict(vocab_offset=6), 1), (dict(vocab_offset=2**31 - 4096), 1),
    (dict(out_max=0x90000, out_idx=None), 1), (dict(out_lse=0x90000), 1),
    (dict(B=65535, V=2**31 - 1, d=8, ldh=8, ldw=8), 1),  # work units beyond 32 bits
    (dict(flags=2), 1), (dict(flags=0x80000001), 1),  # unknown flag bits
    (dict(), 5),                                   # sampling without a workspace
    (dict(out_tile_max=None, out_tile_idx=None), 5),
    (dict(out_tile_max=None, out_tile_idx=None, workspace=0x70000, workspace_bytes=511), 5),
    (dict(out_tile_max=None, out_tile_idx=None, workspace=0x70080, workspace_bytes=4096), 5),
])
def test_bad_arguments_rejected_on_host(lib, kw, want):
    a = _args(**kw)
    assert lib.fs_sample(ctypes.byref(a), None) == want


def test_null_args_rejected(lib):
    assert lib.fs_sample(None, None) == 1


def test_transform_bad_arguments(lib):
    assert lib.fs_gumbel_transform(None, 5, ctypes.c_void_p(0x1000), None) == 1
    assert lib.fs_gumbel_transform(ctypes.c_void_p(0x1000), -1, ctypes.c_void_p(0x1000),
                                   None) == 1
    assert lib.fs_gumbel_transform(None, 0, None, None) == 0  # nothing to do


def test_noise_bad_arguments(lib):
    assert lib.fs_gumbel_noise(None, 0, 0, 0, 1, 0, 1, None, None) == 1
    assert lib.fs_gumbel_noise(None, 0, 0, -1, 1, 0, 1, ctypes.c_void_p(0x1000), None) == 1
    # an empty window is a no-op
    assert lib.fs_gumbel_noise(None, 0, 0, 0, 0, 0, 5, ctypes.c_void_p(0x1000), None) == 0


def test_package_fails_loudly_without_library(tmp_path):
    """With the library missing, the binding raises instead of falling back."""
    import lm_head_gumbel_gb300._binding as bnd
    saved = bnd._lib
    bnd._lib = None
    try:
        with pytest.raises(bnd.FsError):
            bnd.load_library(str(tmp_path / "missing.so"))
    finally:
        bnd._lib = saved


def test_merge_bad_arguments(lib):
    p = ctypes.c_void_p
    z, m, L, o = p(0x10000), p(0x20000), p(0x30000), p(0x40000)
    gm = lib.fs_group_merge
    assert gm(None, m, L, 2, 4, 0, None, 0, 0, o, None, None) == 1      # no z
    assert gm(z, m, L, 0, 4, 0, None, 0, 0, o, None, None) == 1         # P < 1
    assert gm(z, m, L, 2, 0, 0, None, 0, 0, o, None, None) == 1         # B < 1
    assert gm(z, None, L, 2, 4, 0, None, 0, 0, o, None, None) == 1      # exact needs m
    assert gm(z, m, None, 2, 4, 1, None, 0, 0, o, None, None) == 1      # group needs L
    assert gm(z, m, L, 2, 4, 7, None, 0, 0, o, None, None) == 1         # unknown mode
    assert gm(z, m, None, 2, 4, 0, None, 0, 0, o, p(0x50000), None) == 1  # out_L needs L
    assert gm(p(0x10004), m, L, 2, 4, 0, None, 0, 0, o, None, None) == 1  # misaligned z
    om = lib.fs_online_merge
    assert om(None, L, z, L, 4, 0, None, 0, 0, None) == 1
    assert om(z, L, z, L, 0, 0, None, 0, 0, None) == 1
    assert om(z, L, z, L, 4, 2**33, None, 0, 0, None) == 1


def test_topk_workspace_and_bad_arguments(lib):
    import lm_head_gumbel_gb300 as fs
    assert fs.fs_topk_workspace_size(4, 4096, 1) == 4 * 32 * 4 * 8
    assert fs.fs_topk_workspace_size(4, 4096, 5) == 4 * 32 * 16 * 8
    assert fs.fs_topk_workspace_size(4, 4096, 0) == 0
    assert fs.fs_topk_workspace_size(4, 4096, 17) == 0
    o = ctypes.c_void_p(0x90000)
    good = dict(out_tile_max=None, out_tile_idx=None, out_idx=None, workspace=0x100000,
                workspace_bytes=1 << 20)
    f = lib.fs_sample_topk
    assert f(ctypes.byref(_args(**good)), 0, o, None, None) == 1         # K < 1
    assert f(ctypes.byref(_args(**good)), 17, o, None, None) == 1        # K > max
    assert f(ctypes.byref(_args(**good)), 4, None, None, None) == 1      # no output
    assert f(ctypes.byref(_args(**dict(good, out_idx=0x30000))), 4, o, None, None) == 1
    assert f(ctypes.byref(_args(**dict(good, workspace_bytes=100))), 4, o, None, None) == 5
    assert f(ctypes.byref(_args(**dict(good, workspace=None))), 4, o, None, None) == 5
    assert f(None, 4, o, None, None) == 1


def test_host_step_bad_arguments(lib):
    """fs_sample_host checks its own buffers and every fs_sample argument
    before it enqueues anything (so these return without touching CUDA)."""
    p = ctypes.c_void_p
    hin, din, hout = p(0x1000), p(0x2000), p(0x3000)
    ws = dict(out_tile_max=None, out_tile_idx=None, workspace=0x70000, workspace_bytes=4096)
    f = lib.fs_sample_host
    assert f(None, hin, din, 64, hout, 1, None) == 1                               # no args
    assert f(ctypes.byref(_args(**ws)), hin, din, 64, None, 1, None) == 1          # no host_out
    assert f(ctypes.byref(_args(**dict(ws, out_idx=None))), hin, din, 64, hout, 1, None) == 1
    assert f(ctypes.byref(_args(**ws)), None, din, 64, hout, 1, None) == 1         # no host_in
    assert f(ctypes.byref(_args(**ws)), hin, None, 64, hout, 1, None) == 1         # no dev_in
    assert f(ctypes.byref(_args(**dict(ws, B=0))), hin, din, 64, hout, 1, None) == 1
    assert f(ctypes.byref(_args(**dict(ws, workspace=None))), hin, din, 64, hout, 1, None) == 5
    assert f(ctypes.byref(_args(**ws)), hin, din, 64, hout, 3, None) == 1          # bad sync
    assert f(ctypes.byref(_args(**ws)), hin, din, 64, hout, -1, None) == 1


def test_struct_layout_matches_the_header(tmp_path):
    """The ctypes mirror of fs_sample_args has the C compiler's size and
    field offsets (a C program built against the header prints them)."""
    import shutil
    import subprocess
    import lm_head_gumbel_gb300 as fs
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    names = [f[0] for f in fs.FsSampleArgs._fields_]
    src = tmp_path / "layout.c"
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "fs_sample.h"',
             "int main(void) {", '  printf("size %zu\\n", sizeof(fs_sample_args));']
    lines += [f'  printf("{n} %zu\\n", offsetof(fs_sample_args, {n}));' for n in names]
    lines += ['  printf("flag %u\\n", (unsigned)FS_FLAG_OVERLAP_PREVIOUS);', "  return 0;", "}"]
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-std=c99", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True)
    out = dict(line.split() for line in subprocess.run([str(exe)], capture_output=True, text=True,
                                                       check=True).stdout.splitlines())
    assert int(out.pop("size")) == ctypes.sizeof(fs.FsSampleArgs)
    assert int(out.pop("flag")) == fs.FS_FLAG_OVERLAP_PREVIOUS
    for n in names:
        assert int(out[n]) == getattr(fs.FsSampleArgs, n).offset, n
