"""fs_sample_noalloc: the entry point for callers that cannot allocate device
memory (for example a sampler plugged into an engine that owns the whole
device through its own memory pool and offers plugins no allocator).  It must
give what fs_sample gives, using the library's built-in scratch array instead
of a caller workspace.

This file is collected last on purpose, and its test must pass both alone in
a fresh process and after every other test."""
import ctypes
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest
import torch

import lm_head_gumbel_gb300 as fs
from lm_head_gumbel_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

NOALLOC_SCRATCH_BYTES = 64 << 10


def _args(H, W, T, seeds, mask, out_idx, ws, offset):
    B, d = H.shape
    V = W.shape[0]
    return fs.FsSampleArgs(
        H=H.data_ptr(), W=W.data_ptr(), temperature=T.data_ptr(), vocab_mask=mask.data_ptr(),
        mask_ld=mask.stride(0), seeds=seeds.data_ptr(), seed=0, offset=offset, B=B, d=d, V=V,
        ldh=H.stride(0), ldw=W.stride(0), out_idx=out_idx.data_ptr(),
        workspace=None if ws is None else ws.data_ptr(),
        workspace_bytes=0 if ws is None else ws.numel())


def test_noalloc_matches_fs_sample_twice_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = fs.load_library()
    B, d, V = 37, 320, 5000
    W = wl.make_weights(d, V, seed=501, device="cuda")
    H = wl.make_hidden(B, d, seed=502, device="cuda")
    T = wl.make_temperature(wl.WORKLOADS["qwen3-8b"], B, seed=503, device="cuda")
    seeds = wl.make_seeds(B, base=504, device="cuda")
    mask = wl.make_mask(B, V, 0.05, seed=505, device="cuda")
    stream = torch.cuda.current_stream()
    ws = torch.zeros(fs.fs_workspace_size(B, V), dtype=torch.uint8, device="cuda")
    for offset in (11, 12):
        want = torch.full((B,), -7, dtype=torch.int64, device="cuda")
        a = _args(H, W, T, seeds, mask, want, ws, offset)
        assert lib.fs_sample(ctypes.byref(a), ctypes.c_void_p(stream.cuda_stream)) == fs.FS_OK
        for _call in range(2):  # two calls in a row share the scratch array
            got = torch.full((B,), -7, dtype=torch.int64, device="cuda")
            a2 = _args(H, W, T, seeds, mask, got, None, offset)
            st = lib.fs_sample_noalloc(ctypes.byref(a2), ctypes.c_void_p(stream.cuda_stream))
            assert st == fs.FS_OK, fs.fs_status_string(st)
            torch.cuda.synchronize()
            assert np.array_equal(got.cpu().numpy(), want.cpu().numpy())
    st, code = fs.fs_last_device_error()
    assert st == fs.FS_OK and code == 0


def test_noalloc_rejects_problems_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = fs.load_library()
    B, V = 16384, 262144  # workspace 256 + 8 B = 128.25 KiB > 64 KiB
    assert fs.fs_workspace_size(B, V) > NOALLOC_SCRATCH_BYTES
    dummy = torch.empty(8, dtype=torch.int64, device="cuda")
    a = fs.FsSampleArgs(H=dummy.data_ptr(), W=dummy.data_ptr(), out_idx=dummy.data_ptr(),
                        B=B, d=8, V=V, ldh=8, ldw=8)
    assert lib.fs_sample_noalloc(ctypes.byref(a), None) == fs.FS_ERR_WORKSPACE


# Run as a fresh process: its first library call is fs_sample_noalloc, on a
# stream created by torch (non-blocking with respect to the legacy default
# stream), while the legacy default stream is kept busy.  The one-time clear
# of the scratch array must be ordered before that first kernel on the
# caller's own stream; a clear queued behind the busy default stream would
# land in the middle of the sampling kernel and erase row maxima.
_FIRST_CALL_ON_A_SIDE_STREAM = textwrap.dedent("""
    import ctypes, sys
    import numpy as np
    import torch
    sys.path.insert(0, sys.argv[1])
    import lm_head_gumbel_gb300 as fs
    from lm_head_gumbel_gb300 import workloads as wl

    lib = fs.load_library()
    B, d, V = 8160, 1024, 262144       # the largest batch the scratch array holds
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        W = wl.make_weights(d, V, seed=601, device="cuda")
        H = wl.make_hidden(B, d, seed=602, device="cuda")
        T = torch.full((B,), 0.8, dtype=torch.float32, device="cuda")
        got = torch.full((B,), -7, dtype=torch.int64, device="cuda")
        again = torch.full((B,), -7, dtype=torch.int64, device="cuda")
        want = torch.full((B,), -7, dtype=torch.int64, device="cuda")
        ws = torch.zeros(fs.fs_workspace_size(B, V), dtype=torch.uint8, device="cuda")
    side.synchronize()
    torch.cuda.synchronize()

    def args(out, workspace):
        return fs.FsSampleArgs(H=H.data_ptr(), W=W.data_ptr(), temperature=T.data_ptr(),
                               seed=77, offset=5, B=B, d=d, V=V, ldh=d, ldw=d,
                               out_idx=out.data_ptr(),
                               workspace=None if workspace is None else workspace.data_ptr(),
                               workspace_bytes=0 if workspace is None else workspace.numel())

    h = ctypes.c_void_p(side.cuda_stream)
    torch.cuda._sleep(4_000_000)       # the legacy default stream: about 2 ms busy
    a = args(got, None)
    assert lib.fs_sample_noalloc(ctypes.byref(a), h) == fs.FS_OK
    b = args(want, ws)
    assert lib.fs_sample(ctypes.byref(b), h) == fs.FS_OK
    c = args(again, None)
    assert lib.fs_sample_noalloc(ctypes.byref(c), h) == fs.FS_OK
    side.synchronize()
    torch.cuda.synchronize()
    g, w, r = got.cpu().numpy(), want.cpu().numpy(), again.cpu().numpy()
    assert np.all(w >= 0) and np.all(w < V)
    assert np.array_equal(g, w), int(np.sum(g != w))
    assert np.array_equal(r, w), int(np.sum(r != w))
    print("NOALLOC_SIDE_STREAM_OK")
""")


def test_noalloc_first_call_on_a_non_blocking_stream():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fs.load_library()  # the library must exist before the child runs
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _FIRST_CALL_ON_A_SIDE_STREAM, root],
                       capture_output=True, text=True, timeout=600, cwd=root)
    assert r.returncode == 0 and "NOALLOC_SIDE_STREAM_OK" in r.stdout, (r.stdout, r.stderr[-3000:])
