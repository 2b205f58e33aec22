"""fs_sample_noalloc: the entry point for callers that cannot allocate device
memory (for example a sampler plugged into an engine that owns the whole
device through its own memory pool and offers plugins no allocator).  It must
give what fs_sample gives, using the library's built-in scratch array instead
of a caller workspace.

This file is collected last on purpose, and its test must pass both alone in
a fresh process and after every other test."""
import ctypes

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
