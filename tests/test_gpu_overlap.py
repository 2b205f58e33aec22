"""FS_FLAG_OVERLAP_PREVIOUS: a call launched as a programmatic dependent of
the stream's previous kernel gives bit-identical results to a plain call.
The hazards it must respect are exercised directly: back-to-back calls that
share one workspace (the next call's row maxima must not mix with the
previous call's), and a preceding kernel that writes H last."""
import numpy as np
import pytest
import torch

import lm_head_gumbel_gb300 as fs
from gpu_cases import assert_no_device_error, compare, make_problem

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fs.load_library()
    yield
    assert_no_device_error()


def _outputs(B, V, dev, lse):
    nt = fs.fs_num_tiles(V)
    o = {"tile_max": torch.empty((B, nt), dtype=torch.float32, device=dev),
         "tile_idx": torch.empty((B, nt), dtype=torch.int32, device=dev),
         "idx": torch.empty(B, dtype=torch.int64, device=dev)}
    if lse:
        o["tile_lse"] = torch.empty((B, nt), dtype=torch.float32, device=dev)
    return o


def _call(p, o, ws, offset, overlap):
    fs.fs_sample(p["H"], p["W"], temperature=p["temperature"], seeds=p["seeds"],
                 vocab_mask=p["vocab_mask"], seed=3, offset=offset, out_idx=o["idx"],
                 out_tile_max=o["tile_max"], out_tile_idx=o["tile_idx"],
                 out_tile_lse=o.get("tile_lse"), workspace=ws, overlap_previous=overlap)


@pytest.mark.parametrize("B,lse", [(64, False), (256, True), (384, False)])
def test_back_to_back_calls_share_a_workspace(B, lse):
    """20 chained calls, each overlapping the one before and reusing its
    workspace: every call equals the plain call with the same offset.  B = 64
    runs the single-CTA kernel, B = 256 the CTA pairs, B = 384 three batch
    blocks of single CTAs."""
    p = make_problem(B, 512, 30000, T="row-uniform", per_row_seeds=True, mask_frac=0.05,
                     seed=31)
    dev = p["H"].device
    ws = torch.zeros(fs.fs_workspace_size(B, 30000), dtype=torch.uint8, device=dev)
    want = []
    for k in range(20):
        o = _outputs(B, 30000, dev, lse)
        _call(p, o, ws, k, overlap=False)
        torch.cuda.synchronize()
        want.append({n: t.cpu() for n, t in o.items()})
    got = [_outputs(B, 30000, dev, lse) for _ in range(20)]
    for k in range(20):
        _call(p, got[k], ws, k, overlap=True)
    torch.cuda.synchronize()
    for k in range(20):
        for n in want[k]:
            assert torch.equal(got[k][n].cpu(), want[k][n]), (k, n)
    assert not torch.equal(want[0]["idx"], want[1]["idx"])


def test_kernel_that_writes_h_just_before():
    """The preceding kernel writes H as the last rows of a 96 MB buffer: the
    overlapped call must read the new H, not what was there before."""
    B, d, V = 64, 1024, 20000
    p = make_problem(B, d, V, T=1.0, seed=32)
    dev = p["H"].device
    rows = (96 << 20) // (2 * d)
    src = torch.randn(rows, d, device=dev).to(torch.bfloat16)
    src[-B:] = p["H"]
    buf = torch.zeros_like(src)
    H = buf[-B:]  # contiguous rows, 16-byte aligned
    ws = torch.zeros(fs.fs_workspace_size(B, V), dtype=torch.uint8, device=dev)
    ref = fs.fs_sample(p["H"], p["W"], temperature=p["temperature"], seed=9, offset=4,
                       workspace=ws).cpu()
    for it in range(10):
        buf.zero_()
        torch.cuda.synchronize()
        torch.mul(src, 1.0, out=buf)  # H's rows are written last
        out = fs.fs_sample(H, p["W"], temperature=p["temperature"], seed=9, offset=4,
                           workspace=ws, overlap_previous=True)
        assert torch.equal(out.cpu(), ref), it


def test_overlapped_call_matches_oracle():
    p = make_problem(40, 256, 9000, T=0.9, greedy_frac=0.1, seed=33)
    dev = p["H"].device
    ws = torch.zeros(fs.fs_workspace_size(40, 9000), dtype=torch.uint8, device=dev)
    o = _outputs(40, 9000, dev, lse=True)
    _call(p, o, ws, 0, overlap=False)  # something to overlap
    _call(p, o, ws, 5, overlap=True)
    torch.cuda.synchronize()
    dev_out = {k: v.cpu().numpy() for k, v in o.items()}
    st = compare(p, dev_out, seed=3, offset=5, scores=True)  # raises on a mismatch
    assert st["rows"] == 40 and st["tiles"] > 0


def test_topk_overlapped_matches_plain():
    B, V, K = 96, 12000, 8
    p = make_problem(B, 256, V, T=1.0, seed=34)
    dev = p["H"].device
    ws = torch.empty(fs.fs_topk_workspace_size(B, V, K), dtype=torch.uint8, device=dev)
    want = fs.fs_sample_topk(p["H"], p["W"], K, seed=2, offset=1, workspace=ws).cpu()
    outs = [torch.empty((B, K), dtype=torch.int64, device=dev) for _ in range(5)]
    for o in outs:
        fs.fs_sample_topk(p["H"], p["W"], K, seed=2, offset=1, workspace=ws, out_topk_idx=o,
                          overlap_previous=True)
    torch.cuda.synchronize()
    for o in outs:
        assert torch.equal(o.cpu(), want)


def test_overlapped_chain_in_a_cuda_graph():
    """Chained overlapped calls captured in a graph (programmatic edges) and
    replayed give the eager plain results."""
    B, V = 128, 16000
    p = make_problem(B, 384, V, T="row-uniform", seed=35)
    dev = p["H"].device
    ws = torch.zeros(fs.fs_workspace_size(B, V), dtype=torch.uint8, device=dev)
    want = [fs.fs_sample(p["H"], p["W"], temperature=p["temperature"], seed=1, offset=k,
                         workspace=ws).cpu() for k in range(4)]
    outs = [torch.empty(B, dtype=torch.int64, device=dev) for _ in range(4)]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for k in range(4):
                fs.fs_sample(p["H"], p["W"], temperature=p["temperature"], seed=1, offset=k,
                             out_idx=outs[k], workspace=ws, overlap_previous=k > 0, stream=s)
    for _ in range(3):
        for o in outs:
            o.fill_(-7)
        g.replay()
        torch.cuda.synchronize()
        for k in range(4):
            assert torch.equal(outs[k].cpu(), want[k]), k


def test_host_step_with_the_flag():
    """fs_sample_host with inputs already on the device (in_bytes = 0) and the
    flag: the sampling kernel overlaps the kernel before it (here the one that
    wrote H), and the ids equal the plain device call's."""
    import ctypes
    B, V = 32, 20000
    p = make_problem(B, 512, V, T=1.0, per_row_seeds=True, seed=36)
    dev = p["H"].device
    ws = torch.zeros(fs.fs_workspace_size(B, V), dtype=torch.uint8, device=dev)
    want = fs.fs_sample(p["H"], p["W"], temperature=p["temperature"], seeds=p["seeds"], offset=2,
                        workspace=ws).cpu()
    H = torch.empty_like(p["H"])
    out = torch.empty(B, dtype=torch.int64, device=dev)
    host_out = torch.empty(B, dtype=torch.int64).pin_memory()
    args = fs.FsSampleArgs(H=H.data_ptr(), W=p["W"].data_ptr(),
                           temperature=p["temperature"].data_ptr(), seeds=p["seeds"].data_ptr(),
                           offset=2, B=B, d=512, V=V, ldh=512, ldw=512, out_idx=out.data_ptr(),
                           workspace=ws.data_ptr(), workspace_bytes=ws.numel(),
                           flags=fs.FS_FLAG_OVERLAP_PREVIOUS)
    for sync in (fs.FS_SYNC_STREAM, fs.FS_SYNC_IDS):
        H.zero_()
        torch.cuda.synchronize()
        H.copy_(p["H"])  # the kernel just before the sampler writes H
        fs.fs_sample_host(ctypes.byref(args), None, None, host_out, sync=sync)
        assert torch.equal(host_out, want), sync


def test_noalloc_entry_point_with_the_flag():
    import ctypes
    B, V = 16, 9000
    p = make_problem(B, 256, V, T=0.8, seed=37)
    dev = p["H"].device
    want = fs.fs_sample(p["H"], p["W"], temperature=p["temperature"], seed=4, offset=1).cpu()
    out = torch.empty(B, dtype=torch.int64, device=dev)
    lib = fs.load_library()
    a = fs.FsSampleArgs(H=p["H"].data_ptr(), W=p["W"].data_ptr(),
                        temperature=p["temperature"].data_ptr(), seed=4, offset=1, B=B, d=256,
                        V=V, ldh=256, ldw=256, out_idx=out.data_ptr(),
                        flags=fs.FS_FLAG_OVERLAP_PREVIOUS)
    s = torch.cuda.current_stream()
    for _ in range(3):
        out.fill_(-5)  # a kernel right before the call
        assert lib.fs_sample_noalloc(ctypes.byref(a), ctypes.c_void_p(s.cuda_stream)) == fs.FS_OK
        torch.cuda.synchronize()
        assert torch.equal(out.cpu(), want)
