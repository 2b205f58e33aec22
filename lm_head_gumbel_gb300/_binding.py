"""ctypes binding of ``libfs.so`` (declared in ``include/fs_sample.h``).

Argument marshalling only: tensors become device pointers, sizes and strides;
every step of the sampling path runs in the library's CUDA kernels.  PyTorch
provides device memory and the current stream.  When the library has not been
built, every call raises ``FsError`` -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

FS_TILE = 128
LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libfs.so")

FS_OK = 0
FS_ERR_INVALID_ARG = 1
FS_ERR_UNSUPPORTED = 2
FS_ERR_CUDA = 3
FS_ERR_DEVICE_TIMEOUT = 4
FS_ERR_WORKSPACE = 5
FS_TOPK_MAX = 16
FS_SYNC_NONE, FS_SYNC_STREAM, FS_SYNC_IDS = 0, 1, 2
FS_FLAG_OVERLAP_PREVIOUS = 1
FS_MERGE_EXACT = 0
FS_MERGE_GROUP_GUMBEL = 1

_c_i64 = ctypes.c_int64
_c_u64 = ctypes.c_uint64
_c_ptr = ctypes.c_void_p


class FsError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        name = fs_status_string(status) if _lib is not None else str(status)
        super().__init__(f"{what}: {name}" if what else name)


class FsSampleArgs(ctypes.Structure):
    """Mirror of ``fs_sample_args`` (8-byte fields, then the 32-bit flags)."""
    _fields_ = [
        ("H", _c_ptr), ("W", _c_ptr), ("temperature", _c_ptr),
        ("vocab_mask", _c_ptr), ("mask_ld", _c_i64), ("seeds", _c_ptr),
        ("seed", _c_u64), ("offset", _c_u64),
        ("B", _c_i64), ("d", _c_i64), ("V", _c_i64), ("ldh", _c_i64), ("ldw", _c_i64),
        ("out_idx", _c_ptr), ("out_tile_max", _c_ptr), ("out_tile_idx", _c_ptr),
        ("out_tile_lse", _c_ptr), ("workspace", _c_ptr), ("workspace_bytes", ctypes.c_size_t),
        ("vocab_offset", _c_i64), ("out_max", _c_ptr), ("out_lse", _c_ptr),
        ("flags", ctypes.c_uint32),
    ]


_lib = None


def load_library(path: str = LIB_PATH):
    """Load libfs.so (once).  Raises FsError if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise FsError(FS_ERR_UNSUPPORTED,
                      f"{path} is missing; build it with lm_head_gumbel_gb300.build.build()")
    lib = ctypes.CDLL(path)
    lib.fs_num_tiles.argtypes = [_c_i64]
    lib.fs_num_tiles.restype = _c_i64
    lib.fs_workspace_size.argtypes = [_c_i64, _c_i64]
    lib.fs_workspace_size.restype = ctypes.c_size_t
    lib.fs_sample.argtypes = [ctypes.POINTER(FsSampleArgs), _c_ptr]
    lib.fs_sample.restype = ctypes.c_int
    lib.fs_sample_noalloc.argtypes = [ctypes.POINTER(FsSampleArgs), _c_ptr]
    lib.fs_sample_noalloc.restype = ctypes.c_int
    lib.fs_sample_host.argtypes = [ctypes.POINTER(FsSampleArgs), _c_ptr, _c_ptr, ctypes.c_size_t,
                                   _c_ptr, ctypes.c_int, _c_ptr]
    lib.fs_sample_host.restype = ctypes.c_int
    lib.fs_gumbel_noise.argtypes = [_c_ptr, _c_u64, _c_u64, _c_i64, _c_i64, _c_i64, _c_i64,
                                    _c_ptr, _c_ptr]
    lib.fs_gumbel_noise.restype = ctypes.c_int
    lib.fs_gumbel_transform.argtypes = [_c_ptr, _c_i64, _c_ptr, _c_ptr]
    lib.fs_gumbel_transform.restype = ctypes.c_int
    lib.fs_topk_workspace_size.argtypes = [_c_i64, _c_i64, _c_i64]
    lib.fs_topk_workspace_size.restype = ctypes.c_size_t
    lib.fs_sample_topk.argtypes = [ctypes.POINTER(FsSampleArgs), _c_i64, _c_ptr, _c_ptr, _c_ptr]
    lib.fs_sample_topk.restype = ctypes.c_int
    lib.fs_group_merge.argtypes = [_c_ptr, _c_ptr, _c_ptr, _c_i64, _c_i64, ctypes.c_int, _c_ptr,
                                   _c_u64, _c_u64, _c_ptr, _c_ptr, _c_ptr]
    lib.fs_group_merge.restype = ctypes.c_int
    lib.fs_online_merge.argtypes = [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_i64, _c_u64, _c_ptr, _c_u64,
                                    _c_u64, _c_ptr]
    lib.fs_online_merge.restype = ctypes.c_int
    lib.fs_wait_timeout_selftest.argtypes = [_c_u64, _c_ptr]
    lib.fs_wait_timeout_selftest.restype = ctypes.c_int
    lib.fs_last_device_error.argtypes = [_c_ptr, ctypes.POINTER(ctypes.c_int)]
    lib.fs_last_device_error.restype = ctypes.c_int
    lib.fs_status_string.argtypes = [ctypes.c_int]
    lib.fs_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def fs_num_tiles(V: int) -> int:
    return int(load_library().fs_num_tiles(int(V)))


def fs_workspace_size(B: int, V: int) -> int:
    return int(load_library().fs_workspace_size(int(B), int(V)))


def fs_status_string(status: int) -> str:
    return load_library().fs_status_string(int(status)).decode()


def fs_last_device_error(stream=None, device=None):
    """(status, raw error word) of the device, read and cleared after the work
    enqueued on `stream` (default: the current stream), waiting for that
    stream only.  The word is one per device (see the header)."""
    code = ctypes.c_int(0)
    device = torch.device(device or "cuda")
    with torch.cuda.device(device):
        st = load_library().fs_last_device_error(_stream_handle(stream, device),
                                                 ctypes.byref(code))
    return int(st), int(code.value)


def fs_wait_timeout_selftest(limit_ns: int, device=None, stream=None):
    """Run the kernels' bounded wait on a barrier nothing arrives on (see the
    header); the timeout then shows in fs_last_device_error()."""
    lib = load_library()
    device = torch.device(device or "cuda")
    with torch.cuda.device(device):
        st = lib.fs_wait_timeout_selftest(int(limit_ns), _stream_handle(stream, device))
    if st != FS_OK:
        raise FsError(st, "fs_wait_timeout_selftest")


def _check_2d(name, t, dtype):
    if t.dtype != dtype or t.dim() != 2 or t.stride(1) != 1 or not t.is_cuda:
        raise FsError(FS_ERR_INVALID_ARG, f"{name} must be a CUDA {dtype} matrix with unit column stride")


def fs_sample(H, W, *, temperature=None, vocab_mask=None, seeds=None, seed=0, offset=0,
              out_idx=None, out_tile_max=None, out_tile_idx=None, out_tile_lse=None,
              workspace=None, stream=None, reduce=True, vocab_offset=0, out_max=None,
              out_lse=None, overlap_previous=False):
    """Sample one token id per row of H from softmax(H W^T / T) (masked).

    H: bf16 [B, d]; W: bf16 [V, d]; temperature: fp32 [B] or None (T = 1);
    vocab_mask: int32 [B, >= ceil(V/32)] allow-bits or None; seeds: int64 [B]
    holding uint64 bit patterns, or None (``seed`` for every row).  Optional
    per-tile outputs are [B, ceil(V/128)] (fp32 / int32 / fp32).  workspace:
    a uint8 tensor of fs_workspace_size(B, V) bytes that is all-zero before
    its first use (calls leave it zeroed), or None for a fresh one.  Returns
    ``out_idx`` (int64 [B]).  Asynchronous on ``stream`` (default: the
    current stream of H's device).  With ``reduce=False`` only stage 1 runs:
    the per-tile outputs (required then) are written and None is returned.
    vocab_offset: global id of W's first row (W a vocabulary shard); out_max /
    out_lse: optional fp32 [B] row maximum / row log-mass (out_lse needs
    out_tile_lse).  overlap_previous: launch as a programmatic dependent of the
    stream's previous kernel (FS_FLAG_OVERLAP_PREVIOUS: W starts streaming
    while that kernel finishes; it may write H and the per-row inputs, not W)."""
    lib = load_library()
    _check_2d("H", H, torch.bfloat16)
    _check_2d("W", W, torch.bfloat16)
    B, d = H.shape
    V = W.shape[0]
    dev = H.device
    if not reduce:
        if out_tile_max is None or out_tile_idx is None:
            raise FsError(FS_ERR_INVALID_ARG, "reduce=False needs out_tile_max and out_tile_idx")
        out_idx = None
    elif out_idx is None:
        out_idx = torch.empty(B, dtype=torch.int64, device=dev)
    mask_ld = 0
    if vocab_mask is not None:
        if vocab_mask.dtype != torch.int32 or vocab_mask.dim() != 2 or vocab_mask.stride(1) != 1:
            raise FsError(FS_ERR_INVALID_ARG, "vocab_mask must be an int32 matrix")
        mask_ld = vocab_mask.stride(0)
    if seeds is not None and seeds.dtype != torch.int64:
        raise FsError(FS_ERR_INVALID_ARG, "seeds must be int64 (uint64 bit patterns)")
    if temperature is not None and temperature.dtype != torch.float32:
        raise FsError(FS_ERR_INVALID_ARG, "temperature must be float32")
    if reduce and workspace is None:  # zero-filled, as the library requires
        workspace = torch.zeros(fs_workspace_size(B, V), dtype=torch.uint8, device=dev)
    args = FsSampleArgs(
        H=_ptr(H), W=_ptr(W), temperature=_ptr(temperature), vocab_mask=_ptr(vocab_mask),
        mask_ld=mask_ld, seeds=_ptr(seeds), seed=int(seed) & (2**64 - 1),
        offset=int(offset) & (2**64 - 1), B=B, d=d, V=V, ldh=H.stride(0), ldw=W.stride(0),
        out_idx=_ptr(out_idx), out_tile_max=_ptr(out_tile_max), out_tile_idx=_ptr(out_tile_idx),
        out_tile_lse=_ptr(out_tile_lse),
        workspace=_ptr(workspace) if reduce else None,
        workspace_bytes=(workspace.numel() * workspace.element_size()) if reduce else 0,
        vocab_offset=int(vocab_offset), out_max=_ptr(out_max), out_lse=_ptr(out_lse),
        flags=FS_FLAG_OVERLAP_PREVIOUS if overlap_previous else 0)
    with torch.cuda.device(dev):
        st = lib.fs_sample(ctypes.byref(args), _stream_handle(stream, dev))
    if st != FS_OK:
        raise FsError(st, "fs_sample")
    return out_idx


def fs_sample_host(args, host_in, dev_in, host_out, *, sync=True, stream=None, device=None):
    """One decode step from host memory (the C entry point of the same name):
    copy host_in (pinned uint8 host tensor) to dev_in (uint8 device tensor of
    at least the same size), run fs_sample with ``args`` (an FsSampleArgs
    whose input pointers point into dev_in, or elsewhere on the device), copy
    the B sampled ids to host_out (pinned int64 [B] host tensor) and wait:
    ``sync`` is True / FS_SYNC_STREAM (the stream), FS_SYNC_IDS (until the
    ids are in host_out) or False / FS_SYNC_NONE.  host_in may be None
    (nothing to copy).  Pass ``args`` by reference (``ctypes.byref``) to
    reuse one argument block."""
    lib = load_library()
    device = torch.device(device or "cuda")
    n = 0 if host_in is None else host_in.numel() * host_in.element_size()
    if host_in is not None and (host_in.is_cuda or not dev_in.is_cuda
                                or dev_in.numel() * dev_in.element_size() < n):
        raise FsError(FS_ERR_INVALID_ARG, "host_in must be host memory no larger than dev_in")
    if host_out.is_cuda or host_out.dtype != torch.int64 or host_out.numel() < args_batch(args):
        raise FsError(FS_ERR_INVALID_ARG, "host_out must be an int64 host tensor of B entries")
    ref = args if isinstance(args, type(ctypes.byref(FsSampleArgs()))) else ctypes.byref(args)
    with torch.cuda.device(device):
        st = lib.fs_sample_host(ref, _ptr(host_in), _ptr(dev_in) if host_in is not None else None,
                                n, _ptr(host_out), int(sync),
                                _stream_handle(stream, device))
    if st != FS_OK:
        raise FsError(st, "fs_sample_host")
    return host_out


def args_batch(args) -> int:
    """B of an FsSampleArgs (or of a ctypes reference to one)."""
    obj = getattr(args, "_obj", args)
    return int(obj.B)


def fs_topk_workspace_size(B: int, V: int, K: int) -> int:
    return int(load_library().fs_topk_workspace_size(int(B), int(V), int(K)))


def fs_sample_topk(H, W, K, *, temperature=None, vocab_mask=None, seeds=None, seed=0, offset=0,
                   vocab_offset=0, out_topk_idx=None, out_topk_score=None, workspace=None,
                   stream=None, overlap_previous=False):
    """K draws without replacement per row (the K largest noisy scores, in
    draw order).  Returns out_topk_idx (int64 [B, K]); fills out_topk_score
    (fp32 [B, K]) when given.  overlap_previous: as in fs_sample."""
    lib = load_library()
    _check_2d("H", H, torch.bfloat16)
    _check_2d("W", W, torch.bfloat16)
    B, d = H.shape
    V = W.shape[0]
    dev = H.device
    if out_topk_idx is None:
        out_topk_idx = torch.empty((B, K), dtype=torch.int64, device=dev)
    if workspace is None:
        workspace = torch.empty(max(1, fs_topk_workspace_size(B, V, K)), dtype=torch.uint8,
                                device=dev)
    mask_ld = 0 if vocab_mask is None else vocab_mask.stride(0)
    args = FsSampleArgs(
        H=_ptr(H), W=_ptr(W), temperature=_ptr(temperature), vocab_mask=_ptr(vocab_mask),
        mask_ld=mask_ld, seeds=_ptr(seeds), seed=int(seed) & (2**64 - 1),
        offset=int(offset) & (2**64 - 1), B=B, d=d, V=V, ldh=H.stride(0), ldw=W.stride(0),
        workspace=_ptr(workspace), workspace_bytes=workspace.numel() * workspace.element_size(),
        vocab_offset=int(vocab_offset), flags=FS_FLAG_OVERLAP_PREVIOUS if overlap_previous else 0)
    with torch.cuda.device(dev):
        st = lib.fs_sample_topk(ctypes.byref(args), int(K), _ptr(out_topk_idx),
                                _ptr(out_topk_score), _stream_handle(stream, dev))
    if st != FS_OK:
        raise FsError(st, "fs_sample_topk")
    return out_topk_idx


def fs_group_merge(z, *, m=None, L=None, mode=FS_MERGE_EXACT, seeds=None, seed=0, offset=0,
                   out_idx=None, out_L=None, stream=None):
    """One sample per row from P partitions' results z / m / L ([P, B]).
    mode FS_MERGE_EXACT: argmax of m; FS_MERGE_GROUP_GUMBEL: Group-Gumbel-Max
    over L with the merge's own noise.  Returns out_idx (int64 [B])."""
    lib = load_library()
    P, B = z.shape
    dev = z.device
    if out_idx is None:
        out_idx = torch.empty(B, dtype=torch.int64, device=dev)
    with torch.cuda.device(dev):
        st = lib.fs_group_merge(_ptr(z), _ptr(m), _ptr(L), P, B, int(mode), _ptr(seeds),
                                int(seed) & (2**64 - 1), int(offset) & (2**64 - 1),
                                _ptr(out_idx), _ptr(out_L), _stream_handle(stream, dev))
    if st != FS_OK:
        raise FsError(st, "fs_group_merge")
    return out_idx


def fs_online_merge(state_z, state_L, new_z, new_L, step, *, seeds=None, seed=0, offset=0,
                    stream=None):
    """Fold group `step` (new_z, new_L: [B]) into the running (state_z,
    state_L) in place (start from -1 / -inf)."""
    lib = load_library()
    B = state_z.shape[0]
    dev = state_z.device
    with torch.cuda.device(dev):
        st = lib.fs_online_merge(_ptr(state_z), _ptr(state_L), _ptr(new_z), _ptr(new_L), B,
                                 int(step), _ptr(seeds), int(seed) & (2**64 - 1),
                                 int(offset) & (2**64 - 1), _stream_handle(stream, dev))
    if st != FS_OK:
        raise FsError(st, "fs_online_merge")


def fs_gumbel_transform(words, out=None, stream=None):
    """The fp32 Gumbel noise of given 32-bit Philox words (an int32 CUDA
    tensor holding the bit patterns) -- the transform fs_sample applies
    (diagnostic)."""
    lib = load_library()
    if words.dtype != torch.int32 or not words.is_cuda or not words.is_contiguous():
        raise FsError(FS_ERR_INVALID_ARG, "words must be a contiguous int32 CUDA tensor")
    if out is None:
        out = torch.empty(words.shape, dtype=torch.float32, device=words.device)
    with torch.cuda.device(words.device):
        st = lib.fs_gumbel_transform(_ptr(words), int(words.numel()), _ptr(out),
                                     _stream_handle(stream, words.device))
    if st != FS_OK:
        raise FsError(st, "fs_gumbel_transform")
    return out


def fs_gumbel_noise(b0, nb, v0, nv, *, seed=0, offset=0, seeds=None, out=None, device=None,
                    stream=None):
    """The fp32 Gumbel noise g[b, v] that fs_sample adds, for a window of
    rows x vocabulary ids (diagnostic)."""
    lib = load_library()
    device = torch.device(device or (seeds.device if seeds is not None else "cuda"))
    if out is None:
        out = torch.empty((nb, nv), dtype=torch.float32, device=device)
    with torch.cuda.device(device):
        st = lib.fs_gumbel_noise(_ptr(seeds), int(seed) & (2**64 - 1), int(offset) & (2**64 - 1),
                                 int(b0), int(nb), int(v0), int(nv), _ptr(out),
                                 _stream_handle(stream, device))
    if st != FS_OK:
        raise FsError(st, "fs_gumbel_noise")
    return out
