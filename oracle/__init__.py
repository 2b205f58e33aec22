"""CPU oracle for fused LM-head + exact Gumbel-max sampling (FlashSampling).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import or call anything here; the product
library never does, and it shares no code with this package.

The arithmetic lives in ``fs_oracle.c`` (plain fp64 C, one function per step of
the definition); this module only marshals numpy arrays into it.  Group merges
and statistics helpers that sit on top of the per-tile outputs are in
``oracle.merge``.

Pins (what ties the oracle to something other than itself) are in
``tests/test_oracle_pins.py``; planted-mistake checks are in
``tests/test_oracle_mutants.py``.
"""
from __future__ import annotations

import ctypes
import math
import os

import numpy as np

from . import build as _build

_i64 = ctypes.c_int64
_u64 = ctypes.c_uint64
_u32 = ctypes.c_uint32
_ptr = ctypes.c_void_p

TILE = 128  # vocabulary tile width of the per-tile outputs


def _p(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


class Oracle:
    """Thin ctypes view of one compiled oracle library."""

    def __init__(self, libpath: str | None = None):
        self.path = libpath or _build.build()
        self.lib = ctypes.CDLL(self.path)
        L = self.lib
        L.fso_philox4x32_10.argtypes = [_ptr, _ptr, _ptr]
        L.fso_philox4x32_10.restype = None
        L.fso_uniform.argtypes = [_u32]
        L.fso_uniform.restype = ctypes.c_double
        L.fso_gumbel.argtypes = [ctypes.c_double]
        L.fso_gumbel.restype = ctypes.c_double
        L.fso_noise_word.argtypes = [_u64, _u64, _i64, _i64]
        L.fso_noise_word.restype = _u32
        L.fso_noise.argtypes = [_u64, _u64, _i64, _i64]
        L.fso_noise.restype = ctypes.c_double
        L.fso_merge_uniform.argtypes = [_u64, _u64, _i64, _i64]
        L.fso_merge_uniform.restype = ctypes.c_double
        L.fso_noise_grid.argtypes = [_ptr, _u64, _u64, _i64, _i64, _i64, _i64, _ptr]
        L.fso_noise_grid.restype = None
        L.fso_logits.argtypes = [_ptr, _ptr, _i64, _i64, _i64, _i64, _i64, _ptr]
        L.fso_logits.restype = None
        L.fso_sample_rows.argtypes = [
            _ptr, _ptr, _i64, _i64, _i64, _i64, _i64,  # H W B d V ldh ldw
            _ptr, _ptr, _i64, _ptr, _u64, _u64,        # T mask mask_ld seeds seed offset
            _i64, _ptr, _i64,                          # tile rows n_rows
            _ptr, _ptr, _ptr, _ptr, _ptr, _ptr,        # idx gap tmax tidx tlse tgap
            _ptr, _ptr]                                # logits scores
        L.fso_sample_rows.restype = ctypes.c_int
        L.fso_num_threads.argtypes = []
        L.fso_num_threads.restype = ctypes.c_int
        L.fso_set_num_threads.argtypes = [ctypes.c_int]
        L.fso_set_num_threads.restype = None

    # ---- scalar pieces ---------------------------------------------------
    def philox(self, counter, key):
        c = np.ascontiguousarray(counter, dtype=np.uint32)
        k = np.ascontiguousarray(key, dtype=np.uint32)
        out = np.zeros(4, dtype=np.uint32)
        self.lib.fso_philox4x32_10(_p(c), _p(k), _p(out))
        return out

    def uniform(self, word: int) -> float:
        return self.lib.fso_uniform(int(word) & 0xFFFFFFFF)

    def gumbel(self, u: float) -> float:
        return self.lib.fso_gumbel(float(u))

    def noise_word(self, seed: int, offset: int, b: int, v: int) -> int:
        return self.lib.fso_noise_word(seed, offset, b, v)

    def noise(self, seed: int, offset: int, b: int, v: int) -> float:
        return self.lib.fso_noise(seed, offset, b, v)

    def merge_uniform(self, seed: int, offset: int, b: int, k: int) -> float:
        """The uniform a merge draws for row b and partition / step k."""
        return self.lib.fso_merge_uniform(int(seed) & (2**64 - 1), int(offset) & (2**64 - 1), b, k)

    def merge_uniforms(self, seed: int, offset: int, b: int, n: int):
        return np.array([self.merge_uniform(seed, offset, b, k) for k in range(n)])

    def noise_grid(self, b0, nb, v0, nv, seed=0, offset=0, seeds=None):
        out = np.empty((nb, nv), dtype=np.float64)
        sd = None if seeds is None else np.ascontiguousarray(seeds, dtype=np.uint64)
        self.lib.fso_noise_grid(_p(sd), seed, offset, b0, nb, v0, nv, _p(out))
        return out

    def num_threads(self) -> int:
        return self.lib.fso_num_threads()

    def set_num_threads(self, n: int) -> None:
        """Threads of the OpenMP regions from now on (results do not depend on it)."""
        self.lib.fso_set_num_threads(int(n))

    # ---- the definition ------------------------------------------------------
    def logits(self, H, W):
        """fp64 logits l = H W^T from bf16 bit patterns (uint16 arrays)."""
        H = np.ascontiguousarray(H, dtype=np.uint16)
        W = np.ascontiguousarray(W, dtype=np.uint16)
        B, d = H.shape
        V = W.shape[0]
        out = np.empty((B, V), dtype=np.float64)
        self.lib.fso_logits(_p(H), _p(W), B, d, V, d, d, _p(out))
        return out

    def sample(self, H, W, temperature=None, mask=None, seeds=None, seed=0,
               offset=0, rows=None, tile=TILE, want_logits=False,
               want_scores=False):
        """Run the sampling definition on the requested rows.

        H: uint16 [B, d] (bf16 bits); W: uint16 [V, d]; temperature: float32 [B]
        or None (1.0); mask: uint32 [B, ceil(V/32)] allow-bits or None; seeds:
        uint64 [B] or None (``seed`` for every row); rows: row indices or None
        (every row).  Returns a dict of numpy arrays indexed by requested row.
        """
        H = np.ascontiguousarray(H, dtype=np.uint16)
        W = np.ascontiguousarray(W, dtype=np.uint16)
        B, d = H.shape
        V, d2 = W.shape
        if d2 != d:
            raise ValueError("H and W disagree on d")
        T = None if temperature is None else np.ascontiguousarray(temperature, dtype=np.float32)
        M = None if mask is None else np.ascontiguousarray(mask, dtype=np.uint32)
        mask_ld = 0 if M is None else M.shape[1]
        if M is not None and (M.shape[0] != B or mask_ld < (V + 31) // 32):
            raise ValueError("mask must be uint32 [B, >= ceil(V/32)]")
        S = None if seeds is None else np.ascontiguousarray(seeds, dtype=np.uint64)
        R = np.arange(B, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
        n = R.shape[0]
        nt = (V + tile - 1) // tile
        out = {
            "rows": R,
            "idx": np.empty(n, dtype=np.int64),
            "gap": np.empty(n, dtype=np.float64),
            "tile_max": np.empty((n, nt), dtype=np.float64),
            "tile_idx": np.empty((n, nt), dtype=np.int64),
            "tile_lse": np.empty((n, nt), dtype=np.float64),
            "tile_gap": np.empty((n, nt), dtype=np.float64),
        }
        lg = np.empty((n, V), dtype=np.float64) if want_logits else None
        sc = np.empty((n, V), dtype=np.float64) if want_scores else None
        rc = self.lib.fso_sample_rows(
            _p(H), _p(W), B, d, V, d, d, _p(T), _p(M), mask_ld, _p(S),
            int(seed) & (2**64 - 1), int(offset) & (2**64 - 1), tile, _p(R), n,
            _p(out["idx"]), _p(out["gap"]), _p(out["tile_max"]),
            _p(out["tile_idx"]), _p(out["tile_lse"]), _p(out["tile_gap"]),
            _p(lg), _p(sc))
        if rc != 0:
            raise ValueError("oracle rejected its arguments")
        if want_logits:
            out["logits"] = lg
        if want_scores:
            out["scores"] = sc
        return out


def topk_from_scores(scores, K):
    """The ids of the K largest scores of each row, best first, ties to the
    lower id (a library sort is the step); -1 / -inf past the finite count."""
    scores = np.asarray(scores, dtype=np.float64)
    n, V = scores.shape
    idx = np.full((n, K), -1, dtype=np.int64)
    val = np.full((n, K), -np.inf)
    for r in range(n):
        order = np.lexsort((np.arange(V), -scores[r]))  # score desc, then id asc
        keep = [v for v in order[:K] if np.isfinite(scores[r, v])]
        idx[r, :len(keep)] = keep
        val[r, :len(keep)] = scores[r, keep]
    return idx, val


def sample_topk(o, H, W, K, **kw):
    """K draws without replacement per row (the K largest noisy scores):
    returns (ids [n, K], scores [n, K], the oracle's sample dict)."""
    ref = o.sample(H, W, want_scores=True, **kw)
    idx, val = topk_from_scores(ref["scores"], K)
    return idx, val, ref


_default: Oracle | None = None


def default() -> Oracle:
    """The oracle built from ``fs_oracle.c`` (compiled on first use)."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default


EULER_GAMMA = 0.5772156649015329
GUMBEL_VAR = math.pi ** 2 / 6.0
