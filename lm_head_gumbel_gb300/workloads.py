"""Seeded synthetic workloads for the fused LM-head + Gumbel-max sampler.

This module only draws inputs: it holds none of the sampling arithmetic, and
both the CUDA path and the CPU oracle consume what it produces.  Shapes and
distributions follow the workloads the FlashSampling pages evaluate on
(decode-time LM heads of Qwen3-1.7B / Qwen3-8B / Llama-3-8B-sized models and a
large-vocabulary head); the pages publish no dataset for this kernel, so
everything here is synthetic:

  H ~ N(0, 1) in bf16, W ~ N(0, (2/sqrt(d))^2) in bf16 (logit std ~ 2).

Per-row seeds come from a SplitMix64 hash of (base + row); masks are packed
allow-bits (bit v%32 of word v/32 set = token v allowed).
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    d: int
    V: int
    batches: tuple
    temperature: str          # "const" | "row-uniform" (U[0.5,1.5], 10% greedy)
    t_value: float = 1.0
    mask_frac: float = 0.0    # fraction of (row, token) entries masked out
    outlier_frac: float = 0.0 # fraction of W rows scaled by 4 (exact in bf16)
    per_row_seeds: bool = False
    want_lse: bool = False
    partitions: int = 1       # vocabulary partitions the tile LSE is merged over
    steps: int = 1            # decode steps (offset = step)


WORKLOADS = {
    "tiny": Workload("tiny", d=256, V=4096, batches=(4,), temperature="const",
                     t_value=1.0),
    "qwen3-1.7b": Workload("qwen3-1.7b", d=2048, V=151936,
                           batches=(1, 8, 32, 128, 256), temperature="const",
                           t_value=0.7),
    "qwen3-8b": Workload("qwen3-8b", d=4096, V=151936,
                         batches=(1, 16, 64, 256, 512), temperature="row-uniform",
                         per_row_seeds=True, steps=1000),
    "llama3-8b-mask": Workload("llama3-8b-mask", d=4096, V=128256, batches=(128,),
                               temperature="const", t_value=1.0, mask_frac=0.05,
                               outlier_frac=0.03, want_lse=True),
    "large-vocab": Workload("large-vocab", d=5120, V=262144, batches=(512, 1024),
                            temperature="const", t_value=0.8, want_lse=True,
                            partitions=4),
}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) & 0x7FFFFFFFFFFFFFFF)
    return g


def make_weights(d: int, V: int, seed: int = 1, device="cpu",
                 outlier_frac: float = 0.0) -> torch.Tensor:
    """W [V, d] bf16, N(0, (2/sqrt(d))^2); ``outlier_frac`` of rows times 4."""
    g = _gen(seed, device)
    W = torch.empty((V, d), dtype=torch.bfloat16, device=device)
    chunk = max(1, (1 << 26) // d)  # bound the fp32 staging buffer
    for v0 in range(0, V, chunk):
        v1 = min(V, v0 + chunk)
        tmp = torch.randn((v1 - v0, d), generator=g, device=device, dtype=torch.float32)
        W[v0:v1] = (tmp * (2.0 / math.sqrt(d))).to(torch.bfloat16)
    if outlier_frac > 0:
        n = int(round(outlier_frac * V))
        rows = torch.randperm(V, generator=g, device=device)[:n]
        W[rows] = W[rows] * 4  # a power of two: exact in bf16
    return W


def make_hidden(B: int, d: int, seed: int = 2, device="cpu") -> torch.Tensor:
    """H [B, d] bf16, N(0, 1)."""
    g = _gen(seed, device)
    return torch.randn((B, d), generator=g, device=device,
                       dtype=torch.float32).to(torch.bfloat16)


def make_temperature(wl: Workload, B: int, seed: int = 3, device="cpu") -> torch.Tensor:
    """fp32 [B]: a constant, or U[0.5, 1.5] with 10% of rows set to 0 (greedy)."""
    if wl.temperature == "const":
        return torch.full((B,), float(wl.t_value), dtype=torch.float32, device=device)
    g = _gen(seed, "cpu")
    t = torch.rand((B,), generator=g, dtype=torch.float32) + 0.5
    n_greedy = int(round(0.1 * B))
    if n_greedy:
        t[torch.randperm(B, generator=g)[:n_greedy]] = 0.0
    return t.to(device)


def splitmix64(x: int) -> int:
    """SplitMix64 finaliser (Steele, Lea, Flood, OOPSLA'14) of a 64-bit word."""
    m = (1 << 64) - 1
    z = (x + 0x9E3779B97F4A7C15) & m
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & m
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & m
    return z ^ (z >> 31)


def make_seeds(B: int, base: int = 1234, device="cpu") -> torch.Tensor:
    """Per-row 64-bit seeds, stored as the bit patterns of an int64 tensor."""
    vals = [splitmix64((base + b) & ((1 << 64) - 1)) for b in range(B)]
    signed = [v - (1 << 64) if v >= (1 << 63) else v for v in vals]
    return torch.tensor(signed, dtype=torch.int64, device=device)


def make_mask(B: int, V: int, frac_masked: float, seed: int = 4,
              device="cpu") -> torch.Tensor:
    """Packed allow-bits [B, ceil(V/32)] as int32 bit patterns.

    Each row masks out a seeded random ``frac_masked`` of its tokens; bits past
    V are clear."""
    g = _gen(seed, "cpu")
    n_words = (V + 31) // 32
    allow = torch.rand((B, n_words * 32), generator=g) >= frac_masked
    allow[:, V:] = False
    weights = (1 << torch.arange(32, dtype=torch.int64))
    words = (allow.view(B, n_words, 32).to(torch.int64) * weights).sum(-1)
    words = torch.where(words >= (1 << 31), words - (1 << 32), words)
    return words.to(torch.int32).to(device)


def bf16_bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 array of its bit patterns (host copy)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")


def u32_bits(t: torch.Tensor):
    return t.detach().cpu().contiguous().numpy().view("uint32")


def u64_bits(t: torch.Tensor):
    return t.detach().cpu().contiguous().numpy().view("uint64")
