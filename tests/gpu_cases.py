"""Shared driver for the GPU parity tests: draw a seeded synthetic problem, run
the CUDA path through the C ABI, run the oracle on the same inputs, compare.
"""
from __future__ import annotations

import numpy as np
import torch

import lm_head_gumbel_gb300 as fs
from lm_head_gumbel_gb300 import workloads as wl
import oracle
from oracle import parity


def make_problem(B, d, V, *, T=1.0, greedy_frac=0.0, mask_frac=0.0, per_row_seeds=False,
                 outlier_frac=0.0, seed=0, device="cuda", W=None):
    """Seeded inputs on the device; returns a dict of tensors."""
    if W is None:
        W = wl.make_weights(d, V, seed=1000 + seed, device=device, outlier_frac=outlier_frac)
    H = wl.make_hidden(B, d, seed=2000 + seed, device=device)
    if T == "row-uniform":
        temp = wl.make_temperature(wl.WORKLOADS["qwen3-8b"], B, seed=3000 + seed, device=device)
    else:
        temp = torch.full((B,), float(T), dtype=torch.float32, device=device)
        if greedy_frac > 0:
            g = torch.Generator().manual_seed(seed)
            n = max(1, int(round(greedy_frac * B)))
            temp[torch.randperm(B, generator=g)[:n].to(device)] = 0.0
    seeds = wl.make_seeds(B, base=4000 + seed, device=device) if per_row_seeds else None
    mask = wl.make_mask(B, V, mask_frac, seed=5000 + seed, device=device) if mask_frac > 0 else None
    return {"H": H, "W": W, "temperature": temp, "seeds": seeds, "vocab_mask": mask}


def run_device(prob, *, seed=7, offset=0, lse=True, stream=None, tiles=True):
    H, W = prob["H"], prob["W"]
    B, V = H.shape[0], W.shape[0]
    nt = fs.fs_num_tiles(V)
    torch.cuda.synchronize()  # inputs were written on the default stream
    out = {}
    kw = {}
    if tiles:
        out["tile_max"] = torch.empty((B, nt), dtype=torch.float32, device=H.device)
        out["tile_idx"] = torch.empty((B, nt), dtype=torch.int32, device=H.device)
        kw = dict(out_tile_max=out["tile_max"], out_tile_idx=out["tile_idx"])
    if lse:
        out["tile_lse"] = torch.empty((B, nt), dtype=torch.float32, device=H.device)
        kw["out_tile_lse"] = out["tile_lse"]
    out["idx"] = fs.fs_sample(H, W, temperature=prob["temperature"],
                              vocab_mask=prob["vocab_mask"], seeds=prob["seeds"], seed=seed,
                              offset=offset, stream=stream, **kw)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def run_oracle(prob, rows=None, *, seed=7, offset=0, scores=False, W_bits=None):
    o = oracle.default()
    Hb = wl.bf16_bits(prob["H"])
    Wb = W_bits if W_bits is not None else wl.bf16_bits(prob["W"])
    return o.sample(Hb, Wb, temperature=prob["temperature"].cpu().numpy(),
                    mask=None if prob["vocab_mask"] is None else wl.u32_bits(prob["vocab_mask"]),
                    seeds=None if prob["seeds"] is None else wl.u64_bits(prob["seeds"]),
                    seed=seed, offset=offset, rows=rows, want_scores=scores)


def compare(prob, dev, rows=None, *, seed=7, offset=0, scores=False, W_bits=None):
    ref = run_oracle(prob, rows, seed=seed, offset=offset, scores=scores, W_bits=W_bits)
    sel = ref["rows"]
    return parity.check(ref, dev["idx"][sel],
                        dev["tile_max"][sel] if "tile_max" in dev else None,
                        dev["tile_idx"][sel] if "tile_idx" in dev else None,
                        dev["tile_lse"][sel] if "tile_lse" in dev else None,
                        scores=ref.get("scores"))


def assert_no_device_error():
    st, code = fs.fs_last_device_error()
    assert st == fs.FS_OK and code == 0, (st, code)
