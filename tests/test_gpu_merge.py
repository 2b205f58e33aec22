"""Vocabulary partitions and their merges on the GPU, against the oracle.

- Shards of W sampled with their global vocab_offset and merged exactly
  (argmax of the shards' maxima) give the unsharded sample, bit for bit
  (tomesphere abstract: exact because argmax decomposes over partitions).
- The row maximum / log-mass outputs match the oracle.
- Group-Gumbel-Max and the online binary merge (aitrends.kr write-up), fed the
  shards' (z_k, L_k), pick what the oracle picks with the same Philox merge
  uniforms, and their draws follow softmax(l/T) (chi-square).
"""
import numpy as np
import pytest
import scipy.special
import torch

import lm_head_gumbel_gb300 as fs
from lm_head_gumbel_gb300 import workloads as wl
import oracle
from oracle import merge, parity
from gpu_cases import assert_no_device_error, make_problem

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fs.load_library()
    yield
    assert_no_device_error()


def shard_calls(p, bounds, *, seed=7, offset=0, lse=False):
    """fs_sample on each shard W[b_k:b_{k+1}] with vocab_offset b_k; returns
    z, m (and L) as [P, B] device tensors."""
    H, W = p["H"], p["W"]
    B = H.shape[0]
    P = len(bounds) - 1
    z = torch.empty((P, B), dtype=torch.int64, device="cuda")
    m = torch.empty((P, B), dtype=torch.float32, device="cuda")
    L = torch.empty((P, B), dtype=torch.float32, device="cuda") if lse else None
    for k in range(P):
        Wk = W[bounds[k]:bounds[k + 1]]
        kw = {}
        if lse:
            nt = fs.fs_num_tiles(Wk.shape[0])
            kw = dict(out_tile_max=torch.empty((B, nt), dtype=torch.float32, device="cuda"),
                      out_tile_idx=torch.empty((B, nt), dtype=torch.int32, device="cuda"),
                      out_tile_lse=torch.empty((B, nt), dtype=torch.float32, device="cuda"),
                      out_lse=L[k])
        fs.fs_sample(H, Wk, temperature=p["temperature"], vocab_mask=None, seeds=p["seeds"],
                     seed=seed, offset=offset, out_idx=z[k], out_max=m[k],
                     vocab_offset=bounds[k], **kw)
    return z, m, L


@pytest.mark.parametrize("bounds", [[0, 1024, 2048, 3072, 4000], [0, 1000, 2004, 2996, 4000]])
def test_sharded_exact_merge_is_the_unsharded_sample(bounds):
    p = make_problem(24, 128, 4000, T="row-uniform", per_row_seeds=True, seed=31)
    full_max = torch.empty(24, dtype=torch.float32, device="cuda")
    full = fs.fs_sample(p["H"], p["W"], temperature=p["temperature"], seeds=p["seeds"],
                        seed=7, offset=5, out_max=full_max)
    z, m, _ = shard_calls(p, bounds, offset=5)
    got = fs.fs_group_merge(z, m=m, mode=fs.FS_MERGE_EXACT)
    torch.cuda.synchronize()
    full, got, full_max = full.cpu().numpy(), got.cpu().numpy(), full_max.cpu().numpy()
    mmax = m.max(dim=0).values.cpu().numpy()
    if bounds[1] % 256 == 0:  # same vocabulary blocks: identical arithmetic
        assert np.array_equal(got, full)
        assert np.array_equal(mmax, full_max)
    else:  # blocks shifted: fp32 sums may round differently; gate on the oracle's gap
        o = oracle.default()
        ref = o.sample(wl.bf16_bits(p["H"]), wl.bf16_bits(p["W"]),
                       temperature=p["temperature"].cpu().numpy(),
                       seeds=wl.u64_bits(p["seeds"]), offset=5)
        gated = ref["gap"] > parity.GAP
        assert np.array_equal(got[gated], full[gated]) and gated.sum() > 15
        assert np.allclose(mmax, full_max, atol=parity.TOL_MAX)
    # every shard's id lies in its shard
    zc = z.cpu().numpy()
    for k in range(len(bounds) - 1):
        assert np.all((zc[k] >= bounds[k]) & (zc[k] < bounds[k + 1]))


def test_row_max_and_log_mass_match_oracle():
    p = make_problem(12, 96, 3000, T="row-uniform", mask_frac=0.05, seed=32)
    nt = fs.fs_num_tiles(3000)
    out_max = torch.empty(12, dtype=torch.float32, device="cuda")
    out_lse = torch.empty(12, dtype=torch.float32, device="cuda")
    idx = fs.fs_sample(p["H"], p["W"], temperature=p["temperature"],
                       vocab_mask=p["vocab_mask"], seed=3, offset=9, out_max=out_max,
                       out_lse=out_lse,
                       out_tile_max=torch.empty((12, nt), dtype=torch.float32, device="cuda"),
                       out_tile_idx=torch.empty((12, nt), dtype=torch.int32, device="cuda"),
                       out_tile_lse=torch.empty((12, nt), dtype=torch.float32, device="cuda"))
    torch.cuda.synchronize()
    o = oracle.default()
    ref = o.sample(wl.bf16_bits(p["H"]), wl.bf16_bits(p["W"]),
                   temperature=p["temperature"].cpu().numpy(),
                   mask=wl.u32_bits(p["vocab_mask"]), seed=3, offset=9, tile=3000)
    assert np.allclose(out_max.cpu().numpy(), ref["tile_max"][:, 0], atol=parity.TOL_MAX)
    assert np.allclose(out_lse.cpu().numpy(), ref["tile_lse"][:, 0], atol=parity.TOL_LSE)
    gated = ref["gap"] > parity.GAP
    assert np.array_equal(idx.cpu().numpy()[gated], ref["idx"][gated])


def _oracle_partitions(p, width, seed, offset):
    o = oracle.default()
    ref = o.sample(wl.bf16_bits(p["H"]), wl.bf16_bits(p["W"]),
                   temperature=p["temperature"].cpu().numpy(),
                   seeds=None if p["seeds"] is None else wl.u64_bits(p["seeds"]),
                   seed=seed, offset=offset, tile=width)
    return ref


def test_group_gumbel_and_online_merges_match_oracle():
    B, V, w = 48, 4096, 1024
    p = make_problem(B, 64, V, T=0.9, per_row_seeds=True, seed=33)
    bounds = list(range(0, V + 1, w))
    z, _, L = shard_calls(p, bounds, offset=11, lse=True)
    seeds = p["seeds"]
    grp = fs.fs_group_merge(z, L=L, mode=fs.FS_MERGE_GROUP_GUMBEL, seeds=seeds, offset=11)
    sz = torch.full((B,), -1, dtype=torch.int64, device="cuda")
    sL = torch.full((B,), float("-inf"), dtype=torch.float32, device="cuda")
    for k in range(len(bounds) - 1):
        fs.fs_online_merge(sz, sL, z[k], L[k], k, seeds=seeds, offset=11)
    torch.cuda.synchronize()
    grp, sz, sL = grp.cpu().numpy(), sz.cpu().numpy(), sL.cpu().numpy()
    zc, Lc = z.cpu().numpy(), L.cpu().numpy()
    ref = _oracle_partitions(p, w, 7, 11)
    o = oracle.default()
    sd = wl.u64_bits(seeds)
    n_g = n_o = 0
    for b in range(B):
        zr, Lr = ref["tile_idx"][b], ref["tile_lse"][b]
        assert np.allclose(Lc[:, b], Lr, atol=parity.TOL_LSE)
        same_parts = np.all((zc[:, b] == zr) | (ref["tile_gap"][b] <= parity.GAP))
        u = o.merge_uniforms(int(sd[b]), 11, b, len(Lr))
        keys = np.sort(Lr - np.log(-np.log(u)))
        if same_parts and keys[-1] - keys[-2] > 1e-3:
            assert grp[b] == merge.group_gumbel_max(zr, Lr, u), b
            n_g += 1
        zo, Lo = merge.online_merge(zr, Lr, u)
        assert abs(sL[b] - Lo) < 2e-3
        # switches whose probability sits within 1e-5 of the uniform are not gated exactly
        cur = Lr[0]
        near = False
        for k in range(1, len(Lr)):
            new = np.logaddexp(cur, Lr[k])
            near |= abs(u[k] - np.exp(Lr[k] - new)) < 1e-5
            cur = new
        if same_parts and not near:
            assert sz[b] == zo, b
            n_o += 1
    assert n_g > 0.8 * B and n_o > 0.8 * B


@pytest.mark.parametrize("mode", ["group", "online"])
def test_merged_draws_follow_softmax(mode):
    """V = 64 in four shards of 16: the merged draws over 3000 offsets pass a
    chi-square test against softmax(l / T)."""
    V, d, T, n = 64, 16, 1.0, 3000
    p = make_problem(1, d, V, T=T, seed=34)
    bounds = [0, 16, 32, 48, 64]
    probs = scipy.special.softmax(
        oracle.default().logits(wl.bf16_bits(p["H"]), wl.bf16_bits(p["W"]))[0] / T)
    draws = torch.empty(n, dtype=torch.int64, device="cuda")
    sz = torch.empty(1, dtype=torch.int64, device="cuda")
    sL = torch.empty(1, dtype=torch.float32, device="cuda")
    for off in range(n):
        z, _, L = shard_calls(p, bounds, seed=99, offset=off, lse=True)
        if mode == "group":
            fs.fs_group_merge(z, L=L, mode=fs.FS_MERGE_GROUP_GUMBEL, seed=99, offset=off,
                              out_idx=draws[off:off + 1])
        else:
            sz.fill_(-1)
            sL.fill_(float("-inf"))
            for k in range(4):
                fs.fs_online_merge(sz, sL, z[k], L[k], k, seed=99, offset=off)
            draws[off:off + 1].copy_(sz)
    torch.cuda.synchronize()
    counts = np.bincount(draws.cpu().numpy(), minlength=V)
    _, _, pval = merge.chi_square_gof(counts, probs)
    assert pval > 1e-3, pval
