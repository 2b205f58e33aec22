"""Pins for the CPU oracle: each checks the oracle against something other than
itself -- published known-answer vectors, closed forms, numpy/scipy library
routines, brute force on tiny inputs, and distributional facts the
FlashSampling pages rest on (the Gumbel-max identity, argmax decomposition
over partitions, the group log-mass merge).

Every pin is a function ``pin_x(o)`` of an ``oracle.Oracle`` that raises
AssertionError on failure, so the same pins run against the real oracle
(test_oracle_pins.py) and against copies with a planted mistake
(test_oracle_mutants.py).
"""
from __future__ import annotations

import math
import os

import numpy as np
import scipy.special
import scipy.stats

from oracle import EULER_GAMMA, GUMBEL_VAR
from oracle.merge import (chi_square_gof, group_gumbel_max, lse_merge,
                          online_merge, partition_argmax)

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
P_MIN = 1e-3  # significance level of every goodness-of-fit pin


# ---- helpers ----------------------------------------------------------------
def bf16_to_f64(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f32_to_bf16_bits(x):
    """Round-to-nearest-even float32 -> bf16 bit patterns (input generation)."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def make_problem(B, d, V, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    H = f32_to_bf16_bits(rng.standard_normal((B, d)).astype(np.float32))
    W = f32_to_bf16_bits((rng.standard_normal((V, d)) * (2.0 / math.sqrt(d)) * scale).astype(np.float32))
    return H, W


def ref_logits(H, W):
    """The library fp64 matmul of the same bf16 values."""
    return bf16_to_f64(H) @ bf16_to_f64(W).T


def draws(o, H, W, n, T, seed=0, mask=None, row=0, start=0):
    """n samples of one row at offsets start..start+n-1."""
    B = H.shape[0]
    temp = np.full(B, T, dtype=np.float32)
    out = np.empty(n, dtype=np.int64)
    for i in range(n):
        out[i] = o.sample(H, W, temperature=temp, mask=mask, seed=seed,
                          offset=start + i, rows=[row])["idx"][0]
    return out


def pack_mask(allow):
    """bool [B, V] -> uint32 [B, ceil(V/32)] allow-bits."""
    B, V = allow.shape
    n = (V + 31) // 32
    pad = np.zeros((B, n * 32), dtype=bool)
    pad[:, :V] = allow
    w = (pad.reshape(B, n, 32).astype(np.uint64) << np.arange(32, dtype=np.uint64)).sum(-1)
    return w.astype(np.uint32)


# ---- Philox and the noise transform -------------------------------------
def pin_philox_kat(o):
    """Philox4x32-10 reproduces the published known-answer vectors."""
    path = os.path.join(GOLDEN, "philox4x32_10_kat.txt")
    n = 0
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        lhs, rhs = line.split("->")
        ins = [int(x, 16) for x in lhs.split()]
        want = [int(x, 16) for x in rhs.split()]
        got = [int(x) for x in o.philox(ins[:4], ins[4:6])]
        assert got == want, f"philox({lhs.strip()}) = {[hex(g) for g in got]}"
        n += 1
    assert n == 3


def pin_uniform_map(o):
    """u = ((w & 0x7fffff) + 1/2) 2^-23: endpoints, bit use, open interval."""
    assert o.uniform(0) == 2.0 ** -24
    assert o.uniform(0xFFFFFFFF) == 1.0 - 2.0 ** -24
    assert o.uniform(0xFF800000) == 2.0 ** -24       # top 9 bits unused
    assert o.uniform(0x1) == 3.0 * 2.0 ** -24
    assert o.uniform(0x400000) == 0.5 + 2.0 ** -24
    rng = np.random.default_rng(7)
    ws = rng.integers(0, 2 ** 32, size=2000, dtype=np.uint64)
    us = np.array([o.uniform(int(w)) for w in ws])
    assert np.all((us > 0) & (us < 1))
    # exact in fp32
    assert np.all(us.astype(np.float32).astype(np.float64) == us)


def pin_gumbel_closed_forms(o):
    """g(u) = -log(-log u): g(e^-1) = 0, and g inverts the Gumbel CDF."""
    assert abs(o.gumbel(math.exp(-1.0))) < 1e-15
    for x in (-2.0, -0.5, 0.0, 0.3, 1.0, 4.0, 9.0):
        u = math.exp(-math.exp(-x))
        assert abs(o.gumbel(u) - x) < 1e-9 * max(1.0, abs(x)) + 1e-12, x
    # monotone increasing
    us = np.linspace(0.001, 0.999, 101)
    gs = np.array([o.gumbel(u) for u in us])
    assert np.all(np.diff(gs) > 0)


def pin_noise_distribution(o):
    """Noise over a (row, vocab) grid is Gumbel(0,1): KS test, mean gamma,
    variance pi^2/6."""
    g = o.noise_grid(0, 64, 0, 4096, seed=12345, offset=7).ravel()
    n = g.size
    ks = scipy.stats.kstest(g, scipy.stats.gumbel_r.cdf)
    assert ks.pvalue > P_MIN, ks
    assert abs(g.mean() - EULER_GAMMA) < 5 * math.sqrt(GUMBEL_VAR / n)
    assert abs(g.var() - GUMBEL_VAR) < 0.03


def pin_noise_independence(o):
    """No two of (vocab index, row, offset, seed words, offset words) share
    noise: the streams that differ in exactly one of them are uncorrelated."""
    base = o.noise_grid(0, 8, 0, 4096, seed=99, offset=5)

    def corr(a, b):
        return float(np.corrcoef(a.ravel(), b.ravel())[0, 1])

    lim = 0.02
    # adjacent vocab indices (inside one Philox block of four and across)
    for shift in (1, 2, 3, 4):
        c = corr(base[:, :-shift], base[:, shift:])
        assert abs(c) < lim, ("vocab", shift, c)
    assert abs(corr(base[:-1], base[1:])) < lim                       # rows
    other = [
        o.noise_grid(0, 8, 0, 4096, seed=99, offset=6),               # offset
        o.noise_grid(0, 8, 0, 4096, seed=99, offset=5 + (1 << 32)),   # offset hi word
        o.noise_grid(0, 8, 0, 4096, seed=100, offset=5),              # seed
        o.noise_grid(0, 8, 0, 4096, seed=99 + (1 << 32), offset=5),   # seed hi word
    ]
    for k, x in enumerate(other):
        c = corr(base, x)
        assert abs(c) < lim, (k, c)
    # per-row seeds: row b takes seeds[b]
    seeds = np.array([99, 99 + (1 << 40), 7, 99], dtype=np.uint64)
    ps = o.noise_grid(0, 4, 0, 256, seeds=seeds, offset=5)
    assert np.array_equal(ps[0], base[0, :256])
    assert np.array_equal(ps[3], base[3, :256])
    assert abs(corr(ps[1], base[1, :256])) < 0.25


# ---- logits, greedy, tiles ------------------------------------------------
def pin_logits_match_numpy(o):
    """fp64 logits equal numpy's fp64 matmul of the same bf16 values."""
    H, W = make_problem(5, 72, 300, seed=1)
    got = o.logits(H, W)
    want = ref_logits(H, W)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12)
    s = o.sample(H, W, temperature=np.zeros(5, np.float32), want_logits=True)
    assert np.allclose(s["logits"], want, rtol=1e-12, atol=1e-12)


def pin_greedy_is_argmax(o):
    """T = 0 (and T < 0, NaN, inf) is greedy: numpy.argmax of the fp64
    logits, lowest index on exact ties, with per-tile maxima of the logits."""
    B, d, V = 6, 32, 700
    H, W = make_problem(B, d, V, seed=2)
    W[513] = W[2]            # exact duplicates -> exact logit ties,
    W[640] = W[129]          # in another tile and in the same tile
    W[130] = W[129]
    L = ref_logits(H, W)
    for T in (0.0, -1.0, float("nan"), float("inf")):
        r = o.sample(H, W, temperature=np.full(B, T, np.float32), seed=3, offset=4)
        assert np.array_equal(r["idx"], np.argmax(L, axis=1)), T
        for t in range((V + 127) // 128):
            blk = L[:, t * 128:(t + 1) * 128]
            assert np.array_equal(r["tile_idx"][:, t], t * 128 + np.argmax(blk, axis=1))
            assert np.allclose(r["tile_max"][:, t], blk.max(axis=1), rtol=1e-12, atol=1e-12)
            assert np.allclose(r["tile_lse"][:, t], blk.max(axis=1), rtol=1e-12, atol=1e-12)
    # tie rule, forced: make row 0's best logit tie across tiles
    H1 = H[:1].copy()
    W2 = W.copy()
    best = int(np.argmax(L[0]))
    W2[699] = W2[best]
    W2[best + 1 if best + 1 < 699 else best - 1] = W2[best]
    r = o.sample(H1, W2, temperature=np.zeros(1, np.float32))
    L2 = ref_logits(H1, W2)[0]
    assert r["idx"][0] == np.argmax(L2)
    for t in range((V + 127) // 128):   # the tie inside best's tile included
        assert r["tile_idx"][0, t] == t * 128 + np.argmax(L2[t * 128:(t + 1) * 128])


def pin_tile_outputs(o):
    """Per-tile (max, argmax, log-sum-exp, top-2 gap) against brute force
    over the scores, with library logsumexp over the numpy logits; a ragged
    last tile, a masked-out tile and masked entries included."""
    B, d, V, T = 3, 24, 1000, float(np.float32(0.7))
    H, W = make_problem(B, d, V, seed=3)
    allow = np.ones((B, V), dtype=bool)
    rng = np.random.default_rng(0)
    allow &= rng.random((B, V)) > 0.1
    allow[1, 256:384] = False            # a fully masked tile
    mask = pack_mask(allow)
    r = o.sample(H, W, temperature=np.full(B, T, np.float32), mask=mask,
                 seed=5, offset=11, want_scores=True, want_logits=True)
    L = ref_logits(H, W)
    assert np.allclose(r["logits"], L, rtol=1e-12, atol=1e-12)
    S = r["scores"]
    assert np.all(np.isneginf(S[~allow]))
    assert np.all(np.isfinite(S[allow]))
    g = o.noise_grid(0, B, 0, V, seed=5, offset=11)
    assert np.allclose(S[allow], (L / T + g)[allow], rtol=1e-12, atol=1e-12)
    nt = (V + 127) // 128
    for b in range(B):
        for t in range(nt):
            lo, hi = t * 128, min(V, t * 128 + 128)
            s = S[b, lo:hi]
            ok = allow[b, lo:hi]
            if not ok.any():
                assert r["tile_idx"][b, t] == -1
                assert np.isneginf(r["tile_max"][b, t]) and np.isneginf(r["tile_lse"][b, t])
                continue
            assert r["tile_idx"][b, t] == lo + int(np.argmax(s))
            assert r["tile_max"][b, t] == s.max()
            top2 = np.sort(s[ok])[-2:]
            assert np.isclose(r["tile_gap"][b, t], top2[1] - top2[0], rtol=1e-12, atol=1e-12)
            lse = scipy.special.logsumexp(L[b, lo:hi][ok] / T)
            assert np.isclose(r["tile_lse"][b, t], lse, rtol=1e-12, atol=1e-12)
        assert r["idx"][b] == int(np.argmax(S[b]))
        top2 = np.sort(S[b][allow[b]])[-2:]
        assert np.isclose(r["gap"][b], top2[1] - top2[0], rtol=1e-12, atol=1e-12)
    # large logits: the log-sum-exp must not overflow
    Hb, Wb = make_problem(1, 16, 256, seed=4, scale=300.0)
    rb = o.sample(Hb, Wb, temperature=np.full(1, 0.5, np.float32))
    Lb = ref_logits(Hb, Wb)
    for t in range(2):
        want = scipy.special.logsumexp(Lb[0, t * 128:(t + 1) * 128] / 0.5)
        assert np.isfinite(rb["tile_lse"][0, t]) and np.isclose(rb["tile_lse"][0, t], want, rtol=1e-12)


def pin_fully_masked_row(o):
    """A row with every entry masked samples -1; other rows are unaffected."""
    H, W = make_problem(2, 16, 300, seed=6)
    allow = np.ones((2, 300), dtype=bool)
    allow[0] = False
    r = o.sample(H, W, mask=pack_mask(allow), seed=1)
    r2 = o.sample(H, W, seed=1)
    assert r["idx"][0] == -1 and np.all(r["tile_idx"][0] == -1)
    assert r["idx"][1] == r2["idx"][1]


def pin_partition_invariance(o):
    """The argmax decomposes over partitions: tiles of any width and any
    grouping of tiles give the flat argmax, bit for bit."""
    B, d, V = 4, 16, 777
    H, W = make_problem(B, d, V, seed=7)
    T = np.full(B, 0.9, np.float32)
    flat = o.sample(H, W, temperature=T, seed=8, offset=3, tile=V, want_scores=True)
    assert np.array_equal(flat["idx"], np.argmax(flat["scores"], axis=1))
    rng = np.random.default_rng(1)
    for tile in (1, 7, 64, 128, 500):
        r = o.sample(H, W, temperature=T, seed=8, offset=3, tile=tile)
        nt = r["tile_max"].shape[1]
        assert np.array_equal(r["idx"], flat["idx"])
        for b in range(B):
            for _ in range(4):
                cuts = np.sort(rng.choice(np.arange(1, nt), size=min(3, nt - 1), replace=False)) if nt > 1 else []
                bounds = [0, *cuts.tolist(), nt] if nt > 1 else [0, nt]
                i, m = partition_argmax(r["tile_max"][b], r["tile_idx"][b], bounds)
                assert i == flat["idx"][b] and m == flat["scores"][b].max()


def pin_lse_merge(o):
    """log-sum-exp of the tile log-masses is the whole row's log-mass."""
    B, d, V, T = 3, 16, 1000, float(np.float32(1.3))
    H, W = make_problem(B, d, V, seed=9)
    r = o.sample(H, W, temperature=np.full(B, T, np.float32))
    L = ref_logits(H, W)
    for b in range(B):
        assert np.isclose(lse_merge(r["tile_lse"][b]),
                          scipy.special.logsumexp(L[b] / T), rtol=1e-12, atol=1e-12)
    # large logits: the merge of tile log-masses near 1e3 must not overflow
    Hb, Wb = make_problem(1, 16, 512, seed=4, scale=300.0)
    rb = o.sample(Hb, Wb, temperature=np.full(1, 0.5, np.float32))
    Lb = ref_logits(Hb, Wb)[0]
    assert np.max(rb["tile_lse"][0]) > 800.0
    got = lse_merge(rb["tile_lse"][0])
    assert np.isfinite(got) and np.isclose(got, scipy.special.logsumexp(Lb / 0.5), rtol=1e-12)
    assert lse_merge([-np.inf, -np.inf]) == -np.inf and lse_merge([]) == -np.inf


# ---- distribution ------------------------------------------------------------
def pin_chi_square_softmax(o):
    """Seeded draws follow softmax(l / T) exactly (Pearson chi-square)."""
    for (V, d, T, n, seed) in ((16, 16, 0.7, 20000, 11), (64, 8, 1.0, 20000, 12)):
        H, W = make_problem(1, d, V, seed=seed)
        p = scipy.special.softmax(ref_logits(H, W)[0] / T)
        idx = draws(o, H, W, n, T, seed=seed)
        counts = np.bincount(idx, minlength=V)
        stat, dof, pval = chi_square_gof(counts, p)
        assert pval > P_MIN, (V, T, stat, dof, pval)


def pin_two_way_closed_form(o):
    """V = 2: P(token 0) = sigmoid((l0 - l1) / T) (binomial z-test)."""
    H, W = make_problem(1, 8, 2, seed=13)
    L = ref_logits(H, W)[0]
    T, n = 0.6, 20000
    p0 = 1.0 / (1.0 + math.exp(-(L[0] - L[1]) / T))
    k = int(np.sum(draws(o, H, W, n, T, seed=21) == 0))
    z = (k - n * p0) / math.sqrt(n * p0 * (1 - p0))
    assert abs(z) < 4.5, (k, n * p0, z)


def pin_max_stability(o):
    """Max-stability: m_t - L_t ~ Gumbel(0,1) for every tile, over draws."""
    H, W = make_problem(1, 16, 256, seed=14)
    T = np.full(1, 0.8, np.float32)
    n = 6000
    diffs = []
    for off in range(n):
        r = o.sample(H, W, temperature=T, seed=77, offset=off)
        diffs.append(r["tile_max"][0] - r["tile_lse"][0])
    diffs = np.asarray(diffs)
    for t in range(diffs.shape[1]):
        x = diffs[:, t]
        assert abs(x.mean() - EULER_GAMMA) < 4.5 * math.sqrt(GUMBEL_VAR / n), (t, x.mean())
        ks = scipy.stats.kstest(x, scipy.stats.gumbel_r.cdf)
        assert ks.pvalue > P_MIN, (t, ks)


def pin_merge_uniform(o):
    """The merge uniforms: Philox on their own counter domain (second word
    row | 2^31), uniform on (0,1), uncorrelated with the sampling noise of the
    same (row, index), and exact in fp32."""
    seed, off = 4242, (3 << 32) + 17
    for b, k in ((0, 0), (5, 3), (7, 9), (1000, 4)):
        w = o.philox([k >> 2, b | 0x80000000, off & 0xFFFFFFFF, off >> 32],
                     [seed & 0xFFFFFFFF, seed >> 32])[k & 3]
        assert o.merge_uniform(seed, off, b, k) == o.uniform(int(w))
    us = np.array([[o.merge_uniform(seed, off, b, k) for k in range(512)] for b in range(16)])
    assert np.all((us > 0) & (us < 1))
    ks = scipy.stats.kstest(us.ravel(), "uniform")
    assert ks.pvalue > P_MIN, ks
    words = np.array([[o.noise_word(seed, off, b, k) for k in range(512)] for b in range(16)])
    samp = (words & 0x7FFFFF).astype(np.float64)
    assert abs(np.corrcoef(us.ravel(), samp.ravel())[0, 1]) < 0.02


def pin_group_merges(o):
    """Group-Gumbel-Max and the online binary merge over 4 vocabulary groups,
    fed the groups' own samples and log-masses, follow softmax(l / T)."""
    V, d, T, n = 64, 8, 0.9, 12000
    H, W = make_problem(1, d, V, seed=15)
    p = scipy.special.softmax(ref_logits(H, W)[0] / T)
    rng = np.random.default_rng(2)
    temp = np.full(1, T, np.float32)
    hier, online = [], []
    for off in range(n):
        r = o.sample(H, W, temperature=temp, seed=31, offset=off, tile=16)
        z, L = r["tile_idx"][0], r["tile_lse"][0]
        hier.append(group_gumbel_max(z, L, rng.random(4)))
        online.append(online_merge(z, L, rng.random(4))[0])
    for name, idx in (("group", hier), ("online", online)):
        counts = np.bincount(np.asarray(idx), minlength=V)
        stat, dof, pval = chi_square_gof(counts, p)
        assert pval > P_MIN, (name, stat, dof, pval)


def pin_masked_distribution(o):
    """With a mask, draws follow softmax over the allowed tokens only."""
    V, d, T, n = 40, 8, 1.0, 15000
    H, W = make_problem(1, d, V, seed=16)
    allow = np.ones((1, V), dtype=bool)
    allow[0, [0, 3, 17, 18, 33]] = False
    Lg = ref_logits(H, W)[0] / T
    Lg[~allow[0]] = -np.inf
    p = scipy.special.softmax(Lg)
    idx = draws(o, H, W, n, T, seed=41, mask=pack_mask(allow))
    assert np.all(allow[0, idx])
    stat, dof, pval = chi_square_gof(np.bincount(idx, minlength=V)[allow[0]], p[allow[0]])
    assert pval > P_MIN, (stat, dof, pval)


def pin_topk_first_is_sample_and_greedy_sort(o):
    """The first of the K largest scores is the sample; for greedy rows the K
    are numpy's descending sort of the fp64 logits (lowest id on ties)."""
    from oracle import sample_topk
    B, d, V = 5, 24, 700
    H, W = make_problem(B, d, V, seed=41)
    W[650] = W[3]  # an exact tie
    T = np.array([0.8, 1.0, 0.0, 1.3, 0.0], np.float32)
    idx, val, ref = sample_topk(o, H, W, 6, temperature=T, seed=2, offset=3)
    assert np.array_equal(idx[:, 0], ref["idx"])
    assert np.all(np.diff(val, axis=1) <= 0)
    L = ref_logits(H, W)
    for b in (2, 4):
        order = np.lexsort((np.arange(V), -L[b]))[:6]
        assert np.array_equal(idx[b], order)


def pin_topk_plackett_luce(o):
    """Two draws without replacement: P(first = i, second = j) =
    p_i p_j / (1 - p_i) with p = softmax(l / T) (chi-square over ordered pairs)."""
    from oracle import topk_from_scores
    V, d, T, n = 6, 8, 1.0, 12000
    H, W = make_problem(1, d, V, seed=42)
    p = scipy.special.softmax(ref_logits(H, W)[0] / T)
    temp = np.full(1, T, np.float32)
    counts = np.zeros((V, V))
    for off in range(n):
        r = o.sample(H, W, temperature=temp, seed=5, offset=off, want_scores=True)
        ij, _ = topk_from_scores(r["scores"], 2)
        counts[ij[0, 0], ij[0, 1]] += 1
    want = np.array([[p[i] * p[j] / (1 - p[i]) if i != j else 0.0 for j in range(V)]
                     for i in range(V)])
    off_diag = ~np.eye(V, dtype=bool)
    assert counts[~off_diag].sum() == 0
    _, _, pval = chi_square_gof(counts[off_diag], want[off_diag])
    assert pval > P_MIN, pval


# ---- the goodness-of-fit instrument and the merges themselves ---------------
def pin_chi_square_instrument(o):
    """The chi-square helper every distributional pin and GPU test relies on.

    Without pooling it must reproduce scipy.stats.chisquare (statistic and
    p-value); a pooled case worked by hand must give its closed form (two
    degrees of freedom: p = exp(-x/2)); a count in a zero-probability
    category must reject outright; and at the pins' own sample size it must
    reject draws from a law a little off softmax(l / T) -- a flatter
    temperature, or two probabilities swapped -- while accepting draws from
    softmax(l / T) itself.  (The draws here come from numpy's multinomial, not
    from the oracle.)"""
    rng = np.random.default_rng(2024)
    # unpooled: every expected count >= 5
    for V, n in ((16, 20000), (64, 20000), (5, 300)):
        p = rng.dirichlet(np.full(V, 4.0))
        p = np.maximum(p, 0.01)
        p /= p.sum()
        counts = rng.multinomial(n, p)
        stat, dof, pval = chi_square_gof(counts, p)
        ref = scipy.stats.chisquare(counts, p * n)
        assert dof == V - 1, (V, dof)
        assert math.isclose(stat, ref.statistic, rel_tol=1e-12, abs_tol=1e-12), (stat, ref)
        assert math.isclose(pval, ref.pvalue, rel_tol=1e-10, abs_tol=1e-300), (pval, ref)
    # pooled, by hand: n = 100, expected (60, 30, 4, 3, 3) -> bins (60, 30, 10);
    # observed (55, 32, 5, 4, 4) -> (55, 32, 13);
    # x = 25/60 + 4/30 + 9/10 = 1.45 on 2 degrees of freedom, p = exp(-0.725)
    stat, dof, pval = chi_square_gof([55, 32, 5, 4, 4], [0.6, 0.3, 0.04, 0.03, 0.03])
    assert dof == 2 and math.isclose(stat, 1.45, rel_tol=1e-12), (stat, dof)
    assert math.isclose(pval, math.exp(-0.725), rel_tol=1e-12), pval
    # an impossible outcome observed
    stat, dof, pval = chi_square_gof([10, 10, 1], [0.5, 0.5, 0.0])
    assert pval == 0.0, (stat, dof, pval)
    # the pins' own laws: accept the law, reject a nearby one
    for (V, d, T, seed) in ((16, 16, 0.7, 11), (64, 8, 1.0, 12)):
        H, W = make_problem(1, d, V, seed=seed)
        lg = ref_logits(H, W)[0]
        p = scipy.special.softmax(lg / T)
        n = 20000
        _, _, p_ok = chi_square_gof(rng.multinomial(n, p), p)
        assert p_ok > P_MIN, (V, p_ok)
        flat = scipy.special.softmax(lg / (1.15 * T))
        _, _, p_flat = chi_square_gof(rng.multinomial(n, flat), p)
        assert p_flat < P_MIN, (V, "flatter law accepted", p_flat)
        order = np.argsort(p)
        swapped = p.copy()
        hi, mid = order[-1], order[V // 2]
        swapped[hi], swapped[mid] = p[mid], p[hi]
        _, _, p_swap = chi_square_gof(rng.multinomial(n, swapped), p)
        assert p_swap < P_MIN, (V, "swapped law accepted", p_swap)


def pin_group_gumbel_max_law(o):
    """Group-Gumbel-Max picks group k with probability exp(L_k) / sum exp(L)
    (hierarchical factorisation of the categorical): four groups of unequal
    mass, fresh uniforms from numpy, counts against that law with scipy's
    chi-square; a shift of every L_k changes nothing; a group of zero mass is
    never picked, and with no group left the draw is -1."""
    rng = np.random.default_rng(5)
    p = np.array([0.55, 0.25, 0.12, 0.08])
    z = np.array([101, 202, 303, 404])
    n = 20000
    for shift in (0.0, 700.0, -300.0):
        L = np.log(p) + shift
        picks = np.array([group_gumbel_max(z, L, rng.random(4)) for _ in range(n)])
        counts = np.array([np.sum(picks == zk) for zk in z])
        assert counts.sum() == n
        pval = scipy.stats.chisquare(counts, p * n).pvalue
        assert pval > P_MIN, (shift, counts, pval)
    L = np.array([np.log(0.5), -np.inf, np.log(0.5), -np.inf])
    picks = {group_gumbel_max(z, L, rng.random(4)) for _ in range(500)}
    assert picks == {101, 303}, picks
    assert group_gumbel_max(z, np.full(4, -np.inf), rng.random(4)) == -1


def pin_online_merge_law(o):
    """The online binary merge ends in group k with probability
    exp(L_k) / sum exp(L) whatever the order the groups arrive in, and its
    running log-mass ends at scipy's logsumexp of the L_k; groups of zero
    mass leave the state alone."""
    rng = np.random.default_rng(6)
    p = np.array([0.1, 0.45, 0.05, 0.25, 0.15])
    z = np.arange(10, 15)
    L = np.log(p) + 3.0
    n = 20000
    finals = np.empty(n, dtype=np.int64)
    for i in range(n):
        zi, Li = online_merge(z, L, rng.random(len(z)))
        finals[i] = zi
    assert math.isclose(Li, scipy.special.logsumexp(L), rel_tol=1e-12, abs_tol=1e-12), Li
    counts = np.bincount(finals - 10, minlength=len(z))
    pval = scipy.stats.chisquare(counts, p * n).pvalue
    assert pval > P_MIN, (counts, pval)
    zl, Ll = online_merge([7, 8, 9], [0.0, -np.inf, -np.inf], rng.random(3))
    assert zl == 7 and Ll == 0.0


def pin_partition_ties(o):
    """Exact ties between tiles and between partitions (greedy rows with
    duplicated W rows) resolve to the lowest id, as numpy.argmax's first
    occurrence does: the partition merge keeps the earlier tile and the
    earlier partition."""
    B, d, V = 3, 16, 1024
    H, W = make_problem(B, d, V, seed=17)
    L0 = ref_logits(H, W)
    for b in range(B):
        best = int(np.argmax(L0[b]))
        # copies of the row's best W row in later tiles and later partitions
        for v in (best + 1, 300, 640, 1023):
            if v > best:
                W[v] = W[best]
    L = ref_logits(H, W)
    r = o.sample(H, W, temperature=np.zeros(B, np.float32))
    nt = r["tile_max"].shape[1]
    for b in range(B):
        want = int(np.argmax(L[b]))
        assert r["idx"][b] == want
        for bounds in ([0, nt], [0, 1, nt], [0, 2, 3, 5, nt], list(range(nt + 1))):
            i, m = partition_argmax(r["tile_max"][b], r["tile_idx"][b], bounds)
            assert i == want, (b, bounds, i, want)


ALL_PINS = [
    pin_chi_square_instrument,
    pin_philox_kat,
    pin_uniform_map,
    pin_gumbel_closed_forms,
    pin_logits_match_numpy,
    pin_greedy_is_argmax,
    pin_tile_outputs,
    pin_fully_masked_row,
    pin_partition_invariance,
    pin_partition_ties,
    pin_lse_merge,
    pin_group_gumbel_max_law,
    pin_online_merge_law,
    pin_noise_distribution,
    pin_noise_independence,
    pin_two_way_closed_form,
    pin_chi_square_softmax,
    pin_masked_distribution,
    pin_max_stability,
    pin_group_merges,
    pin_merge_uniform,
    pin_topk_first_is_sample_and_greedy_sort,
    pin_topk_plackett_luce,
]
