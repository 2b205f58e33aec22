"""Group merges and goodness-of-fit helpers on top of the oracle's outputs.

TEST INFRASTRUCTURE (see ``oracle/__init__.py``).  Plain numpy, fp64.

The merges restate the exactness arguments of the FlashSampling pages:
  - ``partition_argmax``: the global argmax of the noisy scores equals the
    argmax over any partition of the local maxima (tomesphere abstract, "exact
    because argmax decomposes over partitions"; aitrends.kr write-up, the
    max-stability / decomposability paragraph);
  - ``lse_merge``: the log-mass of a union of groups is the log-sum-exp of the
    groups' log-masses L_k = log sum exp(l_i) (aitrends.kr, tensor-parallel
    paragraph);
  - ``group_gumbel_max``: pick group k with probability proportional to
    exp(L_k), then return that group's own sample z_k (aitrends.kr,
    Group-Gumbel-Max paragraph; "exact by hierarchical factorization" in the
    tomesphere abstract);
  - ``online_merge``: the O(1)-state streaming form of the same choice: on a
    new group (z', L'), L <- logaddexp(L, L') and z <- z' with probability
    exp(L' - L_new) (aitrends.kr, binary merge rule).
The random numbers these merges draw are passed in by the caller.
"""
from __future__ import annotations

import numpy as np


def partition_argmax(tile_max, tile_idx, bounds):
    """Argmax over partitions of per-tile winners.

    tile_max/tile_idx: [n_tiles] (one row).  bounds: increasing tile indices
    [0, t1, ..., n_tiles] delimiting the partitions.  Within a partition the
    local winner is the tile with the largest m_t (lowest tile on ties); the
    global winner is the partition winner with the largest m (lowest partition
    on ties).  Returns (index, max) with index -1 if everything is masked."""
    best_m, best_i = -np.inf, -1
    for p in range(len(bounds) - 1):
        lo, hi = bounds[p], bounds[p + 1]
        m_p, i_p = -np.inf, -1
        for t in range(lo, hi):
            if tile_idx[t] >= 0 and (i_p < 0 or tile_max[t] > m_p):
                m_p, i_p = tile_max[t], tile_idx[t]
        if i_p >= 0 and (best_i < 0 or m_p > best_m):
            best_m, best_i = m_p, i_p
    return int(best_i), float(best_m)


def lse_merge(lses):
    """log sum_k exp(L_k), stable; -inf for an empty or all -inf input."""
    a = np.asarray(lses, dtype=np.float64)
    if a.size == 0:
        return -np.inf
    m = np.max(a)
    if not np.isfinite(m):
        return float(m)
    return float(m + np.log(np.sum(np.exp(a - m))))


def group_gumbel_max(z, L, u):
    """Hierarchical draw: k = argmax_k (L_k - log(-log u_k)), return z_k.

    z: the groups' own samples; L: their log-masses; u: one fresh uniform in
    (0,1) per group (independent of the noise that produced z)."""
    z = np.asarray(z)
    L = np.asarray(L, dtype=np.float64)
    u = np.asarray(u, dtype=np.float64)
    keys = L - np.log(-np.log(u))
    keys = np.where(np.isfinite(L), keys, -np.inf)
    k = int(np.argmax(keys))
    if not np.isfinite(keys[k]):
        return -1
    return int(z[k])


def online_merge(z, L, u):
    """Stream groups one at a time with O(1) state (z, L).

    u[k] (k >= 1) is a fresh uniform for the Bernoulli switch at group k.
    Returns (z, L) after all groups."""
    cur_z, cur_L = int(z[0]), float(L[0])
    for k in range(1, len(z)):
        Lk = float(L[k])
        if not np.isfinite(Lk):
            continue
        new_L = np.logaddexp(cur_L, Lk)
        if u[k] < np.exp(Lk - new_L):
            cur_z = int(z[k])
        cur_L = float(new_L)
    return cur_z, cur_L


def chi_square_gof(counts, probs, min_expected=5.0):
    """Pearson chi-square goodness of fit of ``counts`` against ``probs``.

    Categories whose expected count is below ``min_expected`` are pooled into
    one bin.  Returns (statistic, degrees of freedom, p-value)."""
    from scipy.stats import chi2

    counts = np.asarray(counts, dtype=np.float64)
    probs = np.asarray(probs, dtype=np.float64)
    n = counts.sum()
    exp = probs * n
    big = exp >= min_expected
    obs_b = list(counts[big])
    exp_b = list(exp[big])
    if (~big).any():
        obs_b.append(counts[~big].sum())
        exp_b.append(exp[~big].sum())
    obs_b = np.asarray(obs_b)
    exp_b = np.asarray(exp_b)
    keep = exp_b > 0
    if np.any(obs_b[~keep] > 0):
        return np.inf, int(keep.sum() - 1), 0.0
    stat = float(np.sum((obs_b[keep] - exp_b[keep]) ** 2 / exp_b[keep]))
    dof = int(keep.sum() - 1)
    return stat, dof, float(chi2.sf(stat, dof)) if dof > 0 else 1.0
