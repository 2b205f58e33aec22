"""Parity gate between a device result and the oracle.

TEST INFRASTRUCTURE (see ``oracle/__init__.py``).  Numpy only; it receives the
device outputs as arrays and never calls the device path itself.

The gate (fixed by the target this library is built to):
  - the sampled id equals the oracle's on every row whose oracle top-2 noisy
    score gap exceeds GAP (1e-2; the logit gap for greedy rows); on the other
    rows the device id must still be a near-maximum of the oracle's scores;
  - per-tile maxima agree within TOL_MAX (2e-3 absolute), per-tile argmaxes
    agree where the in-tile gap exceeds GAP, per-tile log-sum-exps agree
    within TOL_LSE (2e-3 absolute);
  - fully masked tiles/rows agree exactly (-inf / -1).
"""
from __future__ import annotations

import numpy as np

GAP = 1e-2
TOL_MAX = 2e-3
TOL_LSE = 2e-3
TILE = 128


class ParityError(AssertionError):
    pass


def check(ref, idx, tile_max=None, tile_idx=None, tile_lse=None, scores=None):
    """ref: dict from Oracle.sample for the rows compared (row order aligned
    with idx/tile_* arrays).  scores: optional oracle scores [n, V].
    Returns a dict of counts; raises ParityError on the first mismatch."""
    idx = np.asarray(idx).astype(np.int64)
    n = len(ref["idx"])
    stats = {"rows": n, "rows_gated": 0, "rows_exact": 0, "tiles": 0, "tiles_gated": 0,
             "max_abs_tile_max": 0.0, "max_abs_tile_lse": 0.0}
    for r in range(n):
        b = int(ref["rows"][r])
        want, got, gap = int(ref["idx"][r]), int(idx[r]), float(ref["gap"][r])
        if want < 0 or gap > GAP:
            stats["rows_gated"] += 1
            if got != want:
                raise ParityError(f"row {b}: sampled {got}, oracle {want} (gap {gap:.3g})")
            stats["rows_exact"] += 1
        else:
            _near_max(ref, r, got, scores)
            stats["rows_exact"] += int(got == want)
        if tile_max is None:
            continue
        rm, ri, rg = ref["tile_max"][r], ref["tile_idx"][r], ref["tile_gap"][r]
        gm, gi = np.asarray(tile_max[r], np.float64), np.asarray(tile_idx[r], np.int64)
        for t in range(len(rm)):
            stats["tiles"] += 1
            if ri[t] < 0:
                if gi[t] != -1 or not np.isneginf(gm[t]):
                    raise ParityError(f"row {b} tile {t}: masked tile reported ({gm[t]}, {gi[t]})")
                if tile_lse is not None and not np.isneginf(tile_lse[r][t]):
                    raise ParityError(f"row {b} tile {t}: masked tile lse {tile_lse[r][t]}")
                continue
            err = abs(gm[t] - rm[t])
            stats["max_abs_tile_max"] = max(stats["max_abs_tile_max"], float(err))
            if not err <= TOL_MAX:
                raise ParityError(f"row {b} tile {t}: max {gm[t]} vs oracle {rm[t]}")
            if rg[t] > GAP:
                stats["tiles_gated"] += 1
                if gi[t] != ri[t]:
                    raise ParityError(f"row {b} tile {t}: argmax {gi[t]} vs oracle {ri[t]} (gap {rg[t]:.3g})")
            elif not (t * TILE <= gi[t] < (t + 1) * TILE):
                raise ParityError(f"row {b} tile {t}: argmax {gi[t]} outside the tile")
            elif scores is not None and not scores[r][gi[t]] >= rm[t] - GAP:
                raise ParityError(f"row {b} tile {t}: argmax {gi[t]} is not a near-maximum")
            if tile_lse is not None:
                e2 = abs(float(tile_lse[r][t]) - ref["tile_lse"][r][t])
                stats["max_abs_tile_lse"] = max(stats["max_abs_tile_lse"], e2)
                if not e2 <= TOL_LSE:
                    raise ParityError(f"row {b} tile {t}: lse {tile_lse[r][t]} vs oracle {ref['tile_lse'][r][t]}")
    return stats


def _near_max(ref, r, got, scores):
    b = int(ref["rows"][r])
    top = np.max(ref["tile_max"][r])
    if got < 0:
        raise ParityError(f"row {b}: sampled -1 but the oracle has unmasked ids")
    if scores is not None:
        if not scores[r][got] >= top - GAP:
            raise ParityError(f"row {b}: sampled {got} (score {scores[r][got]}) not within {GAP} of max {top}")
        return
    t = got // TILE
    if t >= ref["tile_max"].shape[1] or not ref["tile_max"][r][t] >= top - GAP:
        raise ParityError(f"row {b}: sampled {got} lies in a tile far from the maximum")
    if ref["tile_idx"][r][t] != got and not ref["tile_gap"][r][t] <= GAP:
        raise ParityError(f"row {b}: sampled {got} is not its tile's near-maximum")
