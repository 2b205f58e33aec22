"""Seeded random configurations, CUDA path against the oracle element by element.

Each case draws a batch size (both kernels: single CTAs for up to 128 rows or
an odd number of 128-row blocks, CTA pairs for an even number), a hidden size
that is any multiple of 8 (ragged last K slice), a vocabulary size (ragged
last tile and unit), a temperature law (constant, per-row uniform, all or some
greedy rows), a mask density, per-row seeds or one seed, W outlier rows, an
offset anywhere in 64 bits and which per-tile outputs to write.  The
comparison is the one of the other parity tests (oracle/parity.py); the
top-K cases compare K draws without replacement the same way.
"""
import numpy as np
import pytest
import torch

import lm_head_gumbel_gb300 as fs
from gpu_cases import assert_no_device_error, compare, make_problem, run_device

pytestmark = pytest.mark.gpu

MAX_MACS = 2e9  # B * V * d per case: the oracle finishes each in a fraction of a second


def _cases(n, seed):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        kind = rng.integers(3)
        B = int(rng.integers(1, 9) if kind == 0 else rng.integers(9, 129) if kind == 1
                else rng.integers(129, 601))
        V = int(rng.integers(1, 6001))
        d = 8 * int(rng.integers(1, 141))
        while B * V * d > MAX_MACS and d > 8:
            d = max(8, (d // 2) // 8 * 8)
        if B * V * d > MAX_MACS:
            continue
        law = ["1.0", "0.5", "row-uniform", "greedy", "some-greedy"][int(rng.integers(5))]
        out.append(dict(
            B=B, d=d, V=V, law=law,
            mask_frac=[0.0, 0.05, 0.5][int(rng.integers(3))],
            per_row_seeds=bool(rng.integers(2)),
            outlier_frac=[0.0, 0.03][int(rng.integers(2))],
            tiles=bool(rng.integers(4) > 0), lse=bool(rng.integers(2)),
            seed=int(rng.integers(1 << 62)), offset=int(rng.integers(1 << 62)) * 4,
            case_seed=int(rng.integers(1 << 30))))
    return out


CASES = _cases(120, 20241202)
TOPK_CASES = _cases(36, 77)


def _problem(c):
    T, greedy = {"1.0": (1.0, 0.0), "0.5": (0.5, 0.0), "row-uniform": ("row-uniform", 0.0),
                 "greedy": (0.0, 0.0), "some-greedy": (0.9, 0.25)}[c["law"]]
    return make_problem(c["B"], c["d"], c["V"], T=T, greedy_frac=greedy,
                        mask_frac=c["mask_frac"], per_row_seeds=c["per_row_seeds"],
                        outlier_frac=c["outlier_frac"], seed=c["case_seed"])


def _id(c, topk=False):
    if topk:
        return (f"B{c['B']}-d{c['d']}-V{c['V']}-{c['law']}-m{c['mask_frac']}"
                f"{'-seeds' if c['per_row_seeds'] else ''}-K{1 + c['case_seed'] % 16}")
    return (f"B{c['B']}-d{c['d']}-V{c['V']}-{c['law']}-m{c['mask_frac']}"
            f"{'-seeds' if c['per_row_seeds'] else ''}{'-out' if c['outlier_frac'] else ''}"
            f"{'-tiles' if c['tiles'] else ''}{'-lse' if c['lse'] and c['tiles'] else ''}")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fs.load_library()
    yield
    assert_no_device_error()


@pytest.mark.parametrize("c", CASES, ids=[_id(c) for c in CASES])
def test_random_configuration(c):
    p = _problem(c)
    dev = run_device(p, seed=c["seed"], offset=c["offset"], tiles=c["tiles"],
                     lse=c["lse"] and c["tiles"])
    st = compare(p, dev, seed=c["seed"], offset=c["offset"], scores=True)  # raises on a mismatch
    assert st["rows"] == c["B"]


@pytest.mark.parametrize("c", TOPK_CASES, ids=[_id(c, True) for c in TOPK_CASES])
def test_random_topk_configuration(c):
    from test_gpu_topk import check_against_oracle, device_topk
    p = _problem(c)
    K = 1 + c["case_seed"] % 16
    idx, score = device_topk(p, K, seed=c["seed"], offset=c["offset"])
    check_against_oracle(p, K, idx, score, seed=c["seed"], offset=c["offset"])
    # the first draw is the sample of the same call
    one = fs.fs_sample(p["H"], p["W"], temperature=p["temperature"], vocab_mask=p["vocab_mask"],
                       seeds=p["seeds"], seed=c["seed"], offset=c["offset"]).cpu().numpy()
    assert np.array_equal(idx[:, 0], one)
