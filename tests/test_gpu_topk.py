"""K draws without replacement (Gumbel-top-k) on the GPU, against the oracle.

The ids of the K largest noisy scores per row, best first: the first equals
fs_sample's draw; the list matches the oracle where the oracle's consecutive
score gaps exceed the parity gate; the ordered pairs follow the
Plackett-Luce law p_i p_j / (1 - p_i) (chi-square); masked ids never appear
and short rows pad with -1.
"""
import numpy as np
import pytest
import scipy.special
import torch

import lm_head_gumbel_gb300 as fs
from lm_head_gumbel_gb300 import workloads as wl
import oracle
from oracle import merge, parity, sample_topk
from gpu_cases import assert_no_device_error, make_problem

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fs.load_library()
    yield
    assert_no_device_error()


def device_topk(p, K, *, seed=7, offset=0):
    B = p["H"].shape[0]
    score = torch.empty((B, K), dtype=torch.float32, device="cuda")
    idx = fs.fs_sample_topk(p["H"], p["W"], K, temperature=p["temperature"],
                            vocab_mask=p["vocab_mask"], seeds=p["seeds"], seed=seed,
                            offset=offset, out_topk_score=score)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), score.cpu().numpy()


def check_against_oracle(p, K, idx, score, rows=None, *, seed=7, offset=0):
    o = oracle.default()
    ridx, rval, ref = sample_topk(
        o, wl.bf16_bits(p["H"]), wl.bf16_bits(p["W"]), K + 1,
        temperature=p["temperature"].cpu().numpy(),
        mask=None if p["vocab_mask"] is None else wl.u32_bits(p["vocab_mask"]),
        seeds=None if p["seeds"] is None else wl.u64_bits(p["seeds"]), seed=seed,
        offset=offset, rows=rows)
    sel = ref["rows"]
    n_exact = 0
    for r, b in enumerate(sel):
        with np.errstate(invalid="ignore"):
            gaps = -np.diff(rval[r])  # s(j) - s(j+1), j = 0..K-1 (nan past the count)
        for j in range(K):
            if ridx[r, j] < 0:
                assert idx[b, j] == -1
                continue
            assert abs(score[b, j] - rval[r, j]) <= parity.TOL_MAX, (b, j)
            left_ok = j == 0 or gaps[j - 1] > parity.GAP
            if left_ok and gaps[j] > parity.GAP:
                assert idx[b, j] == ridx[r, j], (b, j)
                n_exact += 1
    return n_exact


@pytest.mark.parametrize("K", [1, 3, 4, 8, 16])
def test_topk_matches_oracle_and_first_is_the_sample(K):
    p = make_problem(20, 128, 3000, T="row-uniform", per_row_seeds=True, mask_frac=0.03,
                     seed=40 + K)
    idx, score = device_topk(p, K, offset=3)
    one = fs.fs_sample(p["H"], p["W"], temperature=p["temperature"], vocab_mask=p["vocab_mask"],
                       seeds=p["seeds"], seed=7, offset=3)
    torch.cuda.synchronize()
    assert np.array_equal(idx[:, 0], one.cpu().numpy())
    assert np.all(np.diff(score, axis=1) <= 0)
    for b in range(idx.shape[0]):  # distinct ids
        got = idx[b][idx[b] >= 0]
        assert len(set(got.tolist())) == len(got)
    assert check_against_oracle(p, K, idx, score, offset=3) > 0.8 * 20 * K


def test_topk_short_rows_and_masks():
    p = make_problem(4, 64, 1000, T=1.0, mask_frac=0.02, seed=50)
    m = p["vocab_mask"]
    m[1, :] = 0
    m[1, 3] = 0b1011  # three allowed ids: 96, 97, 99
    m[2, :] = 0       # nothing allowed
    idx, score = device_topk(p, 8, offset=1)
    assert set(idx[1, :3].tolist()) == {96, 97, 99} and np.all(idx[1, 3:] == -1)
    assert np.all(np.isneginf(score[1, 3:]))
    assert np.all(idx[2] == -1)
    mm = m.cpu().numpy().view(np.uint32)
    for b in (0, 3):
        bits = (mm[b, idx[b] // 32] >> (idx[b] % 32)) & 1
        assert np.all(bits == 1)
    check_against_oracle(p, 8, idx, score, offset=1)


def test_topk_pairs_follow_plackett_luce():
    V, d, T, n = 8, 16, 1.0, 6000
    p = make_problem(1, d, V, T=T, seed=51)
    probs = scipy.special.softmax(
        oracle.default().logits(wl.bf16_bits(p["H"]), wl.bf16_bits(p["W"]))[0] / T)
    out = torch.empty((n, 2), dtype=torch.int64, device="cuda")
    ws = torch.empty(fs.fs_topk_workspace_size(1, V, 2), dtype=torch.uint8, device="cuda")
    for off in range(n):
        fs.fs_sample_topk(p["H"], p["W"], 2, temperature=p["temperature"], seed=11, offset=off,
                          out_topk_idx=out[off:off + 1], workspace=ws)
    torch.cuda.synchronize()
    pairs = out.cpu().numpy()
    counts = np.zeros((V, V))
    np.add.at(counts, (pairs[:, 0], pairs[:, 1]), 1)
    want = np.array([[probs[i] * probs[j] / (1 - probs[i]) if i != j else 0.0
                      for j in range(V)] for i in range(V)])
    off_diag = ~np.eye(V, dtype=bool)
    assert counts[~off_diag].sum() == 0
    _, _, pval = merge.chi_square_gof(counts[off_diag], want[off_diag])
    assert pval > 1e-3, pval


def test_topk_on_a_vocabulary_shard():
    """K draws on a shard W[v0:v1] sampled with vocab_offset = v0 return
    global ids, and are the K best of the full row's scores restricted to
    the shard (the oracle's scores of the whole vocabulary, sliced)."""
    B, d, V, K, v0, v1 = 12, 64, 4096, 8, 1024, 3072
    p = make_problem(B, d, V, T="row-uniform", per_row_seeds=True, seed=61)
    out = torch.empty((B, K), dtype=torch.int64, device="cuda")
    score = torch.empty((B, K), dtype=torch.float32, device="cuda")
    fs.fs_sample_topk(p["H"], p["W"][v0:v1], K, temperature=p["temperature"], seeds=p["seeds"],
                      seed=7, offset=5, vocab_offset=v0, out_topk_idx=out, out_topk_score=score)
    torch.cuda.synchronize()
    idx, sc = out.cpu().numpy(), score.cpu().numpy()
    assert np.all((idx >= v0) & (idx < v1))
    o = oracle.default()
    ref = o.sample(wl.bf16_bits(p["H"]), wl.bf16_bits(p["W"]),
                   temperature=p["temperature"].cpu().numpy(), seeds=wl.u64_bits(p["seeds"]),
                   seed=7, offset=5, want_scores=True)
    ridx, rval = oracle.topk_from_scores(ref["scores"][:, v0:v1], K + 1)
    for b in range(B):
        gaps = -np.diff(rval[b])
        for j in range(K):
            assert abs(sc[b, j] - rval[b, j]) <= parity.TOL_MAX, (b, j)
            if (j == 0 or gaps[j - 1] > parity.GAP) and gaps[j] > parity.GAP:
                assert idx[b, j] == v0 + ridx[b, j], (b, j)


@pytest.mark.parametrize("B,V", [(384, 5000), (512, 3000), (136, 40000), (1024, 40000)])
def test_topk_rows_changing_between_units(B, V):
    """Batches whose epilogue threads change rows from unit to unit (three
    128-row blocks on single CTAs) or run long stretches of one row (136
    rows, 313 tiles; and the CTA pairs' grouped order, where a pair keeps one
    batch block: two pair blocks of one unit a pair, and four pair blocks over
    157 vocabulary blocks -- groups walking 9 blocks each plus leftover pairs
    taking the last blocks one batch block after the other): the running
    per-thread lists are flushed at every row change; every row's first id is
    fs_sample's, no row repeats an id, and sampled rows of every batch block
    match the oracle."""
    K = 16
    p = make_problem(B, 64, V, T="row-uniform", per_row_seeds=True, seed=60 + B)
    idx, score = device_topk(p, K, offset=4)
    one = fs.fs_sample(p["H"], p["W"], temperature=p["temperature"], seeds=p["seeds"], seed=7,
                       offset=4)
    torch.cuda.synchronize()
    assert np.array_equal(idx[:, 0], one.cpu().numpy())
    assert np.all(np.diff(score, axis=1) <= 0)
    for b in range(B):
        got = idx[b][idx[b] >= 0]
        assert len(set(got.tolist())) == len(got) == K
    rows = sorted({r for r in (0, 127, 128, 255, 256, 511, 512, 767, 768, B - 1) if r < B})
    assert check_against_oracle(p, K, idx, score, rows=rows, offset=4) >= len(rows) * K * 0.7


@pytest.mark.parametrize("B,K", [(64, 8), (256, 16), (512, 16)])
def test_topk_full_size_head(B, K):
    """Qwen3-8B-shaped head (d=4096, V=151936): the single-CTA kernel (B=64)
    and the CTA-pair kernel in top-K mode (B=256; B=512 in the grouped order:
    37 groups of two pairs walk 16 vocabulary blocks each and the pair left
    over takes the last two, both batch blocks); sampled rows against the
    oracle, every row's first id against fs_sample."""
    w = wl.WORKLOADS["qwen3-8b"]
    W = wl.make_weights(w.d, w.V, seed=77, device="cuda")
    p = make_problem(B, w.d, w.V, T="row-uniform", per_row_seeds=True, seed=B, W=W)
    idx, score = device_topk(p, K, offset=2)
    one = fs.fs_sample(p["H"], W, temperature=p["temperature"], seeds=p["seeds"], offset=2,
                       seed=7)
    torch.cuda.synchronize()
    assert np.array_equal(idx[:, 0], one.cpu().numpy())
    assert np.all((idx >= 0) & (idx < w.V))
    for b in range(B):
        assert len(set(idx[b].tolist())) == K, b
    rows = [0, B // 3, B - 1]
    assert check_against_oracle(p, K, idx, score, rows=rows, offset=2) >= len(rows) * K * 0.6


@pytest.mark.parametrize("name,B,K", [("qwen3-8b", 64, 16), ("qwen3-1.7b", 256, 4)])
def test_topk_whole_batch_against_oracle(name, B, K):
    """Every row of a production-shaped batch against the oracle's fp64
    top-K (gap-gated): the Qwen3-8B head at the benchmark's top-K leg (B = 64,
    K = 16, the single-CTA kernel, whose last units read their noise made
    ahead) and the Qwen3-1.7B head at B = 256 (the CTA-pair kernel); every
    row's first id against fs_sample."""
    w = wl.WORKLOADS[name]
    W = wl.make_weights(w.d, w.V, seed=77, device="cuda")
    p = make_problem(B, w.d, w.V, T="row-uniform", per_row_seeds=True, seed=160 + B, W=W)
    idx, score = device_topk(p, K, offset=9)
    one = fs.fs_sample(p["H"], W, temperature=p["temperature"], seeds=p["seeds"], offset=9,
                       seed=7)
    torch.cuda.synchronize()
    assert np.array_equal(idx[:, 0], one.cpu().numpy())
    for b in range(B):
        assert len(set(idx[b].tolist())) == K, b
    n_exact = check_against_oracle(p, K, idx, score, rows=list(range(B)), offset=9)
    assert n_exact >= B * K * 0.6


@pytest.mark.parametrize("K", [4, 16])
def test_topk_equal_scores_take_the_lowest_ids(K):
    """Every logit of a row equal (all W rows the same): greedy rows tie on
    every id, so their K draws are ids 0..K-1 (the tie rule), and so many
    entries reach the reduction's threshold that it merges every list; sampled
    rows of the same call (distinct noise, no ties) still match the oracle."""
    B, d, V = 8, 64, 40000
    p = make_problem(B, d, V, T=1.0, seed=88)
    p["W"] = p["W"][:1].expand(V, d).contiguous()
    p["temperature"][:4] = 0.0
    idx, score = device_topk(p, K, seed=5, offset=2)
    for b in range(4):
        assert np.array_equal(idx[b], np.arange(K)), (b, idx[b])
        assert np.all(score[b] == score[b, 0])
    check_against_oracle(p, K, idx, score, rows=list(range(4, B)), seed=5, offset=2)
