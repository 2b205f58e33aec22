"""The synthetic workloads at full size, in the launch configuration the
benchmark times: sampled rows against the oracle (which computes them one by
one), and properties that hold at any size on every row."""
import numpy as np
import pytest
import torch

import lm_head_gumbel_gb300 as fs
from lm_head_gumbel_gb300 import workloads as wl
from oracle import merge
from gpu_cases import assert_no_device_error, compare, make_problem, run_device

pytestmark = pytest.mark.gpu

_W_CACHE = {}


def weights(name):
    """Device W of a workload and its host bit patterns (one copy each)."""
    if name not in _W_CACHE:
        _W_CACHE.clear()
        torch.cuda.empty_cache()
        w = wl.WORKLOADS[name]
        W = wl.make_weights(w.d, w.V, seed=77, device="cuda", outlier_frac=w.outlier_frac)
        _W_CACHE[name] = (W, wl.bf16_bits(W))
    return _W_CACHE[name]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fs.load_library()
    yield
    _W_CACHE.clear()
    assert_no_device_error()


def sample_rows(B, k=4, seed=0):
    rng = np.random.default_rng(seed)
    rows = {0, B - 1} | set(rng.integers(0, B, size=k).tolist())
    return sorted(rows)


def whole_batch_properties(prob, dev, V):
    idx, tmax, tidx = dev["idx"], dev["tile_max"], dev["tile_idx"]
    B, nt = tmax.shape
    assert idx.shape == (B,)
    assert np.all((idx >= -1) & (idx < V))
    # stage 2 is the exact argmax over tiles (lowest id on ties)
    for b in range(B):
        ok = tidx[b] >= 0
        if not ok.any():
            assert idx[b] == -1
            continue
        m = np.where(ok, tmax[b], -np.inf)
        t = int(np.argmax(m))
        assert idx[b] == tidx[b, t]
    # every per-tile argmax lies in its tile
    t_of = np.arange(nt)[None, :]
    valid = tidx >= 0
    assert np.all((tidx[valid] // 128) == np.broadcast_to(t_of, tidx.shape)[valid])
    if prob["vocab_mask"] is not None:
        m = prob["vocab_mask"].cpu().numpy().view(np.uint32)
        sel = idx >= 0
        bits = (m[np.arange(B)[sel], idx[sel] // 32] >> (idx[sel] % 32)) & 1
        assert np.all(bits == 1), "a masked token was sampled"


@pytest.mark.parametrize("B", [1, 8, 32, 128, 256])
def test_qwen3_1_7b_head(B):
    W, Wb = weights("qwen3-1.7b")
    p = make_problem(B, W.shape[1], W.shape[0], T=0.7, seed=B, W=W)
    for step in (0, 1):
        dev = run_device(p, seed=2024, offset=step, lse=False)
        whole_batch_properties(p, dev, W.shape[0])
        compare(p, dev, sample_rows(B, seed=step), seed=2024, offset=step, W_bits=Wb)


@pytest.mark.parametrize("B", [1, 16, 64, 256, 512])
def test_qwen3_8b_head(B):
    """Per-row temperatures (10% greedy), per-row seeds, decode steps with the
    offset advancing: every step runs; sampled steps go to the oracle."""
    W, Wb = weights("qwen3-8b")
    p = make_problem(B, W.shape[1], W.shape[0], T="row-uniform", per_row_seeds=True, seed=B, W=W)
    steps = 1000 if B <= 64 else 50
    checked = (0, 1, steps // 2, steps - 1)
    out = torch.empty((steps, B), dtype=torch.int64, device="cuda")
    ws = torch.zeros(fs.fs_workspace_size(B, W.shape[0]), dtype=torch.uint8, device="cuda")
    for step in range(steps):
        fs.fs_sample(p["H"], W, temperature=p["temperature"], seeds=p["seeds"], offset=step,
                     out_idx=out[step], workspace=ws)
    torch.cuda.synchronize()
    out = out.cpu().numpy()
    assert np.all((out >= 0) & (out < W.shape[0]))
    greedy = (p["temperature"].cpu().numpy() <= 0)
    if greedy.any():  # greedy rows do not depend on the step
        assert np.all(out[:, greedy] == out[0:1, greedy])
    for step in checked:
        dev = run_device(p, seed=0, offset=step, lse=False)
        assert np.array_equal(dev["idx"], out[step])
        whole_batch_properties(p, dev, W.shape[0])
        compare(p, dev, sample_rows(B, k=2, seed=step), offset=step, seed=0, W_bits=Wb)


@pytest.mark.parametrize("B", [128, 512])
def test_qwen3_8b_whole_batch_against_oracle(B):
    """Every row of a production-size batch against the oracle: the Qwen3-8B
    head with its per-row temperatures (10% greedy) and seeds, B = 128 on the
    single-CTA kernel and B = 512 on the CTA-pair kernel.  The ids of the call
    the benchmark times (no per-tile outputs) equal those of the call that
    also writes them; then every row's id, and every tile's max, argmax and
    log-sum-exp, go through the parity gate."""
    W, Wb = weights("qwen3-8b")
    V = W.shape[0]
    p = make_problem(B, W.shape[1], V, T="row-uniform", per_row_seeds=True, seed=700 + B, W=W)
    out = torch.empty(B, dtype=torch.int64, device="cuda")
    ws = torch.zeros(fs.fs_workspace_size(B, V), dtype=torch.uint8, device="cuda")
    fs.fs_sample(p["H"], W, temperature=p["temperature"], seeds=p["seeds"], offset=17,
                 out_idx=out, workspace=ws)
    dev = run_device(p, seed=0, offset=17, lse=True)
    assert np.array_equal(out.cpu().numpy(), dev["idx"])
    whole_batch_properties(p, dev, V)
    st = compare(p, dev, list(range(B)), seed=0, offset=17, W_bits=Wb)
    assert st["rows"] == B and st["tiles"] == B * fs.fs_num_tiles(V), st
    # nearly every row is decided by a gap the gate resolves
    assert st["rows_gated"] >= 0.9 * B, st


def test_large_vocab_whole_batch_against_oracle():
    """Every row and tile of the large-vocabulary head (d=5120, V=262144) at
    B = 512 against the oracle: the CTA-pair kernel in its tile-LSE mode, at
    the size the benchmark times."""
    W, Wb = weights("large-vocab")
    V, B = W.shape[0], 512
    p = make_problem(B, W.shape[1], V, T=0.8, seed=900, W=W)
    dev = run_device(p, seed=77, offset=5, lse=True)
    whole_batch_properties(p, dev, V)
    st = compare(p, dev, list(range(B)), seed=77, offset=5, W_bits=Wb)
    assert st["rows"] == B and st["tiles"] == B * fs.fs_num_tiles(V), st
    assert st["rows_gated"] >= 0.9 * B and st["max_abs_tile_lse"] < 2e-3, st


def test_qwen3_1_7b_whole_batch_against_oracle():
    """Every row and tile of the Qwen3-1.7B head (d=2048) at B = 256 (the
    CTA-pair kernel, 32 K slices a unit) against the oracle."""
    W, Wb = weights("qwen3-1.7b")
    V, B = W.shape[0], 256
    p = make_problem(B, W.shape[1], V, T=0.7, seed=901, W=W)
    dev = run_device(p, seed=2024, offset=3, lse=False)
    whole_batch_properties(p, dev, V)
    st = compare(p, dev, list(range(B)), seed=2024, offset=3, W_bits=Wb)
    assert st["rows"] == B and st["rows_gated"] >= 0.9 * B, st


def test_llama3_8b_masked_head():
    W, Wb = weights("llama3-8b-mask")
    B = 128
    p = make_problem(B, W.shape[1], W.shape[0], T=1.0, mask_frac=0.05, seed=3, W=W)
    dev = run_device(p, seed=31, offset=9, lse=True)
    whole_batch_properties(p, dev, W.shape[0])
    compare(p, dev, sample_rows(B), seed=31, offset=9, W_bits=Wb)


@pytest.mark.parametrize("B", [512, 1024])
def test_large_vocab_head_partition_merge(B):
    """d=5120, V=262144: the tile log-sum-exps merged over 4 equal vocabulary
    partitions reproduce the row log-mass, and the exact merge over the
    partitions' maxima reproduces the sampled id on every row."""
    W, Wb = weights("large-vocab")
    V = W.shape[0]
    p = make_problem(B, W.shape[1], V, T=0.8, seed=B, W=W)
    dev = run_device(p, seed=55, offset=1, lse=True)
    whole_batch_properties(p, dev, V)
    nt = dev["tile_max"].shape[1]
    bounds = [0, nt // 4, nt // 2, 3 * nt // 4, nt]
    for b in range(B):
        i, _ = merge.partition_argmax(dev["tile_max"][b], dev["tile_idx"][b], bounds)
        assert i == dev["idx"][b]
    st = compare(p, dev, sample_rows(B, k=2), seed=55, offset=1, W_bits=Wb)
    assert st["max_abs_tile_lse"] < 2e-3
    rows = sample_rows(B, k=2)
    from gpu_cases import run_oracle
    ref = run_oracle(p, rows, seed=55, offset=1, W_bits=Wb)
    for r, b in enumerate(rows):
        parts = [merge.lse_merge(dev["tile_lse"][b, bounds[k]:bounds[k + 1]]) for k in range(4)]
        whole = merge.lse_merge(ref["tile_lse"][r])
        assert abs(merge.lse_merge(parts) - whole) < 2e-3


def test_stage1_only_call_at_full_size():
    """out_idx = NULL: only the per-tile (max, argmax, LSE) are written (the
    per-partition summaries a caller merges itself); they equal those of the
    full call, and their exact merge is its sample."""
    W, Wb = weights("qwen3-8b")
    B = 64
    p = make_problem(B, W.shape[1], W.shape[0], T="row-uniform", per_row_seeds=True, seed=94, W=W)
    full = run_device(p, seed=3, offset=6, lse=True)
    nt = full["tile_max"].shape[1]
    tm = torch.empty((B, nt), dtype=torch.float32, device="cuda")
    ti = torch.empty((B, nt), dtype=torch.int32, device="cuda")
    tl = torch.empty((B, nt), dtype=torch.float32, device="cuda")
    assert fs.fs_sample(p["H"], W, temperature=p["temperature"], seeds=p["seeds"], seed=3,
                        offset=6, out_tile_max=tm, out_tile_idx=ti, out_tile_lse=tl,
                        reduce=False) is None
    torch.cuda.synchronize()
    assert np.array_equal(tm.cpu().numpy(), full["tile_max"])
    assert np.array_equal(ti.cpu().numpy(), full["tile_idx"])
    assert np.array_equal(tl.cpu().numpy(), full["tile_lse"])
    for b in range(B):
        i, _ = merge.partition_argmax(full["tile_max"][b], full["tile_idx"][b], [0, nt])
        assert i == full["idx"][b]


def test_largest_batch():
    """B = 65535, the largest batch the ABI takes (CTA pairs, 256 pair blocks),
    on a ragged vocabulary: sampled rows against the oracle and the
    whole-batch properties."""
    B, d, V = 65535, 64, 520
    p = make_problem(B, d, V, T="row-uniform", per_row_seeds=True, seed=93)
    dev = run_device(p, seed=8, offset=4, lse=False)
    whole_batch_properties(p, dev, V)
    compare(p, dev, [0, 1, 255, 256, 12345, 65279, 65534], seed=8, offset=4)


def test_largest_vocabulary():
    """V = 2^31 - 1, the largest vocabulary the ABI takes (a 32 GiB W at
    d = 8): the first, a middle and the last (partial) tile against the
    oracle's logits and noise at those global ids, ids near 2^31 through the
    packed row keys, and the sample = the best tile's argmax."""
    import oracle
    from oracle import parity
    V, d, B, T = 2**31 - 1, 8, 2, 1.0
    _W_CACHE.clear()
    torch.cuda.empty_cache()
    W = wl.make_weights(d, V, seed=91, device="cuda")
    p = make_problem(B, d, V, T=T, seed=92, W=W)
    dev = run_device(p, seed=5, offset=3, lse=False)
    nt = dev["tile_max"].shape[1]
    assert nt == (V + 127) // 128
    whole_batch_properties(p, dev, V)
    o = oracle.default()
    Hb = wl.bf16_bits(p["H"])
    for t in (0, nt // 2, nt - 1):
        v0, v1 = t * 128, min(V, t * 128 + 128)
        s = o.logits(Hb, wl.bf16_bits(W[v0:v1])) / T + o.noise_grid(0, B, v0, v1 - v0, seed=5,
                                                                     offset=3)
        for b in range(B):
            order = np.argsort(-s[b], kind="stable")
            assert abs(dev["tile_max"][b, t] - s[b, order[0]]) < parity.TOL_MAX, (b, t)
            if s[b, order[0]] - s[b, order[1]] > parity.GAP:
                assert dev["tile_idx"][b, t] == v0 + order[0], (b, t)
    del W, p, dev
    torch.cuda.empty_cache()
