"""CUDA path (through the C ABI) against the CPU oracle on small and ragged
problems, element by element: sampled ids, per-tile maxima, argmaxes and
log-sum-exps (gate and tolerances in oracle/parity.py)."""
import math

import numpy as np
import pytest
import scipy.special
import torch

import lm_head_gumbel_gb300 as fs
from lm_head_gumbel_gb300 import workloads as wl
import oracle
from oracle import merge, parity
from gpu_cases import assert_no_device_error, compare, make_problem, run_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fs.load_library()
    yield
    assert_no_device_error()


def test_noise_matches_oracle():
    """Device Philox + Gumbel vs the oracle's fp64 chain on a window that spans
    several Philox blocks, rows, per-row seeds and a high offset word."""
    o = oracle.default()
    for (seed, offset, seeds) in ((0, 0, None), (123456789123, (7 << 32) + 3, None),
                                  (0, 99, np.array([5, 2**63 + 11, 0, 2**40], np.uint64))):
        sd_t = None if seeds is None else torch.from_numpy(seeds.view(np.int64)).cuda()
        g = fs.fs_gumbel_noise(0, 4, 1000, 777, seed=seed, offset=offset, seeds=sd_t)
        torch.cuda.synchronize()
        want = o.noise_grid(0, 4, 1000, 777, seed=seed, offset=offset, seeds=seeds)
        err = np.abs(g.cpu().numpy().astype(np.float64) - want)
        assert err.max() < 2e-5, err.max()


def test_noise_transform_every_uniform_level():
    """Exhaustive: the device's word -> Gumbel transform for every one of the
    2^23 uniform levels u = (k + 1/2) 2^-23 (only a word's low 23 bits count)
    is within 1e-5 of g = -log(-log u) in fp64, and the high 9 bits are
    ignored."""
    k = torch.arange(1 << 23, dtype=torch.int64)
    g = fs.fs_gumbel_transform(k.to(torch.int32).cuda()).cpu().numpy().astype(np.float64)
    u = (k.numpy().astype(np.float64) + 0.5) * 2.0 ** -23
    want = -np.log(-np.log(u))
    err = np.abs(g - want)
    assert err.max() < 1e-5, (err.max(), int(err.argmax()))
    hi = (k[:4096] | (0x5A5 << 23)).to(torch.int32).cuda()  # other high bits, same level
    assert np.array_equal(fs.fs_gumbel_transform(hi).cpu().numpy(), g[:4096].astype(np.float32))


def test_noise_accuracy_over_all_uniforms():
    """Noise from Philox words over 2^21 consecutive vocabulary ids (many
    Philox blocks) against the oracle's fp64 chain on a subsample."""
    o = oracle.default()
    g = fs.fs_gumbel_noise(0, 1, 0, 1 << 21, seed=42, offset=1).cpu().numpy().ravel()
    sub = np.arange(0, 1 << 21, 997)
    want = np.array([o.noise(42, 1, 0, int(v)) for v in sub])
    assert np.abs(g[sub] - want).max() < 2e-5
    assert np.all(np.isfinite(g)) and g.min() > -3.0 and g.max() < 17.0


@pytest.mark.parametrize("T", [1.0, 0.0, 0.7])
def test_tiny(T):
    """B=4, d=256, V=4096: every row and tile, noisy and greedy."""
    p = make_problem(4, 256, 4096, T=T, seed=1)
    dev = run_device(p, seed=0, offset=0)
    st = compare(p, dev, seed=0, offset=0, scores=True)
    assert st["rows_gated"] >= 3


@pytest.mark.parametrize("B,d,V", [
    (1, 8, 1), (1, 8, 2), (3, 72, 100), (1, 264, 1000), (5, 64, 129), (2, 136, 4097),
    (7, 200, 255), (33, 96, 257), (129, 64, 640), (130, 128, 3000), (300, 64, 1100),
    (256, 72, 100), (256, 64, 1), (260, 64, 300), (512, 40, 700), (511, 64, 1300),
    (4, 16384, 3000), (130, 8200, 700),  # long K loops (256 and 129 slices)
])
def test_ragged_shapes(B, d, V):
    """Odd B (several 128-row blocks, CTA pairs for even block counts), d not
    a multiple of 64, V with a ragged last tile and a ragged last 256-id unit
    (including a vocabulary smaller than one pair's half slice)."""
    p = make_problem(B, d, V, T=0.9, seed=B + d + V)
    dev = run_device(p, seed=3, offset=5)
    compare(p, dev, seed=3, offset=5, scores=True)


def test_strided_inputs():
    """H and W as column slices of wider buffers (row strides ldh, ldw > d)
    and a mask with spare words per row: the same results as on contiguous
    copies, and parity with the oracle."""
    B, d, V = 40, 96, 3000
    p = make_problem(B, d, V, T="row-uniform", per_row_seeds=True, mask_frac=0.04, seed=16)
    Hw = torch.zeros((B, d + 40), dtype=torch.bfloat16, device="cuda")
    Ww = torch.zeros((V, d + 24), dtype=torch.bfloat16, device="cuda")
    Mw = torch.zeros((B, p["vocab_mask"].shape[1] + 5), dtype=torch.int32, device="cuda")
    Hw[:, 8:8 + d] = p["H"]
    Ww[:, :d] = p["W"]
    Mw[:, :p["vocab_mask"].shape[1]] = p["vocab_mask"]
    q = dict(p, H=Hw[:, 8:8 + d], W=Ww[:, :d], vocab_mask=Mw)
    assert q["H"].stride(0) == d + 40 and q["W"].stride(0) == d + 24
    a = run_device(p, seed=3, offset=8)
    b = run_device(q, seed=3, offset=8)
    for k in a:
        assert np.array_equal(a[k], b[k]), k
    compare(p, b, seed=3, offset=8)


def test_mixed_rows_seeds_mask():
    """Per-row seeds, per-row temperatures with greedy rows, a vocab mask with
    fully masked tiles and a fully masked row."""
    B, d, V = 40, 128, 2000
    p = make_problem(B, d, V, T="row-uniform", per_row_seeds=True, mask_frac=0.05, seed=9)
    m = p["vocab_mask"]
    m[3, :] = 0                      # row 3: nothing allowed
    m[5, 4:8] = 0                    # row 5: tile 1 fully masked
    dev = run_device(p, offset=17)
    assert dev["idx"][3] == -1
    assert np.all(dev["tile_idx"][5, 1] == -1)
    compare(p, dev, offset=17, scores=True)


def test_outliers_and_lse():
    """W rows scaled by 4 (heavy logits) with the tile log-sum-exp output."""
    p = make_problem(16, 256, 3000, T=1.0, outlier_frac=0.03, mask_frac=0.05, seed=4)
    dev = run_device(p, offset=2)
    st = compare(p, dev, offset=2, scores=True)
    assert st["max_abs_tile_lse"] < parity.TOL_LSE


def test_workspace_path_matches_tile_outputs():
    p = make_problem(20, 64, 5000, T=0.8, seed=5)
    a = run_device(p, offset=3, lse=False, tiles=False)
    b = run_device(p, offset=3, lse=True, tiles=True)
    assert np.array_equal(a["idx"], b["idx"])


def test_deterministic_across_calls_and_streams():
    p = make_problem(64, 128, 6000, T=1.0, seed=6)
    a = run_device(p, offset=11)
    s = torch.cuda.Stream()
    b = run_device(p, offset=11, stream=s)
    c = run_device(p, offset=11)
    for k in a:
        assert np.array_equal(a[k], b[k]) and np.array_equal(a[k], c[k]), k
    d = run_device(p, offset=12)
    assert not np.array_equal(a["idx"], d["idx"])


@pytest.mark.parametrize("V", [40000, 151936])
def test_rows_do_not_depend_on_the_batch(V):
    """A row's tile outputs and sample are bit-identical whatever batch it sits
    in: B = 64 (one batch block: single CTAs, M = 128 MMAs with an H box of
    64 rows), B = 384 (three batch blocks: single CTAs, M = 128) and B = 256
    (CTA pairs, M = 256).  Every unit covers 256 vocabulary ids and starts its
    K loop at its vocabulary block's own slice, so only the MMA shape
    differs."""
    big = make_problem(384, 512, V, T="row-uniform", per_row_seeds=True, seed=12)
    runs = {}
    for B in (64, 256, 384):
        sub = {k: (None if t is None else t[:B].contiguous()) if k != "W" else t
               for k, t in big.items()}
        runs[B] = run_device(sub, seed=5, offset=6)
    for B in (256, 384):
        for k in ("idx", "tile_max", "tile_idx", "tile_lse"):
            assert np.array_equal(runs[B][k][:64], runs[64][k]), (B, k)
    assert np.array_equal(runs[384]["tile_max"][:256], runs[256]["tile_max"])


@pytest.mark.parametrize("B", [1, 5, 32, 40, 64])
def test_partial_batch_block_is_bit_identical(B):
    """A batch of fewer than 128 rows copies only its own H rows into each
    stage (the MMA's other accumulator rows read whatever follows and are
    never used), so fewer lane quadrants hold rows.  The same rows inside a
    full 128-row block must give bit-identical samples and per-tile maxima and
    argmaxes (masks, greedy rows and per-row seeds included), and both must
    match the oracle."""
    big = make_problem(128, 264, 5000, T="row-uniform", per_row_seeds=True, mask_frac=0.05,
                       seed=120)
    ref = run_device(big, seed=9, offset=4, lse=False)
    sub = {k: (None if t is None else t[:B].contiguous()) if k != "W" else t
           for k, t in big.items()}
    got = run_device(sub, seed=9, offset=4, lse=False)
    for k in ("idx", "tile_max", "tile_idx"):
        assert np.array_equal(got[k], ref[k][:B]), k
    compare(sub, got, seed=9, offset=4, scores=True)


@pytest.mark.parametrize("lse", [False, True])
def test_noise_made_ahead_is_bit_identical(lse):
    """In the single-CTA kernel each CTA's last unit reads noise that its
    epilogue warps wrote into tensor memory while the unit's W slices streamed
    in; every other unit (and every unit of the CTA-pair kernel) makes its
    noise in the epilogue.  Which units are last depends on the batch: at
    B = 128 the last wave covers other vocabulary blocks than at B = 384
    (three batch blocks), and B = 256 runs on CTA pairs.  The same rows must
    give bit-identical samples and tile outputs (greedy rows, masks and
    per-row seeds included) and match the oracle."""
    V = 151936
    big = make_problem(384, 128, V, T="row-uniform", per_row_seeds=True, mask_frac=0.05,
                       seed=121)
    ref = run_device(big, seed=3, offset=8, lse=lse)
    for B in (128, 256):
        sub = {k: (None if t is None else t[:B].contiguous()) if k != "W" else t
               for k, t in big.items()}
        got = run_device(sub, seed=3, offset=8, lse=lse)
        for k in got:
            assert np.array_equal(got[k], ref[k][:B]), (B, k)
    compare(sub, got, rows=[0, 77, 128, 200, 255], seed=3, offset=8)


def test_tiny_temperature_is_effectively_greedy():
    """T = 1e-4 (l/T ~ 1e5, far from fp32 overflow): the sample is the argmax
    of the logits wherever the logit gap is clearly wider than the noise's
    reach, and equals the oracle's id wherever its score gap exceeds 1 (the
    fp32 logit error, ~1e-5, is magnified 1e4 times in the score)."""
    B, d, V = 16, 64, 2000
    p = make_problem(B, d, V, T=1e-4, seed=18)
    dev = run_device(p, seed=4, offset=1, lse=False, tiles=False)
    o = oracle.default()
    Hb, Wb = wl.bf16_bits(p["H"]), wl.bf16_bits(p["W"])
    ref = o.sample(Hb, Wb, temperature=p["temperature"].cpu().numpy(), seed=4, offset=1)
    gated = ref["gap"] > 1.0
    assert gated.sum() >= B // 2 and np.array_equal(dev["idx"][gated], ref["idx"][gated])
    logits = o.logits(Hb, Wb)
    top2 = np.sort(logits, axis=1)[:, -2:]
    clear = (top2[:, 1] - top2[:, 0]) > 40 * 1e-4  # noise spans about 20 nats at most
    assert np.array_equal(dev["idx"][clear], logits.argmax(axis=1)[clear])


def test_nan_logits_are_never_sampled():
    """W rows of NaN (so their logits are NaN in every row) are excluded like
    masked ids; a tile made only of them reports (-inf, -1)."""
    B, d, V = 8, 64, 700
    p = make_problem(B, d, V, T=1.0, seed=19)
    W = p["W"].clone()
    nan_ids = [3, 130, 131, 600]
    W[nan_ids] = float("nan")
    W[256:384] = float("nan")  # all of tile 2
    q = dict(p, W=W)
    for off in range(20):
        dev = run_device(q, seed=2, offset=off, lse=False)
        assert not np.isin(dev["idx"], nan_ids + list(range(256, 384))).any()
        assert np.all(dev["tile_idx"][:, 2] == -1) and np.all(np.isneginf(dev["tile_max"][:, 2]))
    o = oracle.default()
    ref = o.sample(wl.bf16_bits(p["H"]), wl.bf16_bits(W), temperature=p["temperature"].cpu().numpy(),
                   seed=2, offset=19)
    gated = ref["gap"] > parity.GAP
    assert np.array_equal(dev["idx"][gated], ref["idx"][gated])


def test_host_step_matches_device_call():
    """fs_sample_host (host inputs -> device -> sampled ids back in host
    memory, one call) gives what fs_sample gives on the same inputs, with and
    without the wait inside the call, and with nothing to copy in."""
    B, d, V = 24, 128, 5000
    p = make_problem(B, d, V, T="row-uniform", per_row_seeds=True, mask_frac=0.02, seed=14)
    want = run_device(p, seed=5, offset=21, lse=False, tiles=False)["idx"]
    parts = [p["H"].view(torch.uint8).reshape(-1), p["temperature"].view(torch.uint8),
             p["seeds"].view(torch.uint8), p["vocab_mask"].view(torch.uint8).reshape(-1)]
    sizes = [t.numel() for t in parts]
    offs = np.concatenate([[0], np.cumsum([(n + 255) // 256 * 256 for n in sizes])])
    host_in = torch.zeros(int(offs[-1]), dtype=torch.uint8).pin_memory()
    for t, o, n in zip(parts, offs, sizes):
        host_in[int(o):int(o) + n].copy_(t.cpu())
    dev_in = torch.empty_like(host_in, device="cuda")
    dptr = [dev_in.data_ptr() + int(o) for o in offs[:4]]
    out = torch.empty(B, dtype=torch.int64, device="cuda")
    ws = torch.zeros(fs.fs_workspace_size(B, V), dtype=torch.uint8, device="cuda")
    args = fs.FsSampleArgs(H=dptr[0], W=p["W"].data_ptr(), temperature=dptr[1],
                           vocab_mask=dptr[3], mask_ld=p["vocab_mask"].stride(0), seeds=dptr[2],
                           seed=5, offset=21, B=B, d=d, V=V, ldh=d, ldw=d,
                           out_idx=out.data_ptr(), workspace=ws.data_ptr(),
                           workspace_bytes=ws.numel())
    host_out = torch.full((B,), -7, dtype=torch.int64).pin_memory()
    fs.fs_sample_host(args, host_in, dev_in, host_out)
    assert np.array_equal(host_out.numpy(), want)
    host_out.fill_(-7)
    s = torch.cuda.Stream()
    fs.fs_sample_host(args, host_in, dev_in, host_out, sync=False, stream=s)
    s.synchronize()
    assert np.array_equal(host_out.numpy(), want)
    host_out.fill_(-7)
    fs.fs_sample_host(args, None, None, host_out)  # inputs already on the device
    assert np.array_equal(host_out.numpy(), want)
    for _ in range(3):  # waiting on the ids themselves
        host_out.fill_(-7)
        fs.fs_sample_host(args, host_in, dev_in, host_out, sync=fs.FS_SYNC_IDS)
        assert np.array_equal(host_out.numpy(), want)
    torch.cuda.synchronize()
    # an earlier call that did not wait still writes host_out: the waiting
    # call must not take that call's ids for its own
    other = run_device(p, seed=5, offset=22, lse=False, tiles=False)["idx"]
    assert not np.array_equal(other, want)
    s2 = torch.cuda.Stream()
    for _ in range(5):
        args.offset = 22
        fs.fs_sample_host(args, host_in, dev_in, host_out, sync=fs.FS_SYNC_NONE, stream=s2)
        args.offset = 21
        fs.fs_sample_host(args, host_in, dev_in, host_out, sync=fs.FS_SYNC_IDS, stream=s2)
        assert np.array_equal(host_out.numpy(), want)
    torch.cuda.synchronize()
    # pageable (unmapped) host buffers take the copy-engine path
    dev_in.zero_()
    paged_out = torch.full((B,), -7, dtype=torch.int64)
    fs.fs_sample_host(args, host_in.clone(), dev_in, paged_out)
    assert np.array_equal(paged_out.numpy(), want)
    # an unaligned pinned source takes the byte-wise copy kernel
    dev_in.zero_()
    shifted = torch.zeros(host_in.numel() + 1, dtype=torch.uint8).pin_memory()
    shifted[1:].copy_(host_in)
    dev_in2 = torch.empty(host_in.numel() + 16, dtype=torch.uint8, device="cuda")
    fs.fs_sample_host(args, shifted[1:], dev_in2[1:host_in.numel() + 1], host_out)
    assert torch.equal(dev_in2[1:host_in.numel() + 1].cpu(), host_in)


def test_concurrent_host_threads():
    """Four host threads, each with its own stream and workspace, sampling the
    same problems at once give exactly the single-thread results."""
    import threading
    p = make_problem(24, 96, 3000, T="row-uniform", per_row_seeds=True, seed=20)
    want = {off: run_device(p, seed=9, offset=off, lse=False, tiles=False)["idx"]
            for off in range(8)}
    errors = []

    def worker(tid):
        try:
            s = torch.cuda.Stream()
            ws = torch.zeros(fs.fs_workspace_size(24, 3000), dtype=torch.uint8, device="cuda")
            out = torch.empty((8, 24), dtype=torch.int64, device="cuda")
            with torch.cuda.stream(s):
                for rep in range(10):
                    for off in range(8):
                        fs.fs_sample(p["H"], p["W"], temperature=p["temperature"],
                                     seeds=p["seeds"], seed=9, offset=off, out_idx=out[off],
                                     workspace=ws, stream=s)
            s.synchronize()
            for off in range(8):
                if not np.array_equal(out[off].cpu().numpy(), want[off]):
                    errors.append((tid, off))
        except Exception as e:  # reported below
            errors.append((tid, repr(e)))

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors


def test_graph_replay_matches_eager():
    p = make_problem(8, 64, 3000, T=1.0, seed=8)
    eager = run_device(p, offset=4)["idx"]
    out = torch.empty(8, dtype=torch.int64, device="cuda")
    ws = torch.zeros(fs.fs_workspace_size(8, 3000), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        fs.fs_sample(p["H"], p["W"], temperature=p["temperature"], seed=7, offset=4,
                     out_idx=out, workspace=ws)  # first call sets the device up
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fs.fs_sample(p["H"], p["W"], temperature=p["temperature"], seed=7, offset=4,
                     out_idx=out, workspace=ws)
    for _ in range(3):
        out.fill_(-5)
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy(), eager)


def test_host_step_in_a_cuda_graph():
    """fs_sample_host without its wait, captured in a CUDA graph (copy-in
    kernel, overlapped sampling kernel writing mapped host memory): each
    replay picks up new host inputs and delivers their ids to host memory."""
    B, d, V = 16, 64, 3000
    p = make_problem(B, d, V, T=1.0, seed=17)
    hb = p["H"].view(torch.uint8).reshape(-1)
    host_in = torch.zeros(hb.numel(), dtype=torch.uint8).pin_memory()
    dev_in = torch.empty_like(host_in, device="cuda")
    out = torch.empty(B, dtype=torch.int64, device="cuda")
    ws = torch.zeros(fs.fs_workspace_size(B, V), dtype=torch.uint8, device="cuda")
    host_out = torch.full((B,), -7, dtype=torch.int64).pin_memory()
    args = fs.FsSampleArgs(H=dev_in.data_ptr(), W=p["W"].data_ptr(), seed=3, offset=2, B=B, d=d,
                           V=V, ldh=d, ldw=d, out_idx=out.data_ptr(), workspace=ws.data_ptr(),
                           workspace_bytes=ws.numel())
    s = torch.cuda.Stream()
    host_in.copy_(hb.cpu())
    fs.fs_sample_host(args, host_in, dev_in, host_out, stream=s)  # sets the device up
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fs.fs_sample_host(args, host_in, dev_in, host_out, sync=False, stream=s)
    for k in range(3):
        H = wl.make_hidden(B, d, seed=900 + k, device="cuda")
        want = fs.fs_sample(H, p["W"], seed=3, offset=2)
        torch.cuda.synchronize()
        host_in.copy_(H.view(torch.uint8).reshape(-1).cpu())
        host_out.fill_(-7)
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(host_out.numpy(), want.cpu().numpy()), k


def test_chi_square_on_device():
    """Device draws over many offsets follow softmax(l/T) (Pearson
    chi-square), and equal the oracle's draws offset by offset."""
    V, d, T, n = 16, 64, 0.8, 6000
    p = make_problem(1, d, V, T=T, seed=12)
    out = torch.empty(1, dtype=torch.int64, device="cuda")
    ws = torch.zeros(fs.fs_workspace_size(1, V), dtype=torch.uint8, device="cuda")
    draws = torch.empty(n, dtype=torch.int64, device="cuda")
    for off in range(n):
        fs.fs_sample(p["H"], p["W"], temperature=p["temperature"], seed=99, offset=off,
                     out_idx=draws[off:off + 1], workspace=ws)
    torch.cuda.synchronize()
    draws = draws.cpu().numpy()
    o = oracle.default()
    Hb, Wb = wl.bf16_bits(p["H"]), wl.bf16_bits(p["W"])
    logits = o.logits(Hb, Wb)[0]
    probs = scipy.special.softmax(logits / float(np.float32(T)))
    _, _, pval = merge.chi_square_gof(np.bincount(draws, minlength=V), probs)
    assert pval > 1e-3, pval
    agree = 0
    for off in range(0, n, 10):
        r = o.sample(Hb, Wb, temperature=p["temperature"].cpu().numpy(), seed=99, offset=off)
        if r["gap"][0] > parity.GAP:
            assert draws[off] == r["idx"][0], off
            agree += 1
    assert agree > 0.9 * (n // 10)


def test_max_stability_on_device():
    """Max-stability of the device's per-tile outputs: over independent rows
    (the same logits, per-row seeds) m_t - L_t is Gumbel(0, 1) for every tile
    (mean Euler's gamma, Kolmogorov-Smirnov against the Gumbel cdf); this ties
    the noise, the max and the tile log-sum-exp together."""
    import scipy.stats
    B, d, V = 4096, 32, 512
    p = make_problem(1, d, V, T=0.9, seed=15)
    H = p["H"].expand(B, d).contiguous()  # one row of logits, B independent draws
    temperature = p["temperature"].expand(B).contiguous()
    seeds = wl.make_seeds(B, base=77, device="cuda")
    q = {"H": H, "W": p["W"], "temperature": temperature, "seeds": seeds, "vocab_mask": None}
    dev = run_device(q, offset=3)
    x = (dev["tile_max"] - dev["tile_lse"]).astype(np.float64)
    for t in range(x.shape[1]):
        assert abs(x[:, t].mean() - oracle.EULER_GAMMA) < 4.5 * math.sqrt(oracle.GUMBEL_VAR / B)
        assert scipy.stats.kstest(x[:, t], scipy.stats.gumbel_r.cdf).pvalue > 1e-3, t


def test_group_merge_on_device_tiles():
    """Group-Gumbel-Max over 4 vocabulary partitions, fed the device's per-tile
    (max, argmax, log-sum-exp), reproduces the distribution, and the exact
    partition argmax equals the flat sample."""
    V, d, T, n = 512, 32, 1.0, 2000
    p = make_problem(1, d, V, T=T, seed=13)
    probs = None
    rng = np.random.default_rng(0)
    hier = []
    for off in range(n):
        dev = run_device(p, seed=5, offset=off)
        tm, ti, tl = dev["tile_max"][0], dev["tile_idx"][0], dev["tile_lse"][0]
        i, _ = merge.partition_argmax(tm, ti, [0, 1, 2, 3, 4])
        assert i == dev["idx"][0]
        hier.append(merge.group_gumbel_max(ti, tl, rng.random(4)))
        if probs is None:
            Hb, Wb = wl.bf16_bits(p["H"]), wl.bf16_bits(p["W"])
            probs = scipy.special.softmax(oracle.default().logits(Hb, Wb)[0] / T)
    counts = np.bincount(np.asarray(hier), minlength=V)
    _, _, pval = merge.chi_square_gof(counts, probs)
    assert pval > 1e-3, pval
