#!/usr/bin/env python
"""Benchmark of the fused LM-head + exact Gumbel-max sampler (one GPU per rank).

A step is one fs_sample call (one fused kernel launch) over one batch of the
synthetic Qwen3-8B-shaped head (d=4096, V=151936): per-row temperatures
U[0.5,1.5] with 10% greedy rows, per-row seeds, the Philox offset advancing by
one per step.  W (1.24 GB) exceeds L2, so every step streams it from HBM.

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle on a
bounded sample of the same workload instead.  Under torchrun with N > 1 ranks,
each rank runs an independent replica (the batch path has no exchange step).
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "µs/call and % of HBM/tensor roofline, fused LM-head+sample, d=4096 V=151936"
L2_BYTES = 129 * 2**20  # GB300 L2
RAMP_S = 0.5  # untimed calls before the warm-up steps of the headline leg
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="qwen3-8b")
    ap.add_argument("--batch", type=int, default=64)
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--sweep-steps", type=int, default=200)
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="CPU budget of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--library-gemm", action="store_true",
                    help="also time a library bf16 GEMM (torch.matmul) of the same contraction, "
                         "logits written out and no sampling, beside the fused call")
    ap.add_argument("--library-gemm-batches", default="64,256,512")
    ap.add_argument("--sustain", type=float, default=0.0,
                    help="with --library-gemm: also run each for this many seconds back to "
                         "back and report clock, power and energy per call")
    return ap.parse_args()


# ---------------------------------------------------------------------------
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    return dict(FALLBACK_PEAKS, source="fallback")


def algorithmic(B, d, V, *, mask=False, seeds=True, temperature=True, tiles=False):
    """Bytes and flops one sampling call must move / do: W and H once, the
    per-row parameters and mask bits, the sampled ids (int64) and, with
    ``tiles``, the per-(row, 128-id tile) max, argmax and log-mass (4 B each)."""
    by = V * d * 2 + B * d * 2 + B * 8
    by += B * 4 if temperature else 0
    by += B * 8 if seeds else 0
    by += B * ((V + 31) // 32) * 4 if mask else 0
    by += B * ((V + 127) // 128) * 12 if tiles else 0
    return by, 2.0 * B * V * d


def roofline(B, d, V, us, peaks, traffic=None, **kw):
    by, fl = algorithmic(B, d, V, **kw)
    t_hbm = by / (peaks["hbm_gbs"] * 1e9)
    t_tc = fl / (peaks["bf16_tflops"] * 1e12)
    if t_hbm >= t_tc:
        ach = by / (us * 1e-6) / 1e9
        out = {"bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm_gbs"],
               "unit": "GB/s", "frac": round(ach / peaks["hbm_gbs"], 4)}
    else:
        ach = fl / (us * 1e-6) / 1e12
        out = {"bound": "tensor", "achieved": round(ach, 1), "peak": peaks["bf16_tflops"],
               "unit": "TFLOP/s", "frac": round(ach / peaks["bf16_tflops"], 4),
               # the same against the peak measured under the power cap (a GEMM run
               # for seconds), which long tensor-bound runs settle to
               "frac_of_sustained": round(ach / peaks["bf16_tflops_sustained"], 4)}
    out["traffic"] = traffic
    out["algorithmic_bytes"] = by
    out["algorithmic_flops"] = fl
    out["peak_source"] = peaks["source"]
    return out


def kernel_source_hash():
    """Hash of the sampling kernels' device code (host-only edits keep it)."""
    h = hashlib.sha256()
    for rel in ("lm_head_gumbel_gb300/csrc/fs_kernels.cuh", "lm_head_gumbel_gb300/csrc/fs_ptx.cuh",
                "lm_head_gumbel_gb300/csrc/fs_noise.cuh"):
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_traffic(workload, B):
    """DRAM bytes per stage-1 launch from the committed ncu summary, if it was
    taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "stage1_traffic.json")
    if not os.path.exists(path):
        return None
    try:
        with open(path) as f:
            rec = json.load(f)
        if rec.get("source_sha") != kernel_source_hash():
            return None
        ent = rec.get("launches", {}).get(f"{workload}/B={B}")
        return None if ent is None else int(ent["dram_bytes_per_launch"])
    except (OSError, ValueError, KeyError):
        return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons, every 100 ms."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None

    def start(self):
        self.fd, self.path = tempfile.mkstemp(suffix=".csv")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fd, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return []
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        os.close(self.fd)
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    rows.append({"t": ts, "sm": float(parts[1]), "sm_max": float(parts[2]),
                                 "power": parts[3], "active": parts[4],
                                 "hw_slowdown": parts[5], "hw_thermal_slowdown": parts[6],
                                 "sw_thermal_slowdown": parts[7], "sw_power_cap": parts[8]})
                except ValueError:
                    continue
        os.unlink(self.path)
        return rows

    @staticmethod
    def summarize(rows, t0, t1):
        inside = [r for r in rows if t0 <= r["t"] <= t1]
        window = "timed region"
        if not inside:
            inside, window = rows, "measurement phase"
        if not inside:
            return None
        reasons = sorted({k for r in inside for k in ("hw_slowdown", "hw_thermal_slowdown",
                                                      "sw_thermal_slowdown", "sw_power_cap")
                          if r[k].lower() == "active"})
        return {"sm_mhz": statistics.median(r["sm"] for r in inside),
                "sm_max_mhz": max(r["sm_max"] for r in inside), "reasons": reasons,
                "samples": len(inside), "window": window}


# ---------------------------------------------------------------------------
def dist_init(backend):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world, device=None):
    """Everything queued on `device` is done and every rank got here."""
    import torch
    cuda = device is not None and torch.device(device).type == "cuda"
    if cuda:
        torch.cuda.synchronize(device)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    if cuda:
        torch.cuda.synchronize(device)


def max_over_ranks(x, world, device="cpu"):
    """The largest value of x over all ranks (timing: the slowest rank)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def make_inputs(wl_name, B, device):
    import torch
    from lm_head_gumbel_gb300 import workloads as wl
    w = wl.WORKLOADS[wl_name]
    W = wl.make_weights(w.d, w.V, seed=77, device=device, outlier_frac=w.outlier_frac)
    H = wl.make_hidden(B, w.d, seed=2000 + B, device=device)
    T = wl.make_temperature(w, B, seed=3000 + B, device=device)
    seeds = wl.make_seeds(B, base=4000 + B, device=device) if w.per_row_seeds else None
    mask = wl.make_mask(B, w.V, w.mask_frac, seed=5000 + B, device=device) if w.mask_frac else None
    return w, {"H": H, "W": W, "temperature": T, "seeds": seeds, "vocab_mask": mask}


def time_calls(fn, steps, stream):
    import torch
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for k in range(steps):
        fn(k)
    e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1)  # ms


def run_ours(args):
    import torch
    import lm_head_gumbel_gb300 as fs
    from lm_head_gumbel_gb300 import workloads as wl_mod

    world, rank, local = dist_init("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    fs.load_library()
    peaks = load_peaks()
    B = args.batch
    w, inp = make_inputs(args.workload, B, dev)
    d, V = w.d, w.V
    stream = torch.cuda.current_stream(dev)
    out = torch.empty(B, dtype=torch.int64, device=dev)
    ws = torch.zeros(fs.fs_workspace_size(B, V), dtype=torch.uint8, device=dev)
    tiles = tile_outputs(w, B, dev)

    def call(k, base=0):
        fs.fs_sample(inp["H"], inp["W"], temperature=inp["temperature"], seeds=inp["seeds"],
                     vocab_mask=inp["vocab_mask"], offset=base + k, out_idx=out, workspace=ws,
                     stream=stream, **tiles)

    clocks = ClockSampler(local)
    clocks.start()
    # Bring the GPU to the clock it holds under this load before the warm-up
    # steps: calls for RAMP_S seconds (a few warm-up steps after idle input
    # generation run at a lower clock).
    t_ramp = time.time()
    k = 0
    while time.time() - t_ramp < RAMP_S:
        for _ in range(20):
            call(k)
            k += 1
        torch.cuda.synchronize(dev)
    for k in range(max(args.warmup, 3)):
        call(k)
    barrier(world, dev)
    t_wall0 = time.time()
    ms = time_calls(lambda k: call(k, args.warmup), args.steps, stream)
    t_wall1 = time.time()
    barrier(world, dev)
    ms = max_over_ranks(ms, world, dev)
    us_call = ms * 1000.0 / args.steps


    # batch sweep of the same head (same run, same W)
    sweep = []
    if not args.no_sweep and world == 1:
        for b2 in w.batches:
            sweep.append(time_point(w, args.workload, b2, inp["W"], dev, stream, peaks,
                                    args.sweep_steps))
    # The K-draws-without-replacement mode on the same batch (an extension of
    # the headline path; reported beside it, not in it).
    extensions = {}
    if world == 1 and not args.no_sweep:
        for K in (4, 16):
            tk_out = torch.empty((B, K), dtype=torch.int64, device=dev)
            tk_ws = torch.empty(fs.fs_topk_workspace_size(B, V, K), dtype=torch.uint8, device=dev)

            def ctk(k, K=K, tk_out=tk_out, tk_ws=tk_ws):
                fs.fs_sample_topk(inp["H"], inp["W"], K, temperature=inp["temperature"],
                                  seeds=inp["seeds"], vocab_mask=inp["vocab_mask"],
                                  offset=k, out_topk_idx=tk_out,
                                  workspace=tk_ws, stream=stream)

            for k in range(3):
                ctk(k)
            us_tk = time_calls(ctk, args.sweep_steps, stream) * 1000.0 / args.sweep_steps
            extensions[f"topk{K}_us_per_call"] = round(us_tk, 2)
            del tk_out, tk_ws

        # The headline call again, each launched to overlap the call before it
        # (FS_FLAG_OVERLAP_PREVIOUS): its launch and pipeline fill hide behind
        # the previous call's last units, as they would behind the kernel that
        # computes H in a decode step.  Reported beside the headline, not in it.
        def cov(k):
            fs.fs_sample(inp["H"], inp["W"], temperature=inp["temperature"], seeds=inp["seeds"],
                         vocab_mask=inp["vocab_mask"], offset=k, out_idx=out, workspace=ws,
                         stream=stream, overlap_previous=True, **tiles)

        for k in range(3):
            cov(k)
        us_ov = time_calls(cov, args.sweep_steps, stream) * 1000.0 / args.sweep_steps
        extensions["overlap_previous_us_per_call"] = round(us_ov, 2)

    # End to end through the C ABI, one fs_sample_host call per step: the
    # step's inputs (H, temperatures, seeds, mask) go host -> device in one copy
    # from one pinned buffer, the sampling kernel runs from an argument block
    # built once (only the offset changes), and the sampled ids come back
    # device -> host (pinned) before the call returns and the next step starts.
    import ctypes
    lib = fs.load_library()
    parts = [inp["H"].contiguous().view(torch.uint8).view(-1),
             inp["temperature"].contiguous().view(torch.uint8).view(-1)]
    if inp["seeds"] is not None:
        parts.append(inp["seeds"].contiguous().view(torch.uint8).view(-1))
    if inp["vocab_mask"] is not None:
        parts.append(inp["vocab_mask"].contiguous().view(torch.uint8).view(-1))
    sizes = [t.numel() for t in parts]
    pad = [(-n) % 256 for n in sizes]  # keep each input 256-byte aligned
    host_in = torch.empty(sum(sizes) + sum(pad), dtype=torch.uint8).pin_memory()
    dev_in = torch.empty_like(host_in, device=dev)
    pos, views = 0, []
    for t, n, q in zip(parts, sizes, pad):
        host_in[pos:pos + n].copy_(t.cpu())
        views.append(dev_in[pos:pos + n])
        pos += n + q
    Hd = views[0].view(torch.bfloat16).view(B, d)
    Td = views[1].view(torch.float32)
    Sd = views[2].view(torch.int64) if inp["seeds"] is not None else None
    Md = views[-1].view(torch.int32).view(B, -1) if inp["vocab_mask"] is not None else None
    out_h = torch.empty(B, dtype=torch.int64).pin_memory()
    args_c = fs.FsSampleArgs(
        H=Hd.data_ptr(), W=inp["W"].data_ptr(), temperature=Td.data_ptr(),
        vocab_mask=None if Md is None else Md.data_ptr(),
        mask_ld=0 if Md is None else Md.stride(0),
        seeds=None if Sd is None else Sd.data_ptr(), seed=0, offset=0, B=B, d=d, V=V,
        ldh=d, ldw=inp["W"].stride(0), out_idx=out.data_ptr(), workspace=ws.data_ptr(),
        workspace_bytes=ws.numel(),
        out_tile_max=tiles["out_tile_max"].data_ptr() if tiles else None,
        out_tile_idx=tiles["out_tile_idx"].data_ptr() if tiles else None,
        out_tile_lse=tiles["out_tile_lse"].data_ptr() if tiles else None)
    args_ref = ctypes.byref(args_c)
    sh = ctypes.c_void_p(stream.cuda_stream)
    hp, dp = ctypes.c_void_p(host_in.data_ptr()), ctypes.c_void_p(dev_in.data_ptr())
    op, n_in = ctypes.c_void_p(out_h.data_ptr()), host_in.numel()

    def e2e_step(k):
        args_c.offset = k
        # wait for the ids: they feed the next decode step
        if lib.fs_sample_host(args_ref, hp, dp, n_in, op, fs.FS_SYNC_IDS, sh) != fs.FS_OK:
            raise SystemExit("fs_sample_host failed")

    for k in range(3):
        e2e_step(k)
    barrier(world, dev)
    e2e_steps = max(10, min(args.steps, 500))
    ms_e2e = max_over_ranks(time_calls(e2e_step, e2e_steps, stream), world, dev)
    us_e2e = ms_e2e * 1000.0 / e2e_steps
    h2d = host_in.numel()  # bytes copied host -> device per step (inputs + alignment pad)
    d2h = out_h.numel() * 8

    # Every other workload of the benchmark set, each with its own head, batch
    # sizes, temperature law, mask and tile outputs (same run, same clocks).
    others = {}
    if not args.no_sweep and world == 1:
        for name in OTHER_WORKLOADS:
            if name == args.workload:
                continue
            wo = wl_mod.WORKLOADS[name]
            Wo = wl_mod.make_weights(wo.d, wo.V, seed=77, device=dev,
                                     outlier_frac=wo.outlier_frac)
            pts = [time_point(wo, name, bo, Wo, dev, stream, peaks, args.sweep_steps)
                   for bo in wo.batches]
            others[name] = {"config": describe(wo, "/".join(str(x) for x in wo.batches)),
                            "l2": l2_note(wo.V, wo.d), "points": pts}
            del Wo
            torch.cuda.empty_cache()

    clock_rows = clocks.stop()
    # clocks seen while each batch size ran
    for ent in sweep + [p for o in others.values() for p in o["points"]]:
        c = ClockSampler.summarize(clock_rows, *ent.pop("window"))
        ent["sm_mhz"] = None if c is None else c["sm_mhz"]
        ent["clock_reasons"] = None if c is None else c["reasons"]
    st, code = fs.fs_last_device_error()
    if st != fs.FS_OK:
        raise SystemExit(f"device error word {code} after the benchmark")

    rf = roofline(B, d, V, us_call, peaks, traffic=measured_traffic(args.workload, B),
                  seeds=inp["seeds"] is not None, mask=inp["vocab_mask"] is not None,
                  tiles=bool(tiles))
    rf["kernel"] = "fs::stage1_kernel (the whole call: stage 2 is fused into it)"
    rf["duration_us"] = round(us_call, 3)

    line = {
        "metric": METRIC,
        "value": round(us_call, 3),
        "unit": "us/call",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(us_call / 1000.0, 6),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": describe(w, B),
            "B": B, "d": d, "V": V, "global_batch": B * world,
            "l2": l2_note(V, d),
            "parallelism": "replicas" if world > 1 else "single-gpu",
            "clock_ramp_s": RAMP_S,
        },
        "tokens_per_s": round(B * world / (us_call * 1e-6), 1),
        "roofline": rf,
        "e2e": {"value": round(us_e2e, 3), "unit": "us/call",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)},
        "gpu_launches": args.steps,
        "clocks": ClockSampler.summarize(clock_rows, t_wall0, t_wall1),
        "sweep": sweep,
        "workloads": others,
        "extensions": extensions,
    }
    if world == 1 and args.library_gemm:
        batches = [int(x) for x in args.library_gemm_batches.split(",") if x]
        line["library_gemm"] = library_gemm_leg(w, inp["W"], dev, stream, batches,
                                                args.sweep_steps, args.sustain)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(inp, B, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# The benchmark set beside the headline head: each is timed in the default run.
OTHER_WORKLOADS = ("qwen3-8b", "qwen3-1.7b", "llama3-8b-mask", "large-vocab", "tiny")


def l2_note(V, d):
    return (("inputs exceed L2 (W is %.2f GB), no flush" % (V * d * 2 / 1e9))
            if V * d * 2 > L2_BYTES else
            ("W (%.1f MB) fits in L2: warm, no flush" % (V * d * 2 / 1e6)))


def time_point(w, name, B, W, dev, stream, peaks, steps):
    """One (workload, batch) point: `steps` sampling calls back to back, with
    the workload's own per-row inputs and tile outputs, offset = step."""
    import torch
    import lm_head_gumbel_gb300 as fs
    d, V = w.d, w.V
    _, inp = make_inputs_like(w, B, dev, W)
    out = torch.empty(B, dtype=torch.int64, device=dev)
    ws = torch.zeros(fs.fs_workspace_size(B, V), dtype=torch.uint8, device=dev)
    t = tile_outputs(w, B, dev)

    def call(k):
        fs.fs_sample(inp["H"], W, temperature=inp["temperature"], seeds=inp["seeds"],
                     vocab_mask=inp["vocab_mask"], offset=k, out_idx=out, workspace=ws,
                     stream=stream, **t)

    for k in range(5):
        call(k)
    torch.cuda.synchronize()
    ts0 = time.time()
    us = time_calls(call, steps, stream) * 1000.0 / steps
    rf = roofline(B, d, V, us, peaks, traffic=measured_traffic(name, B),
                  seeds=inp["seeds"] is not None, mask=inp["vocab_mask"] is not None,
                  tiles=bool(t))
    ent = {"B": B, "us_per_call": round(us, 2), "tokens_per_s": round(B / (us * 1e-6), 1),
           "bound": rf["bound"], "achieved": rf["achieved"], "unit": rf["unit"],
           "frac": rf["frac"], "traffic": rf["traffic"], "window": (ts0, time.time())}
    if "frac_of_sustained" in rf:
        ent["frac_of_sustained"] = rf["frac_of_sustained"]
    return ent


def make_inputs_like(w, B, device, W):
    from lm_head_gumbel_gb300 import workloads as wl
    H = wl.make_hidden(B, w.d, seed=2000 + B, device=device)
    T = wl.make_temperature(w, B, seed=3000 + B, device=device)
    seeds = wl.make_seeds(B, base=4000 + B, device=device) if w.per_row_seeds else None
    mask = wl.make_mask(B, w.V, w.mask_frac, seed=5000 + B, device=device) if w.mask_frac else None
    return w, {"H": H, "W": W, "temperature": T, "seeds": seeds, "vocab_mask": mask}


def tile_outputs(w, B, device):
    """Per-tile output buffers for workloads that ask for the tile log-mass."""
    import torch
    if not w.want_lse:
        return {}
    nt = (w.V + 127) // 128
    return {"out_tile_max": torch.empty((B, nt), dtype=torch.float32, device=device),
            "out_tile_idx": torch.empty((B, nt), dtype=torch.int32, device=device),
            "out_tile_lse": torch.empty((B, nt), dtype=torch.float32, device=device)}


def describe(w, B):
    """The workload in words, from its definition."""
    if w.temperature == "row-uniform":
        t = "per-row T~U[0.5,1.5] with 10% greedy"
    else:
        t = f"T={w.t_value:g}"
    parts = [f"{w.name} head: d={w.d} V={w.V} B={B}", "bf16 H~N(0,1) W~N(0,(2/sqrt d)^2)", t]
    if w.outlier_frac:
        parts.append(f"{100 * w.outlier_frac:g}% of W rows x4")
    if w.mask_frac:
        parts.append(f"per-row vocab mask ({100 * w.mask_frac:g}% of ids masked)")
    parts.append("per-row seeds" if w.per_row_seeds else "one seed")
    if w.want_lse:
        parts.append("tile max/argmax/LSE written")
    parts.append("offset=step")
    return ", ".join(parts)


def library_gemm_leg(w, W, dev, stream, batches, steps, sustain_s):
    """Context for the tensor-bound points: the same contraction H W^T as one
    library bf16 GEMM (torch.matmul, cuBLAS), logits written to HBM and nothing
    sampled, timed beside the fused sampling call on the same inputs.  Burst:
    ``steps`` calls after warm-up.  With ``sustain_s`` > 0 each also runs back
    to back for that long while nvidia-smi samples clock and power, since at
    large batches both settle at the board power limit."""
    import torch
    import lm_head_gumbel_gb300 as fs
    d, V = w.d, w.V
    entries = []
    for B in batches:
        _, inp = make_inputs_like(w, B, dev, W)
        out = torch.empty(B, dtype=torch.int64, device=dev)
        ws = torch.zeros(fs.fs_workspace_size(B, V), dtype=torch.uint8, device=dev)
        logits = torch.empty(B, V, dtype=torch.bfloat16, device=dev)

        def gemm(k):
            torch.matmul(inp["H"], W.t(), out=logits)

        def fused(k):
            fs.fs_sample(inp["H"], W, temperature=inp["temperature"], seeds=inp["seeds"],
                         vocab_mask=inp["vocab_mask"], offset=k, out_idx=out, workspace=ws,
                         stream=stream)

        ent = {"B": B}
        with torch.cuda.stream(stream):
            for name, fn in (("library_gemm", gemm), ("fused_sample", fused)):
                for k in range(5):
                    fn(k)
                torch.cuda.synchronize()
                us = time_calls(fn, steps, stream) * 1000.0 / steps
                ent[f"{name}_us"] = round(us, 2)
                ent[f"{name}_tflops"] = round(2.0 * B * V * d / us / 1e6, 1)
            if sustain_s > 0:
                sus = {}
                for name, fn in (("library_gemm", gemm), ("fused_sample", fused)):
                    sampler = ClockSampler(dev.index or 0)
                    sampler.start()
                    n, t0 = 0, time.time()
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    while time.time() - t0 < sustain_s:
                        for k in range(50):
                            fn(n + k)
                        n += 50
                        e1.record(stream)
                        e1.synchronize()
                    us = e0.elapsed_time(e1) * 1000.0 / n
                    rows = sampler.stop()
                    # the first half second is the ramp into the power limit
                    rows = [r for r in rows if t0 + 0.5 <= r["t"] <= time.time()]
                    watts = [float(r["power"]) for r in rows if r["power"].replace(".", "", 1).isdigit()]
                    c = ClockSampler.summarize(rows, t0 + 0.5, time.time())
                    p = statistics.median(watts) if watts else None
                    sus[name] = {"us": round(us, 2), "calls": n,
                                 "sm_mhz": None if c is None else c["sm_mhz"],
                                 "power_w": p, "reasons": None if c is None else c["reasons"],
                                 "joules_per_call": None if p is None else round(p * us * 1e-6, 4)}
                    time.sleep(1.0)
                ent["sustained"] = sus
        entries.append(ent)
        del inp, out, ws, logits
    return {"what": "torch.matmul bf16 of the same H W^T (library GEMM, logits written, "
                    "nothing sampled) vs the fused sampling call, same inputs",
            "entries": entries}


def oracle_inputs(inp):
    from lm_head_gumbel_gb300 import workloads as wl
    return (wl.bf16_bits(inp["H"]), wl.bf16_bits(inp["W"]), inp["temperature"].cpu().numpy(),
            None if inp["seeds"] is None else wl.u64_bits(inp["seeds"]),
            None if inp["vocab_mask"] is None else wl.u32_bits(inp["vocab_mask"]))


def cpu_baseline(inp, B, budget_s):
    """The oracle, as it stands, on a bounded sample of the same call: whole
    rows of the batch until the budget is spent; scaled to one call."""
    import oracle
    o = oracle.default()
    Hb, Wb, T, S, M = oracle_inputs(inp)
    t0 = time.perf_counter()
    o.sample(Hb, Wb, temperature=T, seeds=S, mask=M, rows=[0])
    first = time.perf_counter() - t0
    n = int(max(1, min(B - 1, budget_s / max(first, 1e-6))))
    rows = list(range(1, 1 + n))
    t0 = time.perf_counter()
    o.sample(Hb, Wb, temperature=T, seeds=S, mask=M, rows=rows)
    per_row = (time.perf_counter() - t0) / n if n else first
    cores = o.num_threads()
    # the same oracle on one core: one row
    o.set_num_threads(1)
    try:
        t0 = time.perf_counter()
        o.sample(Hb, Wb, temperature=T, seeds=S, mask=M, rows=[0])
        one_core_row = time.perf_counter() - t0
    finally:
        o.set_num_threads(cores)
    return {"value": round(per_row * B * 1e6, 1), "unit": "us/call", "cores": cores,
            "kind": "oracle",
            "sample": f"{n} of the call's {B} rows (fp64, full vocabulary each), scaled to {B} rows",
            "single_core": {"value": round(one_core_row * B * 1e6, 1), "unit": "us/call",
                            "sample": f"1 row on 1 core, scaled to {B} rows"}}


def run_reference(args):
    """The CPU oracle as the reference arm: each step is a bounded sample of
    the same call (one row, or a vocabulary slice of one row when a row is too
    slow for the step budget), scaled to the whole call."""
    world, rank, _ = dist_init("gloo")
    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    import torch
    import oracle
    from lm_head_gumbel_gb300 import workloads as wl
    w = wl.WORKLOADS[args.workload]
    B, d, V = args.batch, w.d, w.V
    _, inp = make_inputs(args.workload, B, "cpu")
    Hb, Wb, T, S, M = oracle_inputs(inp)
    o = oracle.default()
    t0 = time.perf_counter()
    o.sample(Hb, Wb, temperature=T, seeds=S, mask=M, rows=[0])
    row_s = time.perf_counter() - t0
    total = args.steps + args.warmup
    budget = 150.0 / max(total, 1)
    v_used = V if row_s <= budget else max(128, int(V * budget / row_s) // 128 * 128)
    Wsub = Wb[:v_used]
    scale = B * (V / v_used)

    def step(k):
        r = k % B
        o.sample(Hb, Wsub, temperature=T, seeds=S, rows=[r], offset=k,
                 mask=None if M is None else M[:, :(v_used + 31) // 32])

    for k in range(args.warmup):
        step(k)
    times = []
    for k in range(args.steps):
        t0 = time.perf_counter()
        step(args.warmup + k)
        times.append(time.perf_counter() - t0)
    us = statistics.mean(times) * scale * 1e6
    sample = (f"1 row of {B} per step" + ("" if v_used == V else f", vocabulary ids 0..{v_used - 1} of {V}")
              + f"; scaled x{scale:.1f} to one call")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(us, 1), "unit": "us/call",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(statistics.mean(times) * 1000.0, 3), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": describe(w, B), "B": B, "d": d,
                   "V": V, "global_batch": B, "parallelism": "cpu"},
        "cpu_baseline": {"value": round(us, 1), "unit": "us/call", "cores": o.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(us, 1), "unit": "us/call", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
