"""Benchmark of the Lightning Indexer: query-tokens/s of one Top-512 indexer call.

Default workload: cold prefill at 64k context, T = S = 65536 bf16 queries/keys, 64 index heads
of width 128, fp32 head weights, causal, Top-512, seed 2. One step = one ds4idx_score_topk call
(scorer + streaming Top-512, the whole path) over the full workload.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints one JSON line. `value` is device-resident throughput (inputs already in HBM); `e2e`
repeats the measurement through the same C-ABI call with pinned HOST buffers, the host->device
copies of q, w and the key cache and the device->host copy of the outputs inside the timed
region. `roofline` reports the kernel against the measured dense bf16 tensor peak (tensor-bound
workloads) or HBM bandwidth (decode). `cpu_baseline` times the fp64 CPU oracle (test
infrastructure, untuned) on a bounded row sample of the same workload on this host's cores.
`--impl reference` times only that oracle, as the reference arm.
Multi-GPU (torchrun): every rank runs an independent replica of the workload (the indexer has no
exchange step); value = all ranks' query tokens / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from sparse_attention_lightning_indexer_gb300 import inputs  # noqa: E402

METRIC = "indexer query-tokens/s at 64k ctx (top-512) and % of tensor/HBM roofline"
UNIT = "query-tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_OVER_BF16 = 2.0  # nominal dense ratio (4.5 / 2.25 PFLOP/s)


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_sources_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sparse_attention_lightning_indexer_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def traffic_for(workload):
    """DRAM bytes per launch from the committed ncu summary, if taken on the current kernel."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("kernel_sources") != kernel_sources_hash():
        return None
    return e.get("dram_bytes_per_launch")


def algorithmic(prob):
    """Causal flops (visible pairs only) and key-cache bytes of one call."""
    T, S, pos = prob.T, prob.S, prob.pos_offset
    t = np.arange(T, dtype=np.float64)
    pairs = float(np.minimum(pos + t, S - 1).sum() + T)
    flops = 2.0 * inputs.H_I * inputs.D_I * pairs
    row_bytes = inputs.D_I * (2 if prob.dtype == inputs.BF16 else 1)
    key_bytes = float(S * row_bytes + (S * 4 if prob.dtype == inputs.FP8_E4M3 else 0))
    return flops, key_bytes, pairs


def all_bytes(prob):
    """Every byte one call moves at least once: q, w, key cache (+ scales) and both outputs.
    A secondary figure, for information: prefill re-reads keys from L2, not from HBM."""
    row_bytes = inputs.D_I * (2 if prob.dtype == inputs.BF16 else 1)
    q = prob.T * inputs.H_I * row_bytes
    w = prob.T * inputs.H_I * 4
    k = prob.S * row_bytes + (prob.S * 4 if prob.dtype == inputs.FP8_E4M3 else 0)
    out = prob.T * prob.topk * (4 + 4)
    return float(q + w + k + out)


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while running (200 ms period)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def aggregate(local_ms, units_per_rank, device=None):
    """Whole-job throughput across ranks: the slowest rank's time bounds the job.

    Returns (max_ms, units/s over all ranks). With one process this is local_ms and
    units_per_rank / time. Collective use: one MAX all-reduce of a scalar (timing only).
    """
    world = 1
    t_max = float(local_ms)
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        world = torch.distributed.get_world_size()
        tt = torch.tensor([float(local_ms)], dtype=torch.float64, device=device)
        torch.distributed.all_reduce(tt, op=torch.distributed.ReduceOp.MAX)
        t_max = float(tt.item())
    return t_max, world * units_per_rank / (t_max / 1000.0)


DECODE = "decode_8x262144"
# Small configurations of the same kernels, for profiler captures that must stay short.
PROFILE_JOBS = ["decode_8x32768", "fp8_prefill_16k"]
JOBS = sorted(inputs.WORKLOADS) + [DECODE] + PROFILE_JOBS


def load_job(name):
    """(problems, batched): one problem, or the 8 independent decode sequences."""
    if name == DECODE:
        return inputs.decode_batch(**{k: v for k, v in inputs.DECODE_BATCH.items()}), True
    if name == "decode_8x32768":
        return inputs.decode_batch(B=8, S=32768, pos=32767, seed=4), True
    if name == "fp8_prefill_16k":
        return [inputs.make(name, T=16384, S=16384, pos_offset=0, seed=3,
                            dtype=inputs.FP8_E4M3)], False
    return [inputs.workload(name)], False


def cpu_baseline(probs, budget_s=10.0):
    """Times the fp64 oracle on a bounded row sample of the workload (all host threads)."""
    from oracle import oracle as orc
    if len(probs) > 1:  # independent decode sequences: one row each
        t0 = time.perf_counter()
        for p in probs:
            q, k = p.codes()
            orc.topk(p.dtype, q, p.w.numpy(), k, p.kscale.numpy(), p.pos_offset, p.topk)
        dt = time.perf_counter() - t0
        return {"value": len(probs) / dt, "unit": UNIT, "cores": orc.num_threads(),
                "kind": "oracle",
                "sample": f"all {len(probs)} decode queries ({probs[0].S} keys each), {dt:.1f} s "
                          f"(the oracle scores a row on one thread; its key decode uses all)"}
    prob = probs[0]
    q, k = prob.codes()
    ks = None if prob.kscale is None else prob.kscale.numpy()
    w = prob.w.numpy()
    threads = orc.num_threads()
    # calibration: a few rows spread over the sequence
    n_rows = max(1, min(prob.T, threads))
    rows = np.linspace(0, prob.T - 1, n_rows).round().astype(np.int64)
    t0 = time.perf_counter()
    orc.topk(prob.dtype, q, w, k, ks, prob.pos_offset, prob.topk, rows)
    dt = max(time.perf_counter() - t0, 1e-3)
    n_rows = int(min(prob.T, max(n_rows, n_rows * budget_s / dt)))
    rows = np.unique(np.linspace(0, prob.T - 1, n_rows).round().astype(np.int64))
    t0 = time.perf_counter()
    orc.topk(prob.dtype, q, w, k, ks, prob.pos_offset, prob.topk, rows)
    dt = time.perf_counter() - t0
    return {"value": len(rows) / dt, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{len(rows)} query rows evenly spread over t in [0, {prob.T}) of "
                      f"{prob.name} (full causal rows, fp64 scores + full sort), {dt:.1f} s"}


REF_STEP_S = 1.0  # oracle seconds per reference-arm step


def even_rows(T, n, phase):
    """n query rows spread evenly over [0, T) and shifted by `phase` in [0, 1): a sample with the
    workload's mix of causal row lengths, different for each phase."""
    n = max(1, min(int(n), T))
    return np.unique(np.minimum(((np.arange(n) + phase) * (T / n)).astype(np.int64), T - 1))


def run_reference(args, rank, world):
    """Reference arm: the fp64 CPU oracle, timed on this host's cores (rank 0 only). Each step is
    the same kind of sample `cpu_baseline` times: one decode query (the job's sequences in turn),
    or about REF_STEP_S seconds of query rows spread evenly over the sequence (a new phase each
    step)."""
    if rank != 0:
        return
    probs, _ = load_job(args.workload)
    prob = probs[0]
    from oracle import oracle as orc
    threads = orc.num_threads()
    rng = np.random.default_rng(0)
    if len(probs) > 1:  # independent decode sequences: one query per step, in turn
        prepared = [(p, *p.codes()) for p in probs]
        turn = [0]

        def one_step():
            p, q, k = prepared[turn[0] % len(prepared)]
            turn[0] += 1
            orc.topk(p.dtype, q, p.w.numpy(), k, p.kscale.numpy(), p.pos_offset, p.topk)
            return 1
        sample = (f"one decode query ({prob.S} keys) per step, the job's {len(probs)} "
                  f"sequences in turn (the oracle scores a row on one thread; its key decode "
                  f"uses all)")
    else:
        q, k = prob.codes()
        ks = None if prob.kscale is None else prob.kscale.numpy()
        w = prob.w.numpy()
        n_cal = min(prob.T, 4 * threads)
        t0 = time.perf_counter()
        orc.topk(prob.dtype, q, w, k, ks, prob.pos_offset, prob.topk, even_rows(prob.T, n_cal, 0.5))
        dt = max(time.perf_counter() - t0, 1e-3)
        per_step = int(min(prob.T, max(n_cal, n_cal * REF_STEP_S / dt)))

        def one_step():
            rows = even_rows(prob.T, per_step, rng.random())
            orc.topk(prob.dtype, q, w, k, ks, prob.pos_offset, prob.topk, rows)
            return len(rows)
        sample = (f"{per_step} query rows per step spread evenly over t in [0, {prob.T}) with a "
                  f"random phase, of {prob.name} (full causal rows, fp64 scores + full sort)")
    times = []
    done = 0
    for step in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        n = one_step()
        dt = time.perf_counter() - t0
        if step >= args.warmup:
            times.append(dt)
            done += n
    total = sum(times)
    value = done / total
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * total / args.steps,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic",
           "config": {"workload": args.workload, "B": len(probs), "T": prob.T, "S": prob.S,
                      "H_I": inputs.H_I, "d_I": inputs.D_I, "topk": prob.topk,
                      "pos_offset": prob.pos_offset, "seed": prob.meta.get("seed")},
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                            "sample": sample},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def run_ours(args, rank, world, local_rank):
    from sparse_attention_lightning_indexer_gb300 import ds4idx
    from sparse_attention_lightning_indexer_gb300 import build as _build
    torch.cuda.set_device(local_rank)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    if rank == 0 or not _build.up_to_date():
        if world == 1 or rank == 0:
            _build.build()
    if world > 1:
        torch.distributed.barrier()
    ds4idx.load()

    probs, batched = load_job(args.workload)
    prob = probs[0]
    B = len(probs)
    dev = torch.device("cuda", local_rank)
    log(f"[rank {rank}] workload {args.workload}: B={B} T={prob.T} S={prob.S} dtype={prob.dtype}")

    def stacked(attr):
        ts = [getattr(p, attr) for p in probs]
        if ts[0] is None:
            return None
        return torch.stack(ts) if batched else ts[0]

    host = {a: stacked(a) for a in ("q", "w", "k", "kscale")}
    q, w, k = (host[a].to(dev) for a in ("q", "w", "k"))
    ks = None if host["kscale"] is None else host["kscale"].to(dev)
    ix = ds4idx.Indexer(prob.dtype, max_T=prob.T, max_S=prob.S, max_batch=B)
    stream = torch.cuda.current_stream()
    out_shape = (B, prob.T, prob.topk) if batched else (prob.T, prob.topk)
    out_idx = torch.empty(out_shape, dtype=torch.int32, device=dev)
    out_sc = torch.empty(out_shape, dtype=torch.float32, device=dev)
    positions = [p.pos_offset for p in probs]
    units_per_step = B * prob.T

    def step():
        if batched:
            ix.score_topk_batched(q, w, k, ks, positions, out_idx, out_sc, stream=stream)
        else:
            ix.score_topk(q, w, k, ks, prob.pos_offset, out_idx, out_sc, stream=stream)

    for _ in range(args.warmup):
        step()
    ix.sync_status()

    # ---- device-resident timing: K back-to-back steps between two events, barrier + sync on
    # both sides. No event sits between the steps: each launch is a programmatic dependent of
    # the previous one and may start its setup during that launch's tail.
    with ClockSampler(local_rank) as clk:
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        launched0 = ds4idx.kernels_launched()
        ev0.record(stream)
        for i in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        total_ms = ev0.elapsed_time(ev1)
        launched = ds4idx.kernels_launched() - launched0
    ix.sync_status()
    t_max, value = aggregate(total_ms, units_per_step * args.steps, device=dev)
    ms_per_step = t_max / args.steps

    # ---- end to end through the C ABI with pinned host buffers
    hq, hw, hk = (host[a].pin_memory() for a in ("q", "w", "k"))
    hks = None if host["kscale"] is None else host["kscale"].pin_memory()
    ho_idx = torch.empty(out_shape, dtype=torch.int32).pin_memory()
    ho_sc = torch.empty(out_shape, dtype=torch.float32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (hq, hw, hk) + ((hks,) if hks is not None else ()))
    d2h = ho_idx.numel() * 4 + ho_sc.numel() * 4

    def e2e_step():
        q.copy_(hq, non_blocking=True)
        w.copy_(hw, non_blocking=True)
        k.copy_(hk, non_blocking=True)
        if ks is not None:
            ks.copy_(hks, non_blocking=True)
        step()
        ho_idx.copy_(out_idx, non_blocking=True)
        ho_sc.copy_(out_sc, non_blocking=True)

    e2e_steps = max(3, min(args.steps // 2, 20))
    e2e_step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    ix.sync_status()
    e2e_ms, e2e_value = aggregate(e0.elapsed_time(e1), units_per_step * e2e_steps, device=dev)

    # ---- spot parity check of a few rows against the oracle (outside every timed region)
    spot = "skipped"
    if rank == 0:
        try:
            from tests import parity
            gi_all, gs_all = out_idx.cpu().numpy(), out_sc.cpu().numpy()
            checks = ([(b, [0]) for b in (0, B - 1)] if batched
                      else [(0, [0, prob.T // 3, prob.T - 1])])
            for b, rows in checks:
                gi = gi_all[b][rows] if batched else gi_all[rows]
                gs = gs_all[b][rows] if batched else gs_all[rows]
                parity.check_rows(probs[b], rows, gi, gs)
            spot = f"{sum(len(r) for _, r in checks)} rows match the oracle"
        except AssertionError as e:  # reported, never hidden
            spot = f"MISMATCH: {e}"

    if rank != 0:
        if world > 1:
            torch.distributed.barrier()
            torch.distributed.destroy_process_group()
        ix.close()
        return

    peaks, peak_src = load_peaks()
    avg_step_ms = total_ms / args.steps  # this rank's average launch duration
    flops, key_bytes, pairs = algorithmic(prob)
    flops *= B
    key_bytes *= B
    pairs *= B
    moved = all_bytes(prob) * B
    all_bytes_note = {"bytes": moved, "GB/s": moved / (avg_step_ms / 1000.0) / 1e9,
                      "what": "q + w + key cache (+ scales) + out_idx + out_score, once each"}
    if prob.T == 1:
        # decode: every visible key is read once from HBM per query; bytes bound the step
        achieved = key_bytes / (avg_step_ms / 1000.0) / 1e9
        roofline = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                    "traffic": traffic_for(args.workload),
                    "peak_source": f"hbm copy bandwidth, {peak_src}",
                    "algorithmic": f"{key_bytes:.4g} B = {B} x {prob.S} keys x 132 B "
                                   f"(128 B E4M3 + 4 B scale)",
                    "timed": "one indexer launch per step (split lists merged in-kernel); "
                             "average over K back-to-back launches",
                    "all_bytes": all_bytes_note}
    else:
        if prob.dtype == inputs.BF16:
            peak = peaks["bf16_tflops"]
            peak_note = f"bf16 dense, {peak_src} (burst)"
        else:
            peak = peaks["bf16_tflops"] * FP8_OVER_BF16
            peak_note = f"fp8 dense = {peak_src} bf16 burst x {FP8_OVER_BF16} (nominal ratio)"
        achieved = flops / (avg_step_ms / 1000.0) / 1e12
        roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "frac": achieved / peak, "traffic": traffic_for(args.workload),
                    "peak_source": peak_note,
                    "algorithmic": f"{flops:.4g} flop = 2*64*128 * {pairs:.4g} visible pairs",
                    "timed": "one indexer launch per step; average over K back-to-back "
                             "launches",
                    "all_bytes": all_bytes_note}
    cpu = cpu_baseline(probs, budget_s=args.cpu_budget) if args.cpu_budget > 0 else None
    out = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None,
           "dtype": "bf16" if prob.dtype == inputs.BF16 else "fp8_e4m3",
           "data": "synthetic",
           "config": {"workload": args.workload, "B": B, "T": prob.T, "S": prob.S,
                      "H_I": inputs.H_I, "d_I": inputs.D_I, "topk": prob.topk,
                      "pos_offset": positions if batched else prob.pos_offset,
                      "seed": prob.meta.get("seed"),
                      "l2": "inputs larger than L2 (%s is %.0f MiB)" % (
                          ("key cache", k.numel() * k.element_size() / 2**20) if prob.T == 1
                          else ("q", q.numel() * q.element_size() / 2**20)),
                      "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
           "roofline": roofline,
           "cpu_baseline": cpu,
           "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                   "d2h_bytes_per_step": d2h, "steps": e2e_steps},
           "gpu_launches": launched,
           "clocks": clk.summary(),
           "parity_spot_check": spot}
    print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    ix.close()


# The FP8 index-cache writer over the 128k FP8 workload: one step quantises its 131072 query
# tokens (bf16 in, one scale per token, folded into w) and its 131072 new keys (bf16 in).
WRITER_JOBS = {"fp8_cache_write_128k": dict(T=131072, S=131072, seed=3)}


def _timed(step, steps, stream, world, dev, local_rank):
    from sparse_attention_lightning_indexer_gb300 import ds4idx
    with ClockSampler(local_rank) as clk:
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        launched0 = ds4idx.kernels_launched()
        ev0.record(stream)
        for _ in range(steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        launched = ds4idx.kernels_launched() - launched0
    return ev0.elapsed_time(ev1), launched, clk.summary()


def run_writer(args, rank, world, local_rank):
    """Benchmark of the FP8 index-cache writer (HBM-bound): tokens quantised per second."""
    from sparse_attention_lightning_indexer_gb300 import ds4idx
    from sparse_attention_lightning_indexer_gb300 import build as _build
    torch.cuda.set_device(local_rank)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    if world == 1 or rank == 0:
        _build.build()
    if world > 1:
        torch.distributed.barrier()
    ds4idx.load()
    spec = WRITER_JOBS[args.workload]
    T, S, seed = spec["T"], spec["S"], spec["seed"]
    qf, kf, wf = inputs.draw_f32(T, S, seed)
    hq, hk, hw = qf.to(torch.bfloat16), kf.to(torch.bfloat16), wf
    del qf, kf
    dev = torch.device("cuda", local_rank)
    q, k, w = hq.to(dev), hk.to(dev), hw.to(dev)
    qc = torch.empty((T, inputs.H_I, inputs.D_I), dtype=torch.uint8, device=dev)
    wo = torch.empty((T, inputs.H_I), dtype=torch.float32, device=dev)
    qs = torch.empty((T,), dtype=torch.float32, device=dev)
    kc = torch.empty((S, inputs.D_I), dtype=torch.uint8, device=dev)
    ks = torch.empty((S,), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        ds4idx.quantize_queries(q, w, qc, wo, qs, stream=stream)
        ds4idx.quantize_keys(k, kc, ks, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    total_ms, launched, clocks = _timed(step, args.steps, stream, world, dev, local_rank)
    units = T + S
    t_max, value = aggregate(total_ms, units * args.steps, device=dev)

    # end to end: bf16 inputs from pinned host memory, codes, scales and w' back to the host
    pq, pk, pw = hq.pin_memory(), hk.pin_memory(), hw.pin_memory()
    outs = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (qc, wo, qs, kc, ks)]
    h2d = sum(t.numel() * t.element_size() for t in (pq, pk, pw))
    d2h = sum(t.numel() * t.element_size() for t in outs)

    def e2e_step():
        q.copy_(pq, non_blocking=True)
        k.copy_(pk, non_blocking=True)
        w.copy_(pw, non_blocking=True)
        step()
        for h, d in zip(outs, (qc, wo, qs, kc, ks)):
            h.copy_(d, non_blocking=True)

    e2e_steps = max(3, min(args.steps // 2, 20))
    e2e_step()
    torch.cuda.synchronize()
    e2e_ms, _, _ = _timed(e2e_step, e2e_steps, stream, world, dev, local_rank)
    _, e2e_value = aggregate(e2e_ms, units * e2e_steps, device=dev)

    spot = "skipped"
    cpu = None
    if rank == 0:
        from oracle import oracle as orc
        rows = np.linspace(0, T - 1, 64).astype(np.int64)
        c, sc = orc.quantize_rows(hq[rows].float().reshape(len(rows), -1).numpy())
        ok = np.array_equal(qc[rows].cpu().numpy().reshape(len(rows), -1), c) and \
            np.array_equal(qs[rows].cpu().numpy(), sc)
        kr = np.linspace(0, S - 1, 4096).astype(np.int64)
        c2, s2 = orc.quantize_rows(hk[kr].float().numpy())
        ok = ok and np.array_equal(kc[kr].cpu().numpy(), c2) and np.array_equal(ks[kr].cpu().numpy(), s2)
        spot = "64 query tokens and 4096 keys bit-exact with the oracle" if ok else "MISMATCH"
        if args.cpu_budget > 0:
            def oracle_tokens(n):  # n query tokens and n keys
                t0 = time.perf_counter()
                orc.quantize_rows(hq[:n].float().reshape(n, -1).numpy())
                orc.quantize_rows(hk[:n].float().numpy())
                return time.perf_counter() - t0
            n_tok = 256
            dt = oracle_tokens(n_tok)
            n_tok = int(min(T, max(n_tok, n_tok * args.cpu_budget / max(dt, 1e-3))))
            dt = oracle_tokens(n_tok)
            cpu = {"value": 2 * n_tok / dt, "unit": "tokens/s", "cores": orc.num_threads(),
                   "kind": "oracle",
                   "sample": f"the first {n_tok} query tokens and {n_tok} keys of the workload "
                             f"(brute-force E4M3 rounding), {dt:.1f} s"}
    if rank != 0:
        if world > 1:
            torch.distributed.barrier()
            torch.distributed.destroy_process_group()
        return
    peaks, peak_src = load_peaks()
    avg_ms = total_ms / args.steps
    moved = float(T * inputs.H_I * inputs.D_I * (2 + 1) + T * inputs.H_I * 4 * 2 + T * 4
                  + S * inputs.D_I * (2 + 1) + S * 4)
    achieved = moved / (avg_ms / 1000.0) / 1e9
    out = {"metric": "FP8 index-cache writer tokens/s (queries + keys quantised) and % of HBM",
           "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": t_max / args.steps, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "bf16->e4m3", "data": "synthetic",
           "config": {"workload": args.workload, "T": T, "S": S, "H_I": inputs.H_I,
                      "d_I": inputs.D_I, "seed": seed,
                      "l2": "inputs larger than L2 (q is %.0f MiB)" % (q.numel() * 2 / 2**20),
                      "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
           "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                        "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"], "traffic": None,
                        "peak_source": f"hbm copy bandwidth, {peak_src}",
                        "algorithmic": f"{moved:.4g} B: bf16 q and k read once, E4M3 codes, "
                                       f"scales, w read and w' written once",
                        "timed": "two launches per step (queries, keys); average over K steps"},
           "cpu_baseline": cpu,
           "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                   "d2h_bytes_per_step": d2h, "steps": e2e_steps},
           "gpu_launches": launched, "clocks": clocks, "parity_spot_check": spot}
    print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


# Sparse attention over the indexer's Top-512: the last 4096 query tokens of a 64k-token
# sequence (indices from an indexer call on those rows), 128 heads over 576-wide latent rows.
ATTN_JOBS = {"sparse_attn_4k_of_64k": dict(T=4096, S=65536, pos_offset=61440, seed=2)}


def run_attention(args, rank, world, local_rank):
    """Benchmark of sparse attention over the selected keys (tensor-bound): query tokens/s."""
    from sparse_attention_lightning_indexer_gb300 import ds4idx
    from sparse_attention_lightning_indexer_gb300 import build as _build
    torch.cuda.set_device(local_rank)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    if world == 1 or rank == 0:
        _build.build()
    if world > 1:
        torch.distributed.barrier()
    ds4idx.load()
    spec = ATTN_JOBS[args.workload]
    T, S, pos, seed = spec["T"], spec["S"], spec["pos_offset"], spec["seed"]
    dev = torch.device("cuda", local_rank)
    # the selection: the indexer on these queries (untimed)
    prob = inputs.make(args.workload, T=T, S=S, pos_offset=pos, seed=seed, dtype=inputs.BF16)
    with ds4idx.Indexer(inputs.BF16, max_T=T, max_S=S) as ix:
        idx, _ = ix.score_topk(prob.q.to(dev), prob.w.to(dev), prob.k.to(dev), None, pos)
        ix.sync_status()
    g = torch.Generator().manual_seed(seed * 1009 + 11)
    hq = torch.randn(T, ds4idx.SA_HEADS, ds4idx.SA_DQK, generator=g).to(torch.bfloat16)
    hkv = torch.randn(S, ds4idx.SA_DQK, generator=g).to(torch.bfloat16)
    hidx = idx.cpu()
    q, kv = hq.to(dev), hkv.to(dev)
    scale = ds4idx.SA_DQK ** -0.5
    out = torch.empty((T, ds4idx.SA_HEADS, ds4idx.SA_DV), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((T, ds4idx.SA_HEADS), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        ds4idx.sparse_attention(q, kv, idx, scale, out=out, lse=lse, stream=stream)

    for _ in range(args.warmup):
        step()
    ds4idx.sparse_attention_status()
    total_ms, launched, clocks = _timed(step, args.steps, stream, world, dev, local_rank)
    ds4idx.sparse_attention_status()
    t_max, value = aggregate(total_ms, T * args.steps, device=dev)
    pq, pkv, pidx = hq.pin_memory(), hkv.pin_memory(), hidx.pin_memory()
    pout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    plse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (pq, pkv, pidx))
    d2h = pout.numel() * 2 + plse.numel() * 4

    def e2e_step():
        q.copy_(pq, non_blocking=True)
        kv.copy_(pkv, non_blocking=True)
        idx.copy_(pidx, non_blocking=True)
        step()
        pout.copy_(out, non_blocking=True)
        plse.copy_(lse, non_blocking=True)

    e2e_steps = max(3, min(args.steps // 2, 20))
    e2e_step()
    torch.cuda.synchronize()
    e2e_ms, _, _ = _timed(e2e_step, e2e_steps, stream, world, dev, local_rank)
    _, e2e_value = aggregate(e2e_ms, T * e2e_steps, device=dev)
    spot, cpu = "skipped", None
    if rank == 0:
        from oracle import oracle as orc
        rows = np.linspace(0, T - 1, 8).astype(np.int64)
        o_ref, l_ref = orc.sparse_attention(hq, hkv, hidx.numpy(), scale, ds4idx.SA_DV, rows=rows)
        err = float(np.abs(out[rows].float().cpu().numpy() - o_ref).max())
        lerr = float(np.abs(lse[rows].cpu().numpy() - l_ref).max())
        spot = f"8 tokens vs the oracle: max |d out| {err:.3g}, max |d lse| {lerr:.3g}"
        if args.cpu_budget > 0:
            n = max(1, orc.num_threads())
            t0 = time.perf_counter()
            orc.sparse_attention(hq, hkv, hidx.numpy(), scale, ds4idx.SA_DV, rows=np.arange(n))
            dt = time.perf_counter() - t0
            n2 = int(min(T, max(n, n * args.cpu_budget / max(dt, 1e-3))))
            t0 = time.perf_counter()
            orc.sparse_attention(hq, hkv, hidx.numpy(), scale, ds4idx.SA_DV, rows=np.arange(n2))
            dt = time.perf_counter() - t0
            cpu = {"value": n2 / dt, "unit": UNIT, "cores": orc.num_threads(), "kind": "oracle",
                   "sample": f"first {n2} query tokens (fp64, all 128 heads), {dt:.1f} s"}
    if rank != 0:
        if world > 1:
            torch.distributed.barrier()
            torch.distributed.destroy_process_group()
        return
    peaks, peak_src = load_peaks()
    avg_ms = total_ms / args.steps
    valid = int((hidx >= 0).sum())
    flops = 2.0 * ds4idx.SA_HEADS * valid * (ds4idx.SA_DQK + ds4idx.SA_DV)
    achieved = flops / (avg_ms / 1000.0) / 1e12
    out_line = {"metric": "sparse attention query-tokens/s over the Top-512 (128 heads, 576/512 "
                          "latent) and % of bf16 tensor roofline",
                "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": t_max / args.steps,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                "data": "synthetic",
                "config": {"workload": args.workload, "T": T, "S": S, "pos_offset": pos,
                           "heads": ds4idx.SA_HEADS, "d_qk": ds4idx.SA_DQK, "d_v": ds4idx.SA_DV,
                           "topk": 512, "seed": seed,
                           "l2": "q is %.0f MiB (larger than L2); the 72 MiB latent cache fits "
                                 "L2" % (q.numel() * 2 / 2**20),
                           "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
                "roofline": {"bound": "tensor", "achieved": achieved,
                             "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                             "frac": achieved / peaks["bf16_tflops"],
                             "traffic": traffic_for(args.workload),
                             "peak_source": f"bf16 dense, {peak_src} (burst)",
                             "algorithmic": f"{flops:.4g} flop = 2*128*(576+512) * {valid} "
                                            f"selected (token, key) pairs",
                             "timed": "one launch per step; average over K steps"},
                "cpu_baseline": cpu,
                "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                        "d2h_bytes_per_step": d2h, "steps": e2e_steps},
                "gpu_launches": launched, "clocks": clocks, "parity_spot_check": spot}
    print(json.dumps(out_line), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="prefill_64k",
                    choices=JOBS + sorted(WRITER_JOBS) + sorted(ATTN_JOBS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of oracle time for cpu_baseline (0 disables)")
    args = ap.parse_args()
    if args.warmup < 3:
        log("warmup raised to 3 (minimum)")
        args.warmup = 3
    rank, world, local_rank = dist_env()
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        # Plain `python bench.py --gpus N`: start N ranks (one process per GPU) under torchrun.
        cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
               f"--nproc-per-node={args.gpus}", "--master-addr=127.0.0.1",
               f"--master-port={29500 + os.getpid() % 1000}", os.path.abspath(__file__),
               *sys.argv[1:]]
        log("starting", args.gpus, "ranks:", " ".join(cmd))
        sys.exit(subprocess.call(cmd))
    if world != args.gpus:
        log(f"--gpus {args.gpus} disagrees with WORLD_SIZE={world}")
        sys.exit(2)
    if args.impl == "reference":
        run_reference(args, rank, world)
    elif args.workload in WRITER_JOBS:
        run_writer(args, rank, world, local_rank)
    elif args.workload in ATTN_JOBS:
        run_attention(args, rank, world, local_rank)
    else:
        run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
