"""Benchmark: weight-absorbed MLA decode (partial + LSE combine) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config dp16]
                    [--impl reference]

One step is one pass of the whole hot path over one batch: the split plan
(computed once per batch shape, before timing, from the host lengths), the
tensor-core partial decode launch and the LSE-combine launch.  The default
workload is 16 requests x q_len 5 x 96 heads x 100k-token context, BF16
latent KV in 64-token pages with a random page permutation, synthetic N(0,1)
data (seed = rank).

value      attention TFLOP/s over all ranks, inputs resident in HBM
           (algorithmic FLOPs 2*H*(576+512)*sum_b sum_i (L_b - q_len + 1 + i)
           per step / device time), max over ranks of the timed region
e2e        the same metric through the public API from pinned host buffers:
           every step plans itself on the host, copies the queries, page
           table, lengths and plan to the device and reads the output and LSE
           back (the KV cache is resident state); consecutive steps overlap on
           three streams, as a serving loop runs them ("serial": the same
           steps one at a time, i.e. one step's latency)
roofline   the partial-decode kernel alone: algorithmic FLOPs / its mean
           CUDA-event duration inside the timed region vs measured bf16 peak
cpu_baseline  the fp64 oracle on a bounded sample of rows, host cores

With N > 1 (torchrun) every rank decodes its own batch of the same shape
(independent requests, no collective on the data path): weak scaling.
"""
from __future__ import annotations

import argparse
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
sys.path.insert(0, ROOT)

METRIC = ("MLA decode µs/layer & attention TFLOP/s at 100k ctx; "
          "% of GB300 tensor peak")
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "tc_partial_traffic.json")


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="dp16")
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--splits", type=int, default=0, help="0: planner")
    ap.add_argument("--planner", choices=("sched", "parts"), default="sched",
                    help="sched: parts and longest-first launch order "
                         "(mla_plan_sched); parts: parts in part-major order "
                         "(mla_plan_parts)")
    ap.add_argument("--parts-cut", type=int, default=0,
                    help="two parts per request, the first of this many pages "
                         "(reproduces a larger workload's per-request plan on "
                         "fewer requests, e.g. for a traffic capture)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--kv-write-rows", type=int, default=0,
                    help="time mla_kv_write of this many rows to random slots "
                         "instead of the decode step (with --config's KV dtype)")
    ap.add_argument("--projections", action="store_true",
                    help="time mla_absorb_q and mla_project_out at --config's "
                         "rows (B * q_len) and heads instead of the decode step")
    ap.add_argument("--parts", choices=("f32", "bf16"), default="bf16",
                    help="partial outputs between the two launches: bf16 "
                         "(mla_decode_partial_bf16_parts) or fp32")
    ap.add_argument("--fused", action="store_true",
                    help="time mla_decode (partial + combine in one launch) "
                         "instead of mla_decode_partial + mla_lse_combine")
    ap.add_argument("--sweep", action="store_true",
                    help="wave-quantisation sweep: B in 1..24 x context "
                         "{100k, 400k}, the pages' split rule vs the planner "
                         "(one JSON line per point)")
    ap.add_argument("--c0-scan", action="store_true",
                    help="time the scheduler's plans for unit costs c0 in "
                         "{4, 8, 12, 16, 24, 32} on the 100k sweep, dp16, DCP, "
                         "ragged FP8 and FP8 sweep points (refits the planners' "
                         "unit cost), one JSON line per workload")
    ap.add_argument("--sweep-scan", default="",
                    help="extra comma-separated split counts to time at "
                         "every sweep point")
    return ap.parse_args(argv)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def slowest_rank(local, dist=None, device="cpu"):
    """The job's time for a region every rank times on its own clock: the
    slowest rank's (max over ranks; the local value without a process
    group)."""
    if dist is None:
        return float(local)
    import torch
    t = torch.tensor([float(local)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_rank_step, steps, world, seconds):
    """Whole-job throughput: every rank decodes its own batch (data
    parallel, no collective on the data path), so the job processes world x
    the per-rank FLOPs in the slowest rank's time."""
    return world * flops_per_rank_step * steps / seconds / 1e12


def workload_desc(wl):
    lens = wl.seq_lens
    ctx = lens[0] if len(set(lens)) == 1 else f"{min(lens)}..{max(lens)}"
    return (f"{wl.name}: {wl.B} requests x q_len {wl.q_len} x {wl.H} heads x "
            f"{ctx} context, {wl.kv_dtype} latent KV (576-d rows), page "
            f"{wl.page_size}" + (f", {wl.num_shards} interleaved shards"
                                 if wl.num_shards > 1 else ""))


def measured_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))), "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0,
                "bf16_tflops_sustained": 1700.0}, "fallback"


def kernel_source_hash(fp8=False, kernel=None):
    """Hash of the sources the BF16 (or FP8) tensor-core decode kernel
    compiles from, or with kernel="projection" the per-head projection
    kernel's."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mla_latent_decode_gb300", "csrc")
    main = ("mla_absorb.cu" if kernel == "projection"
            else "mla_tc_fp8.cu" if fp8 else "mla_tc.cu")
    for f in (main, "ptx_sm103.cuh", "mla_tma.cuh", "mla_internal.h"):
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(config_name, units, fp8=False, kernel=None):
    """DRAM bytes per launch from a committed ncu summary, only if it was
    taken on the current source of the kernel the workload runs; scaled by
    units if captured smaller."""
    try:
        d = json.load(open(PROFILE_TRAFFIC))
    except Exception:
        return None
    e = d.get("workloads", {}).get(config_name)
    if not e or e.get("kernel_source_hash") != kernel_source_hash(fp8, kernel):
        return None
    return e["dram_bytes_per_launch"] * units / e.get("units", units)


class ClockSampler:
    """nvidia-smi clock/throttle samples taken while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.flush()
        rows = []
        for line in open(self.out.name):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(parts)
            except Exception:
                pass
        os.unlink(self.out.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4)
                          if r[5 + k].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "samples": len(rows), "reasons": reasons}


def oracle_sample(batch, hb, seconds, rank_seed=0):
    """Time the fp64 oracle on a bounded sample of rows; returns the
    cpu_baseline object in the metric's unit (TFLOP/s)."""
    import numpy as np
    import oracle

    wl = batch.wl
    r2t, sl, kl = hb["req_to_token"], hb["seq_lens"], hb["kv_limit"]
    rng = np.random.default_rng(rank_seed)
    threads = oracle.num_threads()

    def rows_flops(rows):
        tot = 0
        per = wl.q_len * wl.H
        for r in rows:
            b, i = divmod(int(r) // wl.H, wl.q_len)
            L = int(sl[b])
            n = int(kl[b, i]) if kl is not None else L - wl.q_len + 1 + i
            tot += 2 * (576 + 512) * max(0, min(n, L))
        return tot

    B_q = wl.B
    shard_r2t = r2t[:B_q]
    shard_sl = sl[:B_q]
    shard_kl = None if kl is None else kl[:B_q]
    # calibrate on one row per thread, then size the sample to `seconds`
    n_rows = max(threads, 1)
    rows = rng.choice(wl.rows, size=min(n_rows, wl.rows), replace=False)
    t0 = time.perf_counter()
    oracle.mla_decode_rows(hb["q_nope"], hb["q_rope"], hb["kv"], batch.kv_is_fp8,
                           hb["kv_scale"], shard_r2t, shard_sl, shard_kl, B_q,
                           wl.q_len, wl.H, wl.sm_scale, rows)
    dt = time.perf_counter() - t0
    want = int(len(rows) * max(1.0, seconds / max(dt, 1e-3)))
    rows = rng.choice(wl.rows, size=min(want, wl.rows), replace=False)
    t0 = time.perf_counter()
    oracle.mla_decode_rows(hb["q_nope"], hb["q_rope"], hb["kv"], batch.kv_is_fp8,
                           hb["kv_scale"], shard_r2t, shard_sl, shard_kl, B_q,
                           wl.q_len, wl.H, wl.sm_scale, rows)
    dt = time.perf_counter() - t0
    fl = rows_flops(rows)
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": threads,
            "kind": "oracle",
            "sample": (f"{len(rows)} of {wl.rows} query rows of the same "
                       f"workload (shard 0 where sharded), full visible "
                       f"context each, {dt:.1f} s wall, fp64"),
            "seconds": dt}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import torch
    from mla_latent_decode_gb300 import synth

    wl = synth.config(args.config)
    batch = synth.make_batch(wl, seed=0, device="cpu")
    hb = synth.host_bits(batch)
    per_step = max(1.0, args.cpu_seconds / max(1, args.steps + args.warmup))
    vals, walls = [], []
    for k in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        cb = oracle_sample(batch, hb, per_step, rank_seed=k)
        if k >= args.warmup:
            vals.append(cb)
            walls.append(time.perf_counter() - t0)
    v = statistics.median(c["value"] for c in vals)
    fl = wl.flops()
    # A step of this arm is one bounded sample of the workload's rows (with
    # its calibration run): ms_per_step is that sample's measured wall time;
    # the full workload at the sampled rate is reported beside it.
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": statistics.median(walls) * 1e3,
        "ms_per_full_step_projected": fl / (v * 1e12) * 1e3,
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": workload_desc(wl)},
        "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": vals[0]["cores"],
                         "kind": "oracle", "sample": vals[0]["sample"]},
        "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


PARTS = {"dtype": "bf16"}  # the --parts choice, read by every step builder


def part_dtype(wl):
    """Element type of the partial outputs (the --parts choice)."""
    import torch
    return torch.bfloat16 if PARTS["dtype"] == "bf16" else torch.float32


def time_pair(mla, batch, wl, S, iters, warmup=3, split_pages=None, work=None):
    """Median device time (ms) of one partial-decode + combine pair at S
    splits, CUDA events on the launching stream.  The steps are enqueued back
    to back (no host synchronisation between them, so the host's launch work
    overlaps the previous step instead of sitting between the events); with
    KV smaller than twice the L2 a 256-MB buffer is written between steps,
    outside the events, so every step reads its inputs from DRAM."""
    import torch
    dev = batch.q_nope.device
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    O_part = torch.empty((S, wl.num_shards, wl.B, wl.q_len, wl.H, 512),
                         dtype=part_dtype(wl), device=dev)
    LSE_part = torch.empty((S, wl.num_shards, wl.B, wl.q_len, wl.H),
                           dtype=torch.float32, device=dev)
    out = torch.empty((wl.B, wl.q_len, wl.H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((wl.B, wl.q_len, wl.H), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def run():
        mla.decode_partial(batch.q_nope, batch.q_rope, batch.kv, batch.kv_scale,
                           batch.req_to_token, batch.seq_lens, batch.kv_limit, S,
                           wl.sm_scale, wl.num_shards, O_part, LSE_part, status,
                           split_pages=split_pages, work=work)
        mla.lse_combine(O_part, LSE_part, out, lse)

    kv_bytes = batch.kv.numel() * batch.kv.element_size()
    flush_buf = (torch.empty(256 * 2**20, dtype=torch.uint8, device=dev)
                 if kv_bytes < 256 * 2**20 else None)
    for _ in range(warmup):
        run()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(iters)]
    for k, (a, b) in enumerate(evs):
        if flush_buf is not None:
            flush_buf.fill_(k & 0xFF)
        a.record(stream)
        run()
        b.record(stream)
    torch.cuda.synchronize()
    ts = [a.elapsed_time(b) for a, b in evs]
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")
    return statistics.median(ts)


def run_c0_scan(args):
    """The scheduler's plans (mla_plan_sched_ex) for a range of unit costs c0,
    each distinct plan timed as a partial + combine pair: the data the
    planners' default unit costs are fitted to."""
    import torch

    import mla_latent_decode_gb300 as mla
    from mla_latent_decode_gb300 import synth
    mla.library()
    c0s = [4.0, 8.0, 12.0, 16.0, 24.0, 32.0]
    configs = [f"sweep_B{B}_L100000" for B in (1, 2, 4, 8, 12, 16, 20, 24)]
    configs += ["dp16", "dcp", "ragged_fp8"]
    configs += [f"sweep8_B{B}_L100000" for B in (4, 8, 16, 24)]
    for name in configs:
        wl = synth.config(name)
        batch = synth.make_batch(wl, seed=0, device="cuda")
        lens = mla.batch_lengths(batch)
        fp8 = wl.kv_dtype != "bf16"
        dev = batch.q_nope.device
        timed, res = {}, {}
        for c0 in c0s:
            S, bnd, work, _, ms = mla.plan_sched_ex(
                lens, wl.q_len, wl.H, 76 if fp8 else 36, 64, 8, c0, 1.0,
                rows_per_unit=128 if fp8 else 256)
            key = (S, bnd.tobytes(), work.tobytes())
            if key not in timed:
                iters = 20 if wl.B * max(wl.seq_lens) < 5e6 else 8
                timed[key] = 1e3 * time_pair(
                    mla, batch, wl, S, iters, split_pages=torch.from_numpy(bnd).to(dev),
                    work=torch.from_numpy(work).to(dev))
            res[str(c0)] = {"splits": S, "us": timed[key], "model_makespan": ms}
        print(json.dumps({"impl": "c0_scan", "config": name,
                          "slots": 76 if fp8 else 36, "unit": "us per layer "
                          "(partial + combine)", "by_c0": res}), flush=True)
        del batch
        torch.cuda.empty_cache()
    return 0


def run_sweep(args):
    """Wave-quantisation sweep: for every (B, context) point, the pair timed
    with the pages' split rule and with the planner's split (and any extra
    split counts asked for), one JSON line per point (time_pair: device time
    per step, the L2 flushed between steps when the KV is smaller than twice
    the L2)."""
    import torch

    import mla_latent_decode_gb300 as mla
    from mla_latent_decode_gb300 import synth

    mla.library()
    extra = [int(x) for x in args.sweep_scan.split(",") if x.strip()]
    slots = mla.cluster_slots()
    for L in (100_000, 400_000):
        for B in (1, 2, 4, 8, 12, 16, 20, 24):
            wl = synth.config(f"sweep_B{B}_L{L}")
            batch = synth.make_batch(wl, seed=0, device="cuda")
            lens = mla.batch_lengths(batch)
            S_plan, eff = mla.plan(wl.B, wl.q_len, wl.H, lens, wl.num_shards,
                                   kv_dtype=wl.kv_dtype)
            S_rule = mla.plan_heuristic(wl.B, wl.q_len)
            fl = wl.flops()
            iters = max(5, min(args.steps, int(2000 / max(1, B * L / 100_000))))
            res = {}
            for S in sorted({S_plan, S_rule, *extra}):
                ms = time_pair(mla, batch, wl, S, iters)
                res[S] = {"us": ms * 1e3, "tflops": fl / (ms * 1e-3) / 1e12}
            S_parts, bnd, eff_parts = mla.plan_parts(
                wl.B, wl.q_len, wl.H, lens, wl.num_shards, kv_dtype=wl.kv_dtype)
            ms = time_pair(mla, batch, wl, S_parts, iters,
                           split_pages=torch.from_numpy(bnd).to(batch.q_nope.device))
            parts = {"splits": S_parts, "wave_eff": eff_parts,
                     "first_part_pages": int(bnd[0][1]), "us": ms * 1e3,
                     "tflops": fl / (ms * 1e-3) / 1e12}
            S_s, bnd_s, wk, eff_s = mla.plan_sched(
                wl.B, wl.q_len, wl.H, lens, wl.num_shards, kv_dtype=wl.kv_dtype)
            dev = batch.q_nope.device
            ms = time_pair(mla, batch, wl, S_s, iters,
                           split_pages=torch.from_numpy(bnd_s).to(dev),
                           work=torch.from_numpy(wk).to(dev))
            sched = {"splits": S_s, "wave_eff": eff_s,
                     "first_part_pages": int(bnd_s[0][1]), "us": ms * 1e3,
                     "tflops": fl / (ms * 1e-3) / 1e12}
            print(json.dumps({
                "impl": "sweep", "B": B, "context": L, "q_len": wl.q_len,
                "H": wl.H, "cluster_slots": slots,
                "pages_rule": {"splits": S_rule, **res[S_rule]},
                "planner": {"splits": S_plan, "wave_eff": eff, **res[S_plan]},
                "parts_planner": parts,
                "scheduler": sched,
                "scan": {str(k): v for k, v in sorted(res.items())},
                "unit": "us per layer (partial + combine), attention TFLOP/s",
            }), flush=True)
            del batch
            torch.cuda.empty_cache()
    return 0


def run_kv_write(args):
    """Cache write: N bf16 latent rows stored at random slots of a pool of 2N
    slots (BF16 copy or FP8 quantise), inputs resident in HBM and larger
    than L2.  HBM-bound: algorithmic bytes per row = the bf16 row and its
    slot read, the stored row (and scale) written."""
    import torch

    import mla_latent_decode_gb300 as mla
    from mla_latent_decode_gb300 import synth
    mla.library()
    wl = synth.config(args.config)
    fp8 = wl.kv_dtype != "bf16"
    n = args.kv_write_rows
    dev = torch.device("cuda", 0)
    gen = torch.Generator(device=dev).manual_seed(0)
    rows = torch.randn((n, 576), generator=gen, device=dev).to(torch.bfloat16)
    slots = torch.randperm(2 * n, device=dev)[:n].to(torch.int32)
    kv = torch.zeros((2 * n, 576), dtype=torch.uint8 if fp8 else torch.bfloat16,
                     device=dev)
    scale = torch.zeros((2 * n,), dtype=torch.float32, device=dev) if fp8 else None
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    for _ in range(max(3, args.warmup)):
        mla.kv_write(rows, slots, kv, scale, status)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(0)
    clocks.start()
    time.sleep(0.1)
    t0.record(stream)
    for _ in range(args.steps):
        mla.kv_write(rows, slots, kv, scale, status)
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")
    ms = t0.elapsed_time(t1) / args.steps
    per_row = 1152 + 4 + (576 + 4 if fp8 else 1152)
    gbs = n * per_row / (ms * 1e-3) / 1e9
    peaks, kind = measured_peaks()
    peak = float(peaks["hbm_gbs"])
    print(json.dumps({
        "metric": "MLA KV cache write GB/s (mla_kv_write)", "value": gbs,
        "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3 (quantise)" if fp8 else "bf16 (copy)",
        "data": "synthetic",
        "config": {"workload": f"{n} bf16 latent rows (576-d) to random slots of "
                               f"a {2 * n}-slot {'E4M3' if fp8 else 'BF16'} pool",
                   "l2": f"inputs larger than L2 ({n * 1152 / 1e9:.2f} GB of rows), no flush"},
        "rows_per_s": n / (ms * 1e-3),
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                     "frac": gbs / peak, "traffic": None,
                     "kernel": "mla_kv_write_kernel",
                     "peak_kind": f"{kind} copy bandwidth",
                     "bytes_per_row": per_row},
        "clocks": clk, "gpu_launches": args.steps}))
    return 0


def run_projections(args):
    """The per-head projections around the decode (query absorption, output
    projection) at the workload's B * q_len rows and H heads with synthetic
    weights.  Weight-bound: R copies of each weight (R x 12.6 MB, more than
    L2) are used in turn, R launches are captured in one CUDA graph and the
    graph is replayed, so each launch reads its weights from DRAM and host
    overhead stays out of the device time; HBM roofline on the algorithmic
    bytes."""
    import torch

    import mla_latent_decode_gb300 as mla
    from mla_latent_decode_gb300 import synth
    mla.library()
    wl = synth.config(args.config)
    B, q, H = wl.B, wl.q_len, wl.H
    R = 16
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev).manual_seed(0)
    q_nope = torch.randn((B, q, H, 128), generator=g, device=dev).to(torch.bfloat16)
    o_lat = torch.randn((B, q, H, 512), generator=g, device=dev).to(torch.bfloat16)
    w_kc = [(torch.randn((H, 128, 512), generator=g, device=dev) / 11.3).to(torch.bfloat16)
            for _ in range(R)]
    w_vc = [(torch.randn((H, 512, 128), generator=g, device=dev) / 22.6).to(torch.bfloat16)
            for _ in range(R)]
    q_abs = torch.empty((B, q, H, 512), dtype=torch.bfloat16, device=dev)
    o_v = torch.empty((B, q, H, 128), dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    peaks, kind = measured_peaks()
    M = B * q
    ops = {
        "mla_absorb_q": (lambda r: mla.absorb_q(q_nope, w_kc[r], q_abs, status),
                         M * H * 128 * 2 + H * 128 * 512 * 2 + M * H * 512 * 2),
        "mla_project_out": (lambda r: mla.project_out(o_lat, w_vc[r], o_v, status),
                            M * H * 512 * 2 + H * 512 * 128 * 2 + M * H * 128 * 2),
    }
    clocks = ClockSampler(0)
    clocks.start()
    time.sleep(0.1)
    res = {}
    for name, (fn, nbytes) in ops.items():
        for r in range(R):
            fn(r)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for r in range(R):
                fn(r)
        for _ in range(max(3, args.warmup)):
            graph.replay()
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        stream = torch.cuda.current_stream()
        t0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        t1.record(stream)
        torch.cuda.synchronize()
        us = t0.elapsed_time(t1) * 1e3 / (args.steps * R)
        res[name] = (us, nbytes / (us * 1e-6) / 1e9, nbytes)
    clk = clocks.stop()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")
    total_us = sum(v[0] for v in res.values())
    total_bytes = sum(v[2] for v in res.values())
    gbs = total_bytes / (total_us * 1e-6) / 1e9
    peak = float(peaks["hbm_gbs"])
    # DRAM bytes of one projection pair (both launches), when profiled on
    # the current kernel source
    traffic = profiled_traffic(f"projections_{args.config}", 1, kernel="projection")
    print(json.dumps({
        "metric": "MLA per-head projections us/layer (mla_absorb_q + mla_project_out)",
        "value": total_us, "unit": "us", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_us / 1e3,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (random weights)",
        "config": {"workload": f"{M} rows (B {B} x q_len {q}) x {H} heads: "
                               "q_nope 128 -> 512 (w_kc), o_latent 512 -> 128 (w_vc)",
                   "l2": f"{R} weight copies used in turn ({R * H * 128 * 512 * 2 / 1e6:.0f} MB "
                         "per projection, more than L2); launches replayed from a CUDA graph"},
        "ops": {k: {"us": v[0], "gbs": v[1], "bytes": v[2]} for k, v in res.items()},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                     "frac": gbs / peak, "traffic": traffic,
                     "kernel": "mla_head_gemm_kernel",
                     "peak_kind": f"{kind} copy bandwidth"},
        "clocks": clk, "gpu_launches": 2 * R * args.steps}))
    return 0


def time_e2e(mla, args, wl, batch, lens, S, split_pages, work, counters,
             status, dev, fl, world, dist):
    """End-to-end throughput through the public API from pinned host buffers.

    Every step plans itself on the host from the host lengths (when the run
    uses a planner), copies its queries, page table, lengths, visibility
    limits and plan to the device, decodes, and reads its output and LSE back;
    the KV cache is resident state.  Consecutive steps overlap as a serving
    loop runs them: two sets of device buffers, uploads on one stream, the
    decode on a second, downloads on a third, ordered by events, while the
    host plans the next step.  Every step's plan and copies lie inside the
    timed region."""
    import numpy as np
    import torch
    fixed = args.parts_cut > 0 or args.splits > 0 or bool(wl.num_splits)

    def replan():
        if fixed:
            return None, None
        if args.planner == "parts":
            S2, b2, _ = mla.plan_parts(wl.B, wl.q_len, wl.H, lens, wl.num_shards,
                                       kv_dtype=wl.kv_dtype)
            w2 = None
        else:
            S2, b2, w2, _ = mla.plan_sched(wl.B, wl.q_len, wl.H, lens,
                                           wl.num_shards, kv_dtype=wl.kv_dtype)
        if S2 != S:
            raise RuntimeError(f"the plan changed between steps: {S2} != {S}")
        return b2, w2

    pin = lambda t: t.cpu().pin_memory()
    host_in = [pin(batch.q_nope), pin(batch.q_rope), pin(batch.req_to_token),
               pin(batch.seq_lens)]
    if batch.kv_limit is not None:
        host_in.append(pin(batch.kv_limit))
    b0, w0 = replan()
    h_sp = [torch.from_numpy(b0.copy()).pin_memory() if b0 is not None else None
            for _ in range(2)]
    h_wk = [torch.from_numpy(w0.copy()).pin_memory() if w0 is not None else None
            for _ in range(2)]
    d_in = [[torch.empty_like(h, device=dev) for h in host_in] for _ in range(2)]
    d_sp = [torch.empty_like(h, device=dev) if h is not None else None for h in h_sp]
    d_wk = [torch.empty_like(h, device=dev) if h is not None else None for h in h_wk]
    O_part = torch.empty((S, wl.num_shards, wl.B, wl.q_len, wl.H, 512),
                         dtype=part_dtype(wl), device=dev)
    LSE_part = torch.empty((S, wl.num_shards, wl.B, wl.q_len, wl.H),
                           dtype=torch.float32, device=dev)
    d_out = [torch.empty((wl.B, wl.q_len, wl.H, 512), dtype=torch.bfloat16,
                         device=dev) for _ in range(2)]
    d_lse = [torch.empty((wl.B, wl.q_len, wl.H), dtype=torch.float32, device=dev)
             for _ in range(2)]
    h_out = [torch.empty_like(d, device="cpu").pin_memory() for d in d_out]
    h_lse = [torch.empty_like(d, device="cpu").pin_memory() for d in d_lse]
    s_in, s_dec, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "dec", "out")}
    for k in ev:  # every event recorded once before the first wait on it
        for e in ev[k]:
            e.record()
    bi = sum(h.numel() * h.element_size() for h in host_in)
    bi += sum(h.numel() * h.element_size() for h in (h_sp[0], h_wk[0]) if h is not None)
    bo = sum(d.numel() * d.element_size() for d in (d_out[0], d_lse[0]))

    def e2e_step(k):
        i = k & 1
        with torch.cuda.stream(s_in):
            s_in.wait_event(ev["dec"][i])  # step k - 2's decode is done with set i
            for d, h in zip(d_in[i], host_in):
                d.copy_(h, non_blocking=True)
        # the host plans while the inputs upload
        b2, w2 = replan()
        ev["in"][i].synchronize()  # step k - 2's uploads have read the staging
        if b2 is not None:
            h_sp[i].numpy()[...] = b2
        if w2 is not None:
            h_wk[i].numpy()[...] = w2
        with torch.cuda.stream(s_in):
            if b2 is not None:
                d_sp[i].copy_(h_sp[i], non_blocking=True)
            if w2 is not None:
                d_wk[i].copy_(h_wk[i], non_blocking=True)
            ev["in"][i].record(s_in)
        q, r, r2t, sl = d_in[i][:4]
        kv_limit = d_in[i][4] if batch.kv_limit is not None else None
        sp = d_sp[i] if b2 is not None else split_pages
        wk = d_wk[i] if w2 is not None else work
        with torch.cuda.stream(s_dec):
            s_dec.wait_event(ev["in"][i])
            s_dec.wait_event(ev["out"][i])  # step k - 2's output was read back
            if args.fused:
                mla.decode_fused(q, r, batch.kv, batch.kv_scale, r2t, sl, kv_limit,
                                 S, wl.sm_scale, wl.num_shards, O_part, LSE_part,
                                 counters, d_out[i], d_lse[i], status,
                                 split_pages=sp, work=wk)
            else:
                mla.decode_partial(q, r, batch.kv, batch.kv_scale, r2t, sl,
                                   kv_limit, S, wl.sm_scale, wl.num_shards, O_part,
                                   LSE_part, status, split_pages=sp, work=wk)
                mla.lse_combine(O_part, LSE_part, d_out[i], d_lse[i])
            ev["dec"][i].record(s_dec)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev["dec"][i])
            h_out[i].copy_(d_out[i], non_blocking=True)
            h_lse[i].copy_(d_lse[i], non_blocking=True)
            ev["out"][i].record(s_out)

    for k in range(3):
        e2e_step(k)
    torch.cuda.synchronize()
    n_e2e = max(10, args.steps // 2)
    t0 = time.perf_counter()
    for k in range(n_e2e):
        e2e_step(k)
    torch.cuda.synchronize()
    e2e_s = slowest_rank(time.perf_counter() - t0, dist, dev)
    # The same steps one at a time (each waited for before the next is
    # planned): the latency of one step, and what the overlap hides.
    t0 = time.perf_counter()
    for k in range(n_e2e):
        e2e_step(k)
        torch.cuda.synchronize()
    serial_s = slowest_rank(time.perf_counter() - t0, dist, dev)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in the e2e loop")
    return {"value": job_tflops(fl, n_e2e, world, e2e_s), "unit": "TFLOP/s",
            "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "steps": n_e2e,
            "plan": "fixed" if fixed else "per step on the host",
            "overlap": "uploads, decode and downloads of consecutive steps on "
                       "three streams, two buffer sets",
            "ms_per_step": e2e_s * 1e3 / n_e2e,
            "serial": {"value": job_tflops(fl, n_e2e, world, serial_s),
                       "ms_per_step": serial_s * 1e3 / n_e2e}}


def main():
    args = parse()
    PARTS["dtype"] = args.parts
    if args.projections:
        return run_projections(args)
    if args.kv_write_rows > 0:
        return run_kv_write(args)
    if args.impl == "reference":
        return run_reference(args)
    if args.sweep:
        return run_sweep(args)
    if args.c0_scan:
        return run_c0_scan(args)
    rank, world, local = dist_env()
    import torch

    import mla_latent_decode_gb300 as mla
    from mla_latent_decode_gb300 import synth

    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    mla.library()  # fail loudly if the CUDA library is missing

    wl = synth.config(args.config)
    batch = synth.make_batch(wl, seed=rank, device="cuda")
    lens = mla.batch_lengths(batch)
    slots = mla.cluster_slots()
    dev = torch.device("cuda", local)
    split_pages, work, plan_desc = None, None, "uniform deal"
    if args.parts_cut > 0:
        import numpy as np
        P = [-(-L // 64) for L in lens]
        bnd = np.array([[0, min(p, args.parts_cut), p] for p in P], dtype=np.int32)
        S, eff = 2, None
        split_pages = torch.from_numpy(bnd).to(dev)
        plan_desc = f"two parts per request, first {args.parts_cut} pages (fixed)"
    elif args.splits > 0:
        S, eff = args.splits, None
    elif wl.num_splits:
        S, eff = wl.num_splits, None
    elif args.planner == "parts":
        # the per-request split planner, part-major launch order (the plan is
        # computed per batch before timing, like the split count)
        S, bnd, eff = mla.plan_parts(wl.B, wl.q_len, wl.H, lens, wl.num_shards,
                                     kv_dtype=wl.kv_dtype)
        split_pages = torch.from_numpy(bnd).to(dev)
        plan_desc = (f"per-request parts (part-major order), first-part "
                     f"boundaries {sorted({r[1] for r in bnd.tolist()})[:4]}"
                     if S > 1 else "one part")
    else:
        # the work-balanced scheduler: per-request parts and the longest-first
        # launch order of the work units (computed per batch before timing)
        S, bnd, wk, eff = mla.plan_sched(wl.B, wl.q_len, wl.H, lens, wl.num_shards,
                                         kv_dtype=wl.kv_dtype)
        split_pages = torch.from_numpy(bnd).to(dev)
        work = torch.from_numpy(wk).to(dev)
        longest = max(bnd.tolist(), key=lambda r: r[-1])
        sizes = [b1 - b0 for b0, b1 in zip(longest, longest[1:]) if b1 > b0]
        plan_desc = (f"scheduler: {S} parts per request at most (the longest "
                     f"request's parts: {sizes} pages), {len(wk)} work units "
                     f"launched longest first")
    S_pages = mla.plan_heuristic(wl.B, wl.q_len)

    status = torch.zeros(1, dtype=torch.int32, device=dev)
    # the fused launch keeps fp32 parts (its merge reads them in the launch)
    O_part = torch.empty((S, wl.num_shards, wl.B, wl.q_len, wl.H, 512),
                         dtype=torch.float32 if args.fused else part_dtype(wl),
                         device=dev)
    LSE_part = torch.empty((S, wl.num_shards, wl.B, wl.q_len, wl.H),
                           dtype=torch.float32, device=dev)
    out = torch.empty((wl.B, wl.q_len, wl.H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((wl.B, wl.q_len, wl.H), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    counters = mla.fused_counters(wl.B, wl.q_len, wl.H, dev)

    def step(ev=None, mid=True):
        if args.fused:
            if ev is not None:
                ev[0].record(stream)
            mla.decode_fused(batch.q_nope, batch.q_rope, batch.kv, batch.kv_scale,
                             batch.req_to_token, batch.seq_lens, batch.kv_limit,
                             S, wl.sm_scale, wl.num_shards, O_part, LSE_part,
                             counters, out, lse, status, split_pages=split_pages,
                             work=work)
            if ev is not None:
                ev[1].record(stream)
                ev[2].record(stream)
            return
        if ev is not None:
            ev[0].record(stream)
        mla.decode_partial(batch.q_nope, batch.q_rope, batch.kv, batch.kv_scale,
                           batch.req_to_token, batch.seq_lens, batch.kv_limit, S,
                           wl.sm_scale, wl.num_shards, O_part, LSE_part, status,
                           split_pages=split_pages, work=work)
        if ev is not None and mid:
            ev[1].record(stream)
        mla.lse_combine(O_part, LSE_part, out, lse)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} after warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)]
           for _ in range(args.steps)]
    # KV smaller than twice the L2 (129 MB on GB300): write a 256-MB buffer
    # between timed steps so every step reads its inputs from DRAM; the
    # value then comes from the per-step CUDA-event spans (flush excluded).
    kv_bytes = batch.kv.numel() * batch.kv.element_size()
    flush = kv_bytes < 256 * 2**20
    flush_buf = torch.empty(256 * 2**20, dtype=torch.uint8, device=dev) if flush else None
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.1)  # let the sampler take its first reading
    # The steps as a caller runs them: an event between the two launches
    # would stop the combine's programmatic overlap with the partial decode's
    # tail (~4 us per step), so these steps carry events around the step only.
    t_start.record(stream)
    for k in range(args.steps):
        if flush:
            flush_buf.fill_(k & 0xFF)
        step(evs[k], mid=False)
    t_end.record(stream)
    torch.cuda.synchronize()
    total_ms = t_start.elapsed_time(t_end)
    if flush:  # time the steps only, not the flushes between them
        total_ms = sum(e[0].elapsed_time(e[2]) for e in evs)
    # The same K steps again with an event between the launches: the partial
    # decode's own duration (the roofline's) and the combine's.
    evk = [[torch.cuda.Event(enable_timing=True) for _ in range(3)]
           for _ in range(args.steps)]
    for k in range(args.steps):
        if flush:
            flush_buf.fill_(k & 0xFF)
        step(evk[k])
    torch.cuda.synchronize()
    clk = clocks.stop()
    if dist:
        dist.barrier()
    part_ms = [e[0].elapsed_time(e[1]) for e in evk]
    comb_ms = [e[1].elapsed_time(e[2]) for e in evk]
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in timed region")
    total_ms = slowest_rank(total_ms, dist, dev)
    fl = wl.flops()
    ms_per_step = total_ms / args.steps
    value = job_tflops(fl, args.steps, world, total_ms * 1e-3)
    peaks, peak_kind = measured_peaks()
    part_mean = statistics.mean(part_ms)
    achieved = fl / (part_mean * 1e-3) / 1e12
    fp8 = wl.kv_dtype != "bf16"
    # The FP8 kernel's contractions are kind::f8f6f4 MMAs: their dense peak is
    # the measured BF16 one times the nominal FP8/BF16 ratio (4.5 / 2.25).
    peak = float(peaks["bf16_tflops"]) * (2.0 if fp8 else 1.0)
    traffic = profiled_traffic(args.config, 1, fp8)

    # end to end through the public API from pinned host buffers
    e2e = None
    if not args.no_e2e:
        e2e = time_e2e(mla, args, wl, batch, lens, S, split_pages, work, counters,
                       status, dev, fl, world, dist)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        hb = synth.host_bits(batch)
        cpu = oracle_sample(batch, hb, args.cpu_seconds)
        cpu.pop("seconds", None)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": ("e4m3 (FP8 tensor-core MMAs on the stored KV bytes; bf16 Q and "
                      "the probabilities each split into two 8-bit parts)") if fp8 else "bf16",
            "data": "synthetic",
            "config": {
                "workload": workload_desc(wl), "B": wl.B, "q_len": wl.q_len,
                "H": wl.H, "context": wl.seq_lens[0] if len(set(wl.seq_lens)) == 1 else "ragged",
                "num_shards": wl.num_shards, "num_splits": S,
                "split_plan": plan_desc,
                "planner_wave_eff": eff, "pages_rule_splits": S_pages,
                "cluster_slots": slots,
                "l2": (f"KV {kv_bytes / 1e6:.1f} MB < 2 x L2: 256-MB L2 flush between timed steps, value from per-step event spans"
                       if flush else f"inputs larger than L2 ({kv_bytes / 1e9:.2f} GB KV), no flush"),
                "parallelism": f"dp{world} (independent requests per rank)",
                "timing": ("value from K steps with events around each step only; "
                           "partial_us, combine_us and the roofline from a second "
                           "pass of K steps with an event between the two launches"),
                "step": ("mla_decode: partial decode and LSE combine fused in one launch"
                         if args.fused else
                         "mla_decode_partial + mla_lse_combine (two launches)"
                         if part_dtype(wl) == torch.float32 else
                         "mla_decode_partial_bf16_parts + mla_lse_combine_bf16_parts "
                         "(two launches, bf16 partial outputs)"),
            },
            "us_per_layer": ms_per_step * 1e3,
            "partial_us": part_mean * 1e3,
            "combine_us": statistics.mean(comb_ms) * 1e3,
            "kv_gbs": sum(wl.seq_lens) * wl.kv_row_bytes() * world * args.steps
                      / (total_ms * 1e-3) / 1e9,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak,
                         "unit": "TFLOP/s", "frac": achieved / peak,
                         "traffic": traffic,
                         "kernel": ("mla_partial_tc_fp8_kernel" if fp8
                                    else "mla_partial_tc_kernel"),
                         "peak_kind": (f"{peak_kind} bf16 burst (cuBLAS) x 2, the "
                                       "nominal FP8/BF16 dense ratio" if fp8 else
                                       f"{peak_kind} bf16 burst (cuBLAS)"),
                         **({"mma_work_per_flop": 2,
                             "note": "two FP8 MMAs per product (hi/lo split): "
                                     "the tensor pipe executes 2x the algorithmic "
                                     "FLOPs, so this design's ceiling is frac 0.5"}
                            if fp8 else {})},
            "hbm_frac": (sum(wl.seq_lens) * wl.kv_row_bytes() / (part_mean * 1e-3)
                         / 1e9) / float(peaks["hbm_gbs"]),
            "clocks": clk,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "gpu_launches": (1 if args.fused else 2) * args.steps,
        }
        print(json.dumps(line))
    if dist:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
