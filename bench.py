"""Benchmark: causal prefill attention TFLOPS and ms/call on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one call of the attention kernel over one batch of the workload
(all of the hot path: TMA loads, both tcgen05 contractions, online softmax,
epilogue).  Inputs are seeded synthetic tensors shaped like the pages' 7B
prefill workloads, resident in HBM before the timed region; the step rotates
over enough input copies that the working set exceeds L2, so every step reads
Q/K/V from HBM.  Time is device time from CUDA events on the launching stream,
bracketed by a barrier and a synchronize, max over ranks; the timed steps run
as back-to-back bursts with an event between bursts, and ms/step is the median
burst (the spread over bursts is printed beside it).  The default workload is
the 8192-token GQA prefill (bf16, hd 128), the largest of the workloads.

Prints one JSON line.  Under torchrun each rank runs its own replica of the
workload on its own GPU (attention over independent (batch, head) problems
needs no exchange); rank 0 prints.  ``--impl reference`` times the f64 CPU
oracle on a bounded sample of the same workload instead.
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
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_BYTES = 129 * 1024 * 1024
REFERENCE_SECONDS = 90.0  # the whole reference arm (warmup + steps), whatever K and W
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
DEFAULT_WORKLOAD = "gqa_s8192_bf16"
BURSTS = 11  # the timed steps are split into this many bursts; ms/step is their median


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--op", choices=["attention", "kv_append"], default="attention",
                    help="attention (the default line) or the K/V-cache append of the workload's whole K/V")
    ap.add_argument("--page-size", type=int, default=0,
                    help="read K/V through a paged pool of this page size (a multiple of 128)")
    ap.add_argument("--path", choices=["auto", "oneshot", "split", "pair"], default="auto",
                    help="kernel: the library's advice for the shape (auto), one-shot, split-KV, or the "
                         "CTA-pair kernel (GQA groups of a multiple of 4, heads 72..128; measurement only)")
    return ap.parse_args(argv)


# ----------------------------------------------------------------- helpers

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value: float, device=None) -> float:
    """The largest `value` over all ranks (identity without a process group).
    Timing uses it so the whole job is as slow as its slowest rank."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_step_per_rank: int, world: int, ms_per_step: float) -> float:
    """Whole-job TFLOP/s: every rank runs its own replica of the workload (weak
    scaling), all ranks' flops over the slowest rank's step time."""
    return flops_per_step_per_rank * world / (ms_per_step * 1e-3) / 1e12


def oneshot_kernel_label(w):
    """The one-shot kernel a head width runs on (heads of 8..64, 72..128 and
    136..256 columns run on the 64-, 128- and 256-column kernels)."""
    if w.hd <= 64:
        return "fa_prefill64_kernel (one-shot, S and P apart in TMEM)"
    if w.hd <= 128:
        return "fa_prefill_kernel (one-shot)"
    return "fa_prefill256_kernel (one-shot)"


def split_kernel_label(fa, w):
    """Which kernels the split-KV path runs for the workload: one piece per CTA
    on the split-KV kernel, several segments per CTA on the persistent kernel;
    the merge kernel after either when pairs are split."""
    import torch
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    sc = fa.debug_schedule(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.causal, sms=sms)
    k = "fa_prefill_sk_kernel (split-KV, one piece per CTA)" if sc["one_segment"] else \
        "fa_prefill_pk_kernel (persistent, stream-K ranges)"
    return k + (" + fa_sk_merge_kernel" if sc["split_pairs"] else "")


CLOCK_WINDOW_S = 1.0  # the clock record covers at least this much load


def keep_loaded(step, first, t_start):
    """When the warm-up and timed steps together last less than the clock
    sampler's window, keep running the same steps (untimed, after the timed
    region) until they do, so that the clock record samples the GPU under this
    load; returns a description of the sampled window."""
    import torch
    i = first
    extra = 0
    while time.time() - t_start < CLOCK_WINDOW_S:
        for _ in range(16):
            step(i)
            i += 1
            extra += 1
        torch.cuda.synchronize()
    if extra == 0:
        return "warm-up and timed steps"
    return f"warm-up and timed steps, then {extra} more of the same steps after the timed region (untimed)"


def burst_spread(per_burst):
    """Median, 10th and 90th percentile (nearest rank) and extremes of the
    per-burst ms/step figures."""
    xs = sorted(per_burst)
    n = len(xs)

    def pct(p):
        return xs[min(n - 1, max(0, math.ceil(p / 100.0 * n) - 1))]
    return {"bursts": n, "median_ms": statistics.median(xs), "p10_ms": pct(10), "p90_ms": pct(90),
            "min_ms": xs[0], "max_ms": xs[-1]}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return pk, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "causal_prefill_flash_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the kernel source as it is now (else None)."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    ent = rec.get(workload)
    if not ent or ent.get("kernel_source_sha") != kernel_source_hash():
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while running."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"fa_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.5)  # let the sampler start before the load does
        self.window = None
        return self

    def mark(self, t0: float, t1: float):
        """Host wall-clock window [t0, t1] of the loaded region."""
        self.window = (t0, t1)

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.out.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        import datetime
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [x.strip() for x in line.split(",")]
                    if len(parts) >= 10:
                        try:
                            ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                        except ValueError:
                            ts = None
                        rows.append([ts] + parts[1:])
            os.remove(self.path)
        except OSError:
            pass
        if self.window is not None:
            inside = [r for r in rows if r[0] is not None and self.window[0] <= r[0] <= self.window[1]]
            if inside:
                rows = inside
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[2]) for r in rows if num(r[2]) is not None]
        mx = [num(r[3]) for r in rows if num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = []
        for i, n in enumerate(names):
            if any(r[6 + i].lower() == "active" for r in rows):
                reasons.append(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max((num(r[4]) or 0.0) for r in rows)}


# --------------------------------------------------------- oracle baseline

def oracle_sample(w, seconds: float, seed: int = 4321):
    """Time the f64 oracle on a bounded random sample of output rows of the
    workload; returns (TFLOP/s, cores, sample description, seconds)."""
    import numpy as np
    import torch

    import oracle
    from causal_prefill_flash_gb300 import workloads as W

    q, k, v = W.make_inputs(w)
    q64, k64, v64 = (t.double().numpy() for t in (q, k, v))
    cores = oracle.default_threads()
    off = w.Skv - w.Sq

    def flops_of(rows):
        tot = 0
        for (_, _, i) in rows:
            vis = min(w.Skv, off + int(i) + 1) if w.causal else w.Skv
            tot += 4 * w.hd * max(0, vis)
        return tot

    n = 64
    while True:
        rows = W.sample_rows(w, n, seed=seed).numpy()
        t0 = time.perf_counter()
        oracle.attention_rows(q64, k64, v64, rows, causal=w.causal, scale=w.scale, nthreads=cores)
        dt = time.perf_counter() - t0
        if dt >= seconds * 0.5 or n >= w.B * w.Hq * w.Sq:
            break
        n = min(w.B * w.Hq * w.Sq, max(n * 2, int(n * seconds / max(dt, 1e-3))))
    fl = flops_of(rows)
    desc = (f"{len(rows)} random output rows (b, head, query) of {w.name}, each over its full "
            f"{w.Skv}-key score row, f64, {cores} threads")
    return fl / dt / 1e12, cores, desc, dt


# ------------------------------------------------------------------- main

def run_reference(args):
    """The reference arm: the f64 oracle on the host cores, timed on a bounded
    random sample of output rows per step.  The whole warmup + steps run fits
    a fixed budget (REFERENCE_SECONDS) whatever K and W are: the oracle's row
    rate is measured once and each step gets the rows its share of the budget
    allows (at least one)."""
    import numpy as np

    import oracle
    from causal_prefill_flash_gb300 import workloads as W

    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    w = W.get(args.workload)
    q, k, v = W.make_inputs(w)
    q64, k64, v64 = (t.double().numpy() for t in (q, k, v))
    cores = oracle.default_threads()
    off = w.Skv - w.Sq
    total_steps = max(1, args.steps + args.warmup)

    def flops_of(rows):
        return sum(4 * w.hd * max(0, (min(w.Skv, off + int(i) + 1) if w.causal else w.Skv)) for (_, _, i) in rows)

    def run_rows(n, seed):
        rows = W.sample_rows(w, n, seed=seed).numpy()
        t0 = time.perf_counter()
        oracle.attention_rows(q64, k64, v64, rows, causal=w.causal, scale=w.scale, nthreads=cores)
        return flops_of(rows), time.perf_counter() - t0

    # calibrate: rows per second at the workload's row length
    fl, dt = run_rows(4 * cores, seed=7)
    rate = 4 * cores / max(dt, 1e-6)
    per_step = REFERENCE_SECONDS / total_steps
    n = max(1, int(rate * per_step))
    vals = []
    for i in range(total_steps):
        fl, dt = run_rows(n, seed=1000 + i)
        if i >= args.warmup:
            vals.append(fl / dt / 1e12)
    value = statistics.median(vals)
    ms = w.flops() / (value * 1e12) * 1e3
    desc = (f"{n} random output rows (b, head, query) of {w.name} per step, each over its full "
            f"{w.Skv}-key score row, f64, {cores} threads")
    line = {
        "impl": "reference",
        "metric": "causal prefill attention TFLOPS (ms/call, % of dense peak)",
        "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Sq": w.Sq, "Skv": w.Skv,
                   "hd": w.hd, "causal": w.causal, "input_dtype": w.dtype},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import torch

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import causal_prefill_flash_gb300 as fa
    from causal_prefill_flash_gb300 import workloads as W

    w = W.get(args.workload)
    q, k, v = W.make_inputs(w)
    io = w.io_bytes()
    ncopy = max(2, math.ceil(3 * L2_BYTES / io))
    copies = []
    for c in range(ncopy):
        copies.append((q.to(dev), k.to(dev), v.to(dev), torch.empty_like(q, device=dev)))
    stream = torch.cuda.current_stream(dev)
    split = (args.path == "split" or
             (args.path == "auto" and fa.split_kv_advised(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.causal, w.hd)))
    paged = args.page_size > 0
    pair = args.path == "pair"
    if pair:
        if paged or (w.Hq // w.Hkv) % 4 != 0 or not 64 < w.hd <= 128:
            raise SystemExit("--path pair: the CTA-pair kernel takes contiguous K/V, GQA groups of a multiple "
                             "of 4 query heads and heads 72..128 wide")
        fa.debug_force_path("pair")
    if paged:  # each copy's K/V scattered over a pool in shuffled page order
        page = args.page_size
        npg = (w.Skv + page - 1) // page
        g = torch.Generator(device="cpu")
        g.manual_seed(w.seed)
        pcopies = []
        for dq, dk, dv, do in copies:
            perm = torch.randperm(w.B * npg, generator=g).reshape(w.B, npg).to(torch.int32)
            kp = torch.zeros((w.B * npg, page, w.Hkv, w.hd), dtype=dk.dtype, device=dev)
            vp = torch.zeros_like(kp)
            for b in range(w.B):
                for p_ in range(npg):
                    r0, r1 = p_ * page, min(w.Skv, (p_ + 1) * page)
                    kp[int(perm[b, p_]), : r1 - r0] = dk[b, r0:r1]
                    vp[int(perm[b, p_]), : r1 - r0] = dv[b, r0:r1]
            pcopies.append((dq, kp, vp, perm.to(dev), do))
        bf = int(w.dtype == "bf16")
        pws = torch.zeros(fa.workspace_bytes(w.hd), dtype=torch.uint8, device=dev) if split else None

        def step(i):
            dq, kp, vp, tb, do = pcopies[i % ncopy]
            if split:
                st = fa.fa_prefill_paged_ws(dq, kp, vp, tb, do, w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.hd, page, npg,
                                            w.B * npg, int(w.causal), w.scale, bf, pws, pws.numel(), stream)
            else:
                st = fa.fa_prefill_paged(dq, kp, vp, tb, do, w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.hd, page, npg,
                                         w.B * npg, int(w.causal), w.scale, bf, stream)
            if st != 0:
                raise fa.FaError(st, "fa_prefill_paged")
    elif split:
        fn = fa.fa_prefill_ws_bf16 if w.dtype == "bf16" else fa.fa_prefill_ws
        ws = torch.empty(fa.workspace_bytes(w.hd), dtype=torch.uint8, device=dev)  # needs no initialisation
        extra = (ws, ws.numel())
    else:
        fn = fa.fa_prefill_bf16 if w.dtype == "bf16" else fa.fa_prefill
        extra = ()
    if not paged:
        def step(i):
            dq, dk, dv, do = copies[i % ncopy]
            st = fn(dq, dk, dv, do, w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.hd, int(w.causal), w.scale, *extra, stream)
            if st != 0:
                raise fa.FaError(st, fn.__name__)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    peaks, peak_src = load_peaks()
    with ClockSampler(local) as clocks:
        t_load0 = time.time()
        for i in range(args.warmup):
            step(i)
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        # the K timed steps in back-to-back bursts, one CUDA event between
        # bursts (an event between two launches ends their overlap, so there
        # is one per burst, not one per step)
        nb = max(1, min(BURSTS, args.steps))
        sizes = [args.steps // nb + (1 if b < args.steps % nb else 0) for b in range(nb)]
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(nb + 1)]
        ev[0].record(stream)
        i = 0
        for b in range(nb):
            for _ in range(sizes[b]):
                step(i)
                i += 1
            ev[b + 1].record(stream)
        torch.cuda.synchronize()
        load_window = keep_loaded(step, args.steps, t_load0)
        clocks.mark(t_load0, time.time())
        barrier()
        torch.cuda.synchronize()
    per_burst = [ev[b].elapsed_time(ev[b + 1]) / sizes[b] for b in range(nb)]
    ms_total = max_over_ranks(ev[0].elapsed_time(ev[nb]), dev)
    ms_step = max_over_ranks(statistics.median(per_burst), dev)
    spread = burst_spread(per_burst)
    flops = w.flops()
    value = job_throughput(flops, world, ms_step)
    watchdog = fa.debug_status()

    # end to end through the public API: pinned host inputs -> device -> kernel
    # -> host O, every step.  Three streams and two device buffer sets: step
    # i+1's host-to-device copies run under step i's kernel and step i-1's
    # device-to-host copy (opposite copy directions use separate engines).
    # Events order each buffer set's reuse: the copy-in of step i waits for
    # the kernel of step i-2 (done reading that set), the kernel of step i for
    # its own copy-in and for the copy-out of step i-2 (done reading its O).
    e2e = None
    if not args.no_e2e and not paged:  # the e2e leg times the contiguous public API only
        hq_, hk_, hv_ = q.pin_memory(), k.pin_memory(), v.pin_memory()
        hos = [torch.empty_like(q).pin_memory() for _ in range(2)]
        sets = [(torch.empty_like(q, device=dev), torch.empty_like(k, device=dev), torch.empty_like(v, device=dev),
                 torch.empty_like(q, device=dev)) for _ in range(2)]
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_used = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]

        def e2e_step(i):
            bi = i % 2
            dq, dk, dv, do = sets[bi]
            if i >= 2:
                s_in.wait_event(ev_used[bi])
            with torch.cuda.stream(s_in):
                dq.copy_(hq_, non_blocking=True)
                dk.copy_(hk_, non_blocking=True)
                dv.copy_(hv_, non_blocking=True)
            ev_in[bi].record(s_in)
            stream.wait_event(ev_in[bi])
            if i >= 2:
                stream.wait_event(ev_out[bi])
            fa.attention(dq, dk, dv, causal=w.causal, scale=w.scale, out=do, split=split, stream=stream)
            ev_used[bi].record(stream)
            s_out.wait_event(ev_used[bi])
            with torch.cuda.stream(s_out):
                hos[bi].copy_(do, non_blocking=True)
            ev_out[bi].record(s_out)

        def drain():
            stream.wait_event(ev_out[0])
            stream.wait_event(ev_out[1])

        for i in range(3):
            e2e_step(i)
        drain()
        torch.cuda.synchronize()
        barrier()
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record(s_in)
        for i in range(args.e2e_steps):
            e2e_step(i)
        drain()
        a1.record(stream)
        torch.cuda.synchronize()
        ms_e2e = max_over_ranks(a0.elapsed_time(a1) / args.e2e_steps, dev)
        e2e = {"value": job_throughput(flops, world, ms_e2e), "unit": "TFLOP/s",
               "ms_per_step": ms_e2e,
               "h2d_bytes_per_step": int((q.numel() + k.numel() + v.numel()) * q.element_size()),
               "d2h_bytes_per_step": int(q.numel() * q.element_size()),
               "pipeline": "copy-in, kernel and copy-out of consecutive steps on three streams, "
                           "two device buffer sets"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tf, cores, desc, _ = oracle_sample(w, args.cpu_seconds)
        cpu = {"value": tf, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc}

    if rank != 0:
        torch.distributed.destroy_process_group()
        return 0
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    peak_sus = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    achieved = flops / (ms_step * 1e-3) / 1e12
    traffic = recorded_traffic(w.name + (":split" if split else "") + (":paged" if paged else "") +
                               (":pair" if pair else ""))
    line = {
        "metric": "causal prefill attention TFLOPS (ms/call, % of dense peak)",
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic",
        "spread": dict(spread, ms_total=ms_total, note="ms/step of each burst of the timed steps; "
                       "value and ms_per_step use the median"),
        "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Sq": w.Sq, "Skv": w.Skv,
                   "hd": w.hd, "causal": w.causal, "scale": w.scale,
                   "flops_per_call": flops, "flop_convention": "4*hd*visible (query,key) pairs",
                   "l2": f"inputs rotated over {ncopy} resident copies ({ncopy * io / 1e6:.0f} MB > L2)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "kernel": split_kernel_label(fa, w) if split else
                   ("fa_prefill_pair_kernel (CTA pairs, paired MMAs M = 256)" if pair else oneshot_kernel_label(w)),
                   "kv_layout": f"paged, {args.page_size}-token pages in shuffled order" if paged
                   else "contiguous BSHD"},
        "pct_of_peak": 100.0 * achieved / peak,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak,
                     "peak_source": f"{peak_src} bf16 dense burst (f16 nominal rate = bf16)",
                     # the same kernel against the measured back-to-back (power-capped) GEMM
                     # rate, the fair denominator once a timed region runs for seconds
                     "peak_sustained": peak_sus, "frac_sustained": achieved / peak_sus,
                     "traffic": traffic,
                     "algorithmic_bytes": io,
                     "achieved_hbm_gbs": io / (ms_step * 1e-3) / 1e9},
        "clocks": dict(clocks.summary(), window=load_window),
        "e2e": e2e,
        "cpu_baseline": cpu,
        "gpu_launches": args.steps * (2 if split and "merge" in split_kernel_label(fa, w) else 1),
        # split-KV: the attention kernel, and the merge when pairs are split
        "watchdog_status": watchdog,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_append(args):
    """The K/V-cache append on one GPU: the workload's whole K and V (Skv tokens
    per sequence, f32) rounded into 16-bit caches at positions 0..Skv-1.  HBM
    bound: reports GB/s of algorithmic traffic (f32 read, 16-bit written,
    positions read) against the measured copy bandwidth."""
    import torch
    import causal_prefill_flash_gb300 as fa
    from causal_prefill_flash_gb300 import workloads as W

    rank, world, local = dist_env()
    if world > 1 and rank != 0:
        return 0
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = W.get(args.workload)
    B, T, Hkv, hd = w.B, w.Skv, w.Hkv, w.hd
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    k_new = torch.randn((B, T, Hkv, hd), generator=g, dtype=torch.float32)
    v_new = torch.randn((B, T, Hkv, hd), generator=g, dtype=torch.float32)
    pos = torch.arange(T, dtype=torch.int32).repeat(B, 1).contiguous()
    dt = w.torch_dtype
    n = B * T * Hkv * hd
    step_bytes = 2 * n * 4 + 2 * n * 2 + B * T * 4
    ncopy = max(2, math.ceil(3 * L2_BYTES / step_bytes))
    copies = [(k_new.to(dev), v_new.to(dev), pos.to(dev), torch.empty((B, T, Hkv, hd), dtype=dt, device=dev),
               torch.empty((B, T, Hkv, hd), dtype=dt, device=dev)) for _ in range(ncopy)]
    stream = torch.cuda.current_stream(dev)

    # arguments marshalled once: a call costs the C entry point, not Python
    lib = fa.load()
    sp = int(stream.cuda_stream)
    bf = int(dt == torch.bfloat16)
    argv = [tuple(t.data_ptr() for t in c) + (B, T, Hkv, hd, T, bf, sp) for c in copies]

    def step(i):
        st = lib.fa_kv_append(*argv[i % ncopy])
        if st != 0:
            raise fa.FaError(st, "fa_kv_append")

    peaks, peak_src = load_peaks()
    with ClockSampler(local) as clocks:
        t0 = time.time()
        for i in range(args.warmup):
            step(i)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(args.steps):
            step(i)
        e1.record(stream)
        torch.cuda.synchronize()
        load_window = keep_loaded(step, args.steps, t0)
        clocks.mark(t0, time.time())
    ms = e0.elapsed_time(e1) / args.steps
    gbs = step_bytes / (ms * 1e-3) / 1e9
    peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    line = {
        "metric": "K/V-cache append GB/s", "value": gbs, "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32->" + w.dtype, "data": "synthetic",
        "config": {"workload": w.name + " K/V append", "B": B, "T": T, "Hkv": Hkv, "hd": hd,
                   "bytes_per_step": step_bytes,
                   "l2": f"inputs rotated over {ncopy} copies ({ncopy * step_bytes / 1e6:.0f} MB > L2)"},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                     "peak_source": f"{peak_src} copy bandwidth",
                     "traffic": recorded_traffic(w.name + ":append")},
        "clocks": dict(clocks.summary(), window=load_window), "gpu_launches": args.steps,
        "watchdog_status": fa.debug_status(),
    }
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    if args.op == "kv_append":
        return run_append(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
