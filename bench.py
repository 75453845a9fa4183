#!/usr/bin/env python3
"""Benchmark of exact attention (forward + backward) on GB300.

One step = one pass of the whole path over one batch: fa_fwd (O, LSE) then
fa_bwd (dQ, dK, dV) on the causal, key-padded workload
B=4, H=16, N=4096, d=128 with per-batch key lengths uniform in [1024, 4096]
(seeded synthetic bf16 inputs). Throughput is TFLOP/s with the
causal-adjusted count: 4*d FLOPs per visible (query, key) pair forward and
10*d backward (the five backward products, recompute included).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--shard heads] [--no-extras]

Prints one JSON line (rank 0). Beside the step it carries, unless
``--no-extras``, the forward alone on the other forward workloads (head dim
64/128, 2K-128K tokens, causal and not), the packed variable-length batch, the
deterministic backward, the FP8 forward and one paged decoding step, each with
its own roofline. ``--impl reference`` times the fp64 CPU oracle on the same
workload, one (batch, head) slice per host worker per step.

Multi-GPU: replicas by default (every rank its own seeded batch, weak
scaling); ``--shard heads`` splits one seeded batch's (batch, head) problems
into contiguous ranges, one per rank (strong scaling). Neither needs a
collective on the data path.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd/bwd TFLOP/s (bf16, causal-adjusted) and % of GB300 dense BF16 peak"
WORKLOAD = "fwd+bwd B4 H16 N4096 d128 causal, key padding kv_lens~U[1024,4096]"
# DRAM bytes (read + write) of one fa_bwd_kernel launch on the C4 step in an ncu
# capture of `bench.py --profile bwd --profile-workload C4` (the step's inputs
# and launch), or None until the current kernel has been captured.
BWD_NCU_DRAM_BYTES = 782162176 + 462234112

# DRAM bytes (read + write) of one fa_decode_kernel launch in an ncu capture
# of the smaller decoding step (synth.D_SMALL, `bench.py --profile decode`),
# and that launch's algorithmic bytes. Traffic grows with the cached bytes, so
# the full workload's traffic is scaled from it. Valid for the current kernel.
DECODE_NCU_DRAM_BYTES = 351337216 + 3775744
DECODE_NCU_ALGO_BYTES = 350388836

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=100)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="bound on the oracle sample")
    ap.add_argument("--profile", choices=["decode", "fp8", "fwd", "bwd", "bwd_det", "varlen"], default=None,
                    help="run only a small case of one kernel a few times (for profiler captures); prints one "
                         "line with its mean time")
    ap.add_argument("--profile-workload", default="C4",
                    help="fwd / bwd profile case: a workload key (C2, C2C, C3, C4, C5, L1, NC), optionally with "
                         "its batch cut, e.g. C2:1 for one batch entry")
    ap.add_argument("--profile-reps", type=int, default=3)
    ap.add_argument("--no-extras", action="store_true",
                    help="time the step only (skip the forward workloads, packed batch, deterministic backward, "
                         "FP8 forward and decoding step)")
    ap.add_argument("--shard", choices=["none", "heads"], default="none",
                    help="heads: ranks split one batch's (b, h) problems (strong scaling) instead of running "
                         "replicas")
    ap.add_argument("--cpu-workers", type=int, default=0, help="host processes for the oracle (0 = all cores)")
    return ap.parse_args()


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def flops_per_step(w):
    vis = w.visible_pairs()
    return 4 * w.d * vis, 10 * w.d * vis, vis


# ---------------------------------------------------------------------------
# CPU oracle timing (reference arm and cpu_baseline)
# ---------------------------------------------------------------------------
def slice_inputs(w, b, h):
    """fp64 values of the (b, h) slice of Q, K, V, dO (untimed)."""
    from exact_io_aware_29_gb300 import synth
    return [synth.bf16_bits_to_f64(w.slice_bits(st, b, h))
            for st in (synth.STREAM_Q, synth.STREAM_K, synth.STREAM_V, synth.STREAM_DO)]


def oracle_slice_pass(w, b, inputs):
    """fp64 oracle forward + backward on one (b, h) slice; returns its FLOP count
    (same causal-adjusted count as the GPU arm: 14*d per visible pair)."""
    import oracle
    q, k, v, do = inputs
    lens = w.kv_lens()
    L = None if lens is None else int(lens[b])
    oracle.attention_forward(q, k, v, w.scale, w.causal, L)
    oracle.attention_backward(q, k, v, do, w.scale, w.causal, L)
    if L is None:
        L = w.N
    vis = L * (L + 1) // 2 + (w.N - L) * L if w.causal else w.N * L
    return 14 * w.d * vis


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _oracle_worker(job):
    """One host process of the oracle timing: oracle forward + backward on the
    workload's (b, h) slices i = wid, wid + n, ... until ``seconds`` of oracle
    time or ``max_slices`` slices. Input generation is not timed."""
    wid, nworkers, seconds, max_slices = job
    from exact_io_aware_29_gb300 import synth
    w = synth.C4
    pairs = [(b, h) for b in range(w.B) for h in range(w.H)]
    flops, busy, done, i = 0, 0.0, 0, wid
    while done < max_slices:
        b, h = pairs[i % len(pairs)]
        inputs = slice_inputs(w, b, h)
        t0 = time.perf_counter()
        flops += oracle_slice_pass(w, b, inputs)
        busy += time.perf_counter() - t0
        done += 1
        i += nworkers
        if busy >= seconds:
            break
    return flops, busy, done


class OraclePool:
    """Spawned host processes (one per core, single-threaded BLAS each) that
    run the oracle on (b, h) slices in parallel. Spawned, not forked, so that
    no child inherits a CUDA context."""

    def __init__(self, workers=0):
        import multiprocessing as mp
        self.n = workers if workers > 0 else host_cores()
        saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
        for k in saved:
            os.environ[k] = "1"
        try:
            self.pool = mp.get_context("spawn").Pool(self.n)
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v

    def run(self, seconds, max_slices=1 << 30):
        """Every worker runs slices for about ``seconds``; returns (total FLOPs,
        seconds of the busiest worker, slices done)."""
        res = self.pool.map(_oracle_worker, [(i, self.n, seconds, max_slices) for i in range(self.n)])
        return sum(r[0] for r in res), max(r[1] for r in res), sum(r[2] for r in res)

    def close(self):
        self.pool.close()
        self.pool.join()


def reference_arm(args, info):
    if not info.is_root:
        return
    pool = OraclePool(args.cpu_workers)
    try:
        for _ in range(args.warmup):
            pool.run(0.0, 1)
        flops, elapsed = 0, 0.0
        for _ in range(args.steps):
            f, busy, _ = pool.run(0.0, 1)  # one slice per worker, in parallel
            flops += f
            elapsed += busy
    finally:
        pool.close()
    value = flops / elapsed / 1e12
    sample = (f"{pool.n} (b,h) slices per step, one per host process (single-threaded BLAS): fp64 oracle forward "
              f"+ backward, N=4096 d=128, {args.steps} steps; step time = the slowest process")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * elapsed / max(args.steps, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded SplitMix64 / Box-Muller, bf16-rounded)",
        "config": {"workload": WORKLOAD, "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": pool.n, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# Clock sampling during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu):
        self.gpu = gpu
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [v for v in (num(r[1]) for r in rows) if v is not None]
        mx = [v for v in (num(r[2]) for r in rows) if v is not None]
        pw = [v for v in (num(r[3]) for r in rows) if v is not None]
        reasons = sorted({n for r in rows for n, v in zip(self.NAMES, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(pw) if pw else None}


# ---------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------
def group_visible_pairs(w, b0, b1, h0, h1):
    """Exact visible (query, key) pairs of batch entries b0..b1-1, heads h0..h1-1."""
    lens = w.kv_lens()
    total = 0
    for b in range(b0, b1):
        L = w.N if lens is None else int(min(lens[b], w.N))
        total += L * (L + 1) // 2 + (w.N - L) * L if w.causal else w.N * L
    return total * (h1 - h0)


def ours_arm(args, info):
    import numpy as np
    import torch
    from exact_io_aware_29_gb300 import binding, build, multi, synth

    # The host oracle processes start before the first CUDA call (spawned).
    want_cpu = info.is_root and info.world_size == 1 and not args.no_cpu_baseline
    cpu_pool = OraclePool(args.cpu_workers) if want_cpu else None

    build.build()
    binding.load_library()
    torch.cuda.set_device(info.local_rank)
    dev = torch.device("cuda", info.local_rank)
    w0 = synth.C4
    sharded = args.shard == "heads"
    seed = w0.seed if sharded else multi.rank_seed(w0.seed, info.rank)
    w = synth.Workload(w0.name, w0.B, w0.H, w0.N, w0.d, w0.causal, seed,
                       q_sigma=w0.q_sigma, kv_len_range=w0.kv_len_range, backward=True)
    # The (b, h) problems of this rank, as calls over contiguous heads.
    items = multi.shard(w.B * w.H, info.rank, info.world_size) if sharded else range(w.B * w.H)
    groups = multi.head_groups(items, w.H)
    vis = sum(group_visible_pairs(w, *g) for g in groups)
    fwd_flops, bwd_flops = 4 * w.d * vis, 10 * w.d * vis
    step_flops = fwd_flops + bwd_flops

    def host(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).pin_memory()

    full = {"q": w.q(), "k": w.k(), "v": w.v(), "do": w.do()}
    lens_all = w.kv_lens().astype(np.int32)
    G = []  # per call: pinned host inputs, device buffers
    for (b0, b1, h0, h1) in groups:
        g = {"h": {n: host(x[b0:b1, h0:h1]) for n, x in full.items()}}
        g["h"]["kv"] = torch.from_numpy(lens_all[b0:b1].copy()).pin_memory()
        d = {n: t.to(dev) for n, t in g["h"].items()}
        d["o"] = torch.empty_like(d["q"])
        d["lse"] = torch.empty(d["q"].shape[:3], dtype=torch.float32, device=dev)
        d["dq"], d["dk"], d["dv"] = (torch.empty_like(d["q"]) for _ in range(3))
        Bg, Hg = b1 - b0, h1 - h0
        d["ws"] = torch.empty(binding.fa_bwd_workspace_size(Bg, Hg, w.N, w.d), dtype=torch.uint8, device=dev)
        g["d"] = d
        G.append(g)
    del full
    stream = torch.cuda.current_stream(dev)

    def run(d, st):
        binding.fa_fwd(d["q"], d["k"], d["v"], d["o"], d["lse"], w.scale, True, d["kv"], st)
        binding.fa_bwd(d["q"], d["k"], d["v"], d["o"], d["lse"], d["do"], d["dq"], d["dk"], d["dv"], w.scale, True,
                       d["kv"], d["ws"], st)

    def step():
        for g in G:
            run(g["d"], stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    if binding.fa_check_status(stream) != binding.FA_OK:
        raise RuntimeError("device status error during warm-up")

    # ---- device-timed region: inputs resident in HBM. No per-kernel events
    # here: the backward's kernels are launched programmatically, each
    # starting while the one before it drains, which events between them
    # would prevent.
    visible = [x.strip() for x in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if x.strip()]
    sampler = ClockSampler(visible[info.local_rank] if info.local_rank < len(visible) else info.local_rank)
    sampler.start()
    multi.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    multi.barrier()
    clocks = sampler.stop()
    ms_total = e0.elapsed_time(e1)
    if binding.fa_check_status(stream) != binding.FA_OK:
        raise RuntimeError("device status error in the timed region")
    value, slowest_s = multi.aggregate_throughput(step_flops * args.steps / 1e12, ms_total / 1e3)

    # ---- per-kernel times: the same steps again with an event pair around
    # every kernel (plain launches), for the breakdown and the roofline.
    kt_steps = max(1, min(args.steps, 200))
    binding.fa_timing_begin(kt_steps * max(len(G), 1))
    for _ in range(kt_steps):
        step()
    torch.cuda.synchronize()
    kt = {kind: binding.fa_timing_read(kind) for kind in range(4)}
    binding.fa_timing_end()

    # ---- end to end through the public API: pinned host in, host out. Steps
    # run on three streams (host->device copies, compute, device->host copies)
    # over two sets of device buffers, so step k's results travel back while
    # step k+1's inputs arrive; every step copies its own inputs in and its own
    # results out inside the timed region.
    e2e_steps = max(1, min(args.e2e_steps, args.steps))
    for g in G:
        h, d = g["h"], g["d"]
        for n in ("o", "dq", "dk", "dv"):
            h[n] = torch.empty_like(h["q"]).pin_memory()
        h["lse"] = torch.empty(d["lse"].shape, dtype=torch.float32).pin_memory()
        g["sets"] = [d, {n: torch.empty_like(t) for n, t in d.items()}]
    s_in, s_run, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_run = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_step(i):
        x = i % 2
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_run[x])  # step i-2 has finished reading this set's inputs
            for g in G:
                for n in ("q", "k", "v", "do", "kv"):
                    g["sets"][x][n].copy_(g["h"][n], non_blocking=True)
            ev_in[x].record(s_in)
        with torch.cuda.stream(s_run):
            s_run.wait_event(ev_in[x])
            if i >= 2:
                s_run.wait_event(ev_out[x])  # step i-2's results are back on the host
            for g in G:
                run(g["sets"][x], s_run)
            ev_run[x].record(s_run)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_run[x])
            for g in G:
                for n in ("o", "lse", "dq", "dk", "dv"):
                    g["h"][n].copy_(g["sets"][x][n], non_blocking=True)
            ev_out[x].record(s_out)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    multi.barrier()
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(s_in)
    s_run.wait_event(a0)
    s_out.wait_event(a0)
    for i in range(e2e_steps):
        e2e_step(i)
    s_out.wait_event(ev_run[(e2e_steps - 1) % 2])
    a1.record(s_out)
    torch.cuda.synchronize()
    multi.barrier()
    if binding.fa_check_status() != binding.FA_OK:
        raise RuntimeError("device status error in the end-to-end steps")
    e2e_value, _ = multi.aggregate_throughput(step_flops * e2e_steps / 1e12, a0.elapsed_time(a1) / 1e3)
    h2d = sum(t.numel() * t.element_size() for g in G for n, t in g["h"].items() if n in ("q", "k", "v", "do", "kv"))
    d2h = sum(t.numel() * t.element_size() for g in G for n, t in g["h"].items()
              if n in ("o", "lse", "dq", "dk", "dv"))

    # ---- roofline of the dominant kernel (largest share of device time). Its
    # launches are event-timed inside a short region (well under a second at
    # the default step count), so the burst peak is the denominator; the
    # fraction of the sustained (power-capped) peak is given beside it.
    peaks, peak_src = load_peaks()
    names = {0: "fa_fwd_kernel", 1: "fa_bwd_pre_kernel", 2: "fa_bwd_kernel", 3: "fa_bwd_dq_kernel"}
    kflops = {0: fwd_flops, 2: bwd_flops}
    dom = max(kt, key=lambda kd: kt[kd][0])
    sustained = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    burst = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    # per step: the kernel's FLOPs over its summed launch time in one step
    achieved = kflops.get(dom, 0) * kt_steps / (kt[dom][0] / 1e3) / 1e12
    fwd_ms = kt[0][0] / kt_steps
    bwd_ms = sum(kt[i][0] for i in (1, 2, 3)) / kt_steps

    def tf(fl, ms):
        return fl / (ms / 1e3) / 1e12

    line = {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": info.world_size,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": 1e3 * slowest_s / args.steps,
        "higher_is_better": True,
        "scaling": "strong" if sharded and info.world_size > 1 else "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded SplitMix64 / Box-Muller, bf16-rounded), "
                + ("one batch shared by all ranks" if sharded else "per-rank seed"),
        "config": {"workload": WORKLOAD, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": True,
                   "kv_lens": [int(x) for x in w.kv_lens()], "visible_pairs": vis,
                   "flops_fwd": fwd_flops, "flops_bwd": bwd_flops,
                   "flops_fwd_nominal": 4 * w.B * w.H * w.N * w.N * w.d // 2,
                   "flops_note": "headline counts exact visible (query, key) pairs (key lengths included); the "
                                 "nominal count is 4 B H N^2 d / 2 for causal, ignoring key lengths",
                   "l2": "not flushed: the per-step working set (Q,K,V,O,dO,dQ,dK,dV bf16 and the fp32 dQ "
                         "accumulator, 0.73 GB) is larger than the 129 MB L2",
                   "parallelism": (f"head shards x{info.world_size}: rank r runs (b,h) problems "
                                   f"shard(B*H, r, N) of one batch, no collective" if sharded else
                                   f"replicas x{info.world_size} (independent (b,h) problems, no collective)"),
                   "calls_per_step": len(G)},
        "pct_of_peak": {"step": 100 * value / info.world_size / burst,
                        "denominator": f"bf16_tflops burst {burst} ({peak_src})"},
        "breakdown": {
            "fwd_ms": fwd_ms, "fwd_tflops": tf(fwd_flops, fwd_ms),
            "fwd_pct_peak_burst": 100 * tf(fwd_flops, fwd_ms) / burst,
            "bwd_ms": bwd_ms, "bwd_tflops": tf(bwd_flops, bwd_ms),
            "bwd_pct_peak_burst": 100 * tf(bwd_flops, bwd_ms) / burst,
            "fwd_exps_per_s": vis / (fwd_ms / 1e3), "bwd_exps_per_s": vis / (bwd_ms / 1e3),
            "bwd_main_ms": kt[2][0] / kt_steps, "bwd_pre_ms": kt[1][0] / kt_steps,
            "bwd_dq_ms": kt[3][0] / kt_steps,
            "kernel_times": f"CUDA event pairs around each kernel over {kt_steps} further steps with plain "
                            "launches; the timed steps launch the backward's kernels programmatically, so the "
                            "step can be shorter than the sum",
        },
        "roofline": {"kernel": names[dom], "bound": "tensor", "achieved": achieved, "peak": burst,
                     "unit": "TFLOP/s", "frac": achieved / burst,
                     "traffic": BWD_NCU_DRAM_BYTES if names[dom] == "fa_bwd_kernel" else None,
                     "peak_source": f"bf16_tflops burst ({peak_src}): kernel event-timed in a short region",
                     "frac_of_sustained": achieved / sustained},
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps,
                "how": "pinned host buffers; host->device, compute and device->host on three streams over two "
                       "device buffer sets (step k's results return while step k+1's inputs arrive)"},
        "gpu_launches": 4 * args.steps * len(G),
        "clocks": clocks,
    }
    if not args.no_extras and info.is_root:
        line["forward_workloads"] = forward_sweep(dev, burst, sustained, peak_src)
        line["varlen"] = varlen_measure(dev, burst, sustained, peak_src)
        line["deterministic"] = deterministic_measure(G[0]["d"], w, groups[0], burst, sustained, peak_src)
        line["fp8_forward"] = fp8_measure(dev, burst, peak_src)
        line["decode"] = decode_measure(dev, peaks, peak_src)
    if cpu_pool is not None:
        try:
            cpu_pool.run(0.0, 1)
            flops, el, n = cpu_pool.run(args.cpu_seconds)
        finally:
            cpu_pool.close()
        line["cpu_baseline"] = {"value": flops / el / 1e12, "unit": "TFLOP/s", "cores": cpu_pool.n,
                                "kind": "oracle",
                                "sample": f"{n} (b,h) slices of the workload, fp64 oracle forward + backward, on "
                                          f"{cpu_pool.n} host processes (single-threaded BLAS) for {el:.1f} s"}
    if info.is_root:
        print(json.dumps(line), flush=True)


def tensor_roofline(kernel, tflops, burst, sustained, peak_src, note=None):
    r = {"kernel": kernel, "bound": "tensor", "achieved": tflops, "peak": burst, "unit": "TFLOP/s",
         "frac": tflops / burst, "traffic": None,
         "peak_source": f"bf16_tflops burst ({peak_src}): kernel event-timed in a short region",
         "frac_of_sustained": tflops / sustained}
    if note:
        r["note"] = note
    return r


def forward_sweep(dev, burst, sustained, peak_src, reps=20):
    """Forward-only TFLOP/s on the other forward workloads (device-resident
    random bf16 inputs of each workload's shape and Q spread), from the
    library's event pair around every fa_fwd_kernel launch."""
    import torch
    from exact_io_aware_29_gb300 import binding, synth
    out = {}
    g = torch.Generator(device=dev)
    for key in synth.FORWARD_SWEEP:
        w = synth.WORKLOADS[key]
        g.manual_seed(w.seed)
        shape = (w.B, w.H, w.N, w.d)
        q = (torch.randn(shape, device=dev, generator=g) * w.q_sigma).to(torch.bfloat16)
        k = torch.randn(shape, device=dev, generator=g).to(torch.bfloat16)
        v = torch.randn(shape, device=dev, generator=g).to(torch.bfloat16)
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
        for _ in range(3):
            binding.fa_fwd(q, k, v, o, lse, w.scale, w.causal)
        torch.cuda.synchronize()
        binding.fa_timing_begin(reps)
        for _ in range(reps):
            binding.fa_fwd(q, k, v, o, lse, w.scale, w.causal)
        torch.cuda.synchronize()
        tot, n = binding.fa_timing_read(binding.KERNEL_FWD)
        binding.fa_timing_end()
        ms = tot / max(n, 1)
        tflops = 4 * w.d * w.visible_pairs() / (ms / 1e3) / 1e12
        out[key] = {"workload": w.name, "ms": ms, "tflops": tflops, "pct_of_burst_peak": 100 * tflops / burst,
                    "exps_per_s": w.visible_pairs() / (ms / 1e3),
                    "roofline": tensor_roofline("fa_fwd_kernel", tflops, burst, sustained, peak_src)}
        del q, k, v, o, lse
    if binding.fa_check_status() != binding.FA_OK:
        raise RuntimeError("device status error in the forward workloads")
    return out


def fp8_measure(dev, burst, peak_src, reps=20):
    """FP8 forward TFLOP/s (4 d flops per visible pair, same count as bf16) on
    device-resident random inputs of each workload's shape and Q spread,
    quantised once by the library's block quantiser (timed on its own).
    Denominator: the measured bf16 burst peak x 2, the nominal fp8:bf16 ratio
    of the tensor cores."""
    import torch
    from exact_io_aware_29_gb300 import binding, synth
    peak = 2 * burst
    out = {"peak_tflops": peak, "peak_source": f"2 x bf16_tflops burst ({peak_src}), nominal fp8:bf16 ratio"}
    g = torch.Generator(device=dev)
    for key in ("C3", "C5", "C4"):
        w = synth.WORKLOADS[key]
        g.manual_seed(w.seed)
        shape = (w.B, w.H, w.N, w.d)
        q = (torch.randn(shape, device=dev, generator=g) * w.q_sigma).to(torch.bfloat16)
        k = torch.randn(shape, device=dev, generator=g).to(torch.bfloat16)
        v = torch.randn(shape, device=dev, generator=g).to(torch.bfloat16)
        kv = None if w.kv_len_range is None else torch.tensor(w.kv_lens(), dtype=torch.int32, device=dev)
        o = torch.empty_like(q)
        lse = torch.empty(shape[:3], dtype=torch.float32, device=dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        q8, sq = binding.quantize_fp8(q, False)
        k8, sk = binding.quantize_fp8(k, False)
        v8t, sv = binding.quantize_fp8(v, True)
        e1.record()
        torch.cuda.synchronize()
        quant_ms = e0.elapsed_time(e1)
        for _ in range(3):
            binding.fa_fwd_fp8(q8, k8, v8t, sq, sk, sv, o, lse, w.scale, w.causal, kv)
        torch.cuda.synchronize()
        binding.fa_timing_begin(reps)
        for _ in range(reps):
            binding.fa_fwd_fp8(q8, k8, v8t, sq, sk, sv, o, lse, w.scale, w.causal, kv)
        torch.cuda.synchronize()
        tot, n = binding.fa_timing_read(binding.KERNEL_FWD_FP8)
        binding.fa_timing_end()
        ms = tot / max(n, 1)
        tflops = 4 * w.d * w.visible_pairs() / (ms / 1e3) / 1e12
        out[w.name] = {"ms": ms, "tflops": tflops, "pct_of_fp8_peak": 100 * tflops / peak,
                       "pct_of_bf16_burst_peak": 100 * tflops / burst, "quantize_qkv_ms": quant_ms,
                       "roofline": {"kernel": "fa_fwd_fp8_kernel", "bound": "tensor", "achieved": tflops,
                                    "peak": peak, "unit": "TFLOP/s", "frac": tflops / peak, "traffic": None}}
        del q, k, v, o, lse, q8, k8, v8t
    if binding.fa_check_status() != binding.FA_OK:
        raise RuntimeError("device status error in the FP8 measurement")
    return out


def decode_measure(dev, peaks, peak_src, reps=50, workload=None):
    """One decoding step over the paged KV cache (16 sequences of 1K..32K
    cached tokens, pages of 512 scattered over the pool): seeded lengths and
    block table, device random bf16 values; kernel times from the library's
    event pairs. Roofline: HBM, algorithmic bytes = the cached K and V the step
    must read + q, O, LSE, lengths and the used block-table entries."""
    import torch
    from exact_io_aware_29_gb300 import binding, synth
    w = workload or synth.D1
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed)
    shape = (w.n_blocks, w.block_size, w.H, w.d)
    kp = torch.randn(shape, device=dev, generator=g).to(torch.bfloat16)
    vp = torch.randn(shape, device=dev, generator=g).to(torch.bfloat16)
    q = torch.randn((w.B, w.H, w.d), device=dev, generator=g).to(torch.bfloat16)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H), dtype=torch.float32, device=dev)
    table = torch.from_numpy(w.block_table()).to(dev)
    lens = torch.from_numpy(w.seq_lens()).to(dev)
    max_len = int(w.seq_lens().max())
    ws = torch.empty(max(binding.fa_decode_workspace_size(w.B, w.H, w.d, max_len), 1), dtype=torch.uint8,
                     device=dev)

    def step():
        binding.fa_decode_paged(q, kp, vp, o, lse, table, lens, max_len, w.scale, ws)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    binding.fa_timing_begin(reps)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        step()
    e1.record()
    torch.cuda.synchronize()
    kt = {kind: binding.fa_timing_read(kind) for kind in (binding.KERNEL_DECODE, binding.KERNEL_DECODE_MERGE)}
    binding.fa_timing_end()
    if binding.fa_check_status() != binding.FA_OK:
        raise RuntimeError("device status error in the decode measurement")
    main_ms = kt[binding.KERNEL_DECODE][0] / max(kt[binding.KERNEL_DECODE][1], 1)
    merge_ms = kt[binding.KERNEL_DECODE_MERGE][0] / max(kt[binding.KERNEL_DECODE_MERGE][1], 1)
    step_ms = e0.elapsed_time(e1) / reps
    algo = (w.cache_bytes() + 2 * q.numel() * 2 + lse.numel() * 4 + w.B * 4
            + int(w.pages().sum()) * 4)
    peak = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    gbs = algo / (main_ms / 1e3) / 1e9
    return {"workload": w.name, "cached_tokens": int(w.seq_lens().sum()), "bytes_per_step": algo,
            "ms_per_step": step_ms, "kernel_ms": main_ms, "merge_ms": merge_ms,
            "tokens_per_s": w.B / (step_ms / 1e3),
            "roofline": {"kernel": "fa_decode_kernel", "bound": "hbm", "achieved": gbs, "peak": peak,
                         "unit": "GB/s", "frac": gbs / peak,
                         "traffic": round(algo * DECODE_NCU_DRAM_BYTES / DECODE_NCU_ALGO_BYTES),
                         "traffic_source": "ncu dram bytes of the 0.35 GB profile case, scaled by algorithmic bytes",
                         "peak_source": f"hbm_gbs ({peak_src})"},
            "data": "seeded lengths and block table; device random bf16 values (torch.randn, seeded)",
            "l2": "not flushed: the 2.6 GB of cached K/V read per step is far larger than the 129 MB L2"}


def deterministic_measure(d, w, group, burst, sustained, peak_src, reps=50):
    """fa_bwd_deterministic on the step's inputs (the first call of a step):
    per-kernel event times, and whether two calls give bitwise identical
    gradients."""
    import torch
    from exact_io_aware_29_gb300 import binding
    bwd_flops = 10 * w.d * group_visible_pairs(w, *group)
    grads = [tuple(torch.empty_like(d["q"]) for _ in range(3)) for _ in range(2)]

    def bwd(g):
        binding.fa_bwd_deterministic(d["q"], d["k"], d["v"], d["o"], d["lse"], d["do"], *g, w.scale, True, d["kv"],
                                     d["ws"])

    binding.fa_fwd(d["q"], d["k"], d["v"], d["o"], d["lse"], w.scale, True, d["kv"])
    for _ in range(3):
        bwd(grads[0])
    torch.cuda.synchronize()
    binding.fa_timing_begin(reps)
    for _ in range(reps):
        bwd(grads[0])
    torch.cuda.synchronize()
    kt = {kind: binding.fa_timing_read(kind) for kind in (1, 2, 3)}
    binding.fa_timing_end()
    bwd(grads[1])
    torch.cuda.synchronize()
    if binding.fa_check_status() != binding.FA_OK:
        raise RuntimeError("device status error in the deterministic backward")
    same = all(torch.equal(a.view(torch.int16), b.view(torch.int16)) for a, b in zip(*grads))
    ms = sum(kt[i][0] for i in (1, 2, 3)) / max(kt[2][1], 1)
    tflops = bwd_flops / (ms / 1e3) / 1e12
    main_ms = kt[2][0] / max(kt[2][1], 1)
    main_tf = bwd_flops / (main_ms / 1e3) / 1e12
    return {"bwd_ms": ms, "bwd_main_ms": main_ms, "bwd_tflops": tflops,
            "bwd_pct_of_burst_peak": 100 * tflops / burst, "bitwise_repeatable": same,
            "roofline": tensor_roofline("fa_bwd_kernel (deterministic order)", main_tf, burst, sustained, peak_src)}


def varlen_measure(dev, burst, sustained, peak_src, reps=20):
    """Forward and backward TFLOP/s on the packed batch (16 sequences of
    512..8192 tokens): seeded lengths, device-resident random bf16 values,
    CUDA events around `reps` calls of each pass."""
    import torch
    from exact_io_aware_29_gb300 import binding, synth
    w = synth.V1
    cu = torch.from_numpy(w.cu_seqlens()).to(dev)
    L = int(w.lens().max())
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed)
    q, k, v, do = (torch.randn((w.total, w.H, w.d), device=dev, generator=g).to(torch.bfloat16) for _ in range(4))
    o = torch.empty_like(q)
    lse = torch.empty((w.H, w.total), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(binding.fa_bwd_workspace_size(w.n_seq, w.H, L, w.d), dtype=torch.uint8, device=dev)

    def fwd():
        binding.fa_fwd_varlen(q, k, v, o, lse, cu, cu, L, L, w.scale, w.causal)

    def bwd():
        binding.fa_bwd_varlen(q, k, v, o, lse, do, dq, dk, dv, cu, cu, L, L, w.scale, w.causal, ws)

    out = {"workload": w.name, "total_tokens": w.total, "lens": [int(x) for x in w.lens()],
           "visible_pairs": w.visible_pairs(),
           "data": "seeded lengths; device random bf16 values (torch.randn, seeded)"}
    for name, fn, per_pair in (("fwd", fwd, 4), ("bwd", bwd, 10)):
        for _ in range(3):
            fwd()
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        tflops = per_pair * w.d * w.visible_pairs() / (ms / 1e3) / 1e12
        out[f"{name}_ms"] = ms
        out[f"{name}_tflops"] = tflops
        out[f"{name}_pct_of_burst_peak"] = 100 * tflops / burst
        out[f"{name}_roofline"] = tensor_roofline(f"{name} pass, all kernels", tflops, burst, sustained, peak_src,
                                                  note="CUDA events around whole calls")
    if binding.fa_check_status() != binding.FA_OK:
        raise RuntimeError("device status error in the packed-batch measurement")
    return out


def profile_attention(args, info):
    """A few forward (or forward + backward) calls on one workload (device
    random inputs of its shape, key lengths and Q spread), for profiler
    captures; prints the mean event time of the profiled kernel."""
    import torch
    from exact_io_aware_29_gb300 import binding, build, synth
    build.build()
    binding.load_library()
    dev = torch.device("cuda", info.local_rank)
    key, _, cut = args.profile_workload.partition(":")
    w = synth.WORKLOADS[key]
    B = int(cut) if cut else w.B
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed)
    shape = (B, w.H, w.N, w.d)
    q = (torch.randn(shape, device=dev, generator=g) * w.q_sigma).to(torch.bfloat16)
    k, v, do = (torch.randn(shape, device=dev, generator=g).to(torch.bfloat16) for _ in range(3))
    kv = None if w.kv_len_range is None else torch.tensor(w.kv_lens()[:B], dtype=torch.int32, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty(shape[:3], dtype=torch.float32, device=dev)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    ws = torch.empty(binding.fa_bwd_workspace_size(B, w.H, w.N, w.d), dtype=torch.uint8, device=dev)
    binding.fa_timing_begin(args.profile_reps)
    for _ in range(args.profile_reps):
        binding.fa_fwd(q, k, v, o, lse, w.scale, w.causal, kv)
        if args.profile == "bwd":
            binding.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, w.scale, w.causal, kv, ws)
        elif args.profile == "bwd_det":
            binding.fa_bwd_deterministic(q, k, v, o, lse, do, dq, dk, dv, w.scale, w.causal, kv, ws)
    torch.cuda.synchronize()
    kind = binding.KERNEL_FWD if args.profile == "fwd" else binding.KERNEL_BWD_MAIN
    tot, n = binding.fa_timing_read(kind)
    binding.fa_timing_end()
    print(json.dumps({"profile": f"{args.profile} {w.name} B={B}", "kernel_ms": tot / max(n, 1),
                      "status": binding.fa_check_status()}), flush=True)


def profile_varlen(args, info):
    """A few forward + backward calls on the packed batch V1 (seeded lengths,
    device random values), for profiler captures."""
    import torch
    from exact_io_aware_29_gb300 import binding, build, synth
    build.build()
    binding.load_library()
    dev = torch.device("cuda", info.local_rank)
    w = synth.V1
    cu = torch.from_numpy(w.cu_seqlens()).to(dev)
    L = int(w.lens().max())
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed)
    q, k, v, do = (torch.randn((w.total, w.H, w.d), device=dev, generator=g).to(torch.bfloat16) for _ in range(4))
    o = torch.empty_like(q)
    lse = torch.empty((w.H, w.total), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(binding.fa_bwd_workspace_size(w.n_seq, w.H, L, w.d), dtype=torch.uint8, device=dev)
    binding.fa_timing_begin(args.profile_reps)
    for _ in range(args.profile_reps):
        binding.fa_fwd_varlen(q, k, v, o, lse, cu, cu, L, L, w.scale, w.causal)
        binding.fa_bwd_varlen(q, k, v, o, lse, do, dq, dk, dv, cu, cu, L, L, w.scale, w.causal, ws)
    torch.cuda.synchronize()
    f_ms = binding.fa_timing_read(binding.KERNEL_FWD)
    b_ms = binding.fa_timing_read(binding.KERNEL_BWD_MAIN)
    binding.fa_timing_end()
    print(json.dumps({"profile": "varlen " + w.name, "fwd_kernel_ms": f_ms[0] / max(f_ms[1], 1),
                      "bwd_kernel_ms": b_ms[0] / max(b_ms[1], 1), "status": binding.fa_check_status()}), flush=True)


def main():
    args = parse_args()
    from exact_io_aware_29_gb300 import multi
    info = multi.rank_info()
    if args.impl == "reference":
        if info.world_size > 1:
            multi.init("gloo")
        reference_arm(args, info)
        return
    import torch
    if info.world_size > 1:
        torch.cuda.set_device(info.local_rank)
        multi.init("nccl")
    if args.profile == "decode":
        from exact_io_aware_29_gb300 import binding, build, synth
        build.build()
        binding.load_library()
        peaks, src = load_peaks()
        r = decode_measure(torch.device("cuda", info.local_rank), peaks, src, reps=3, workload=synth.D_SMALL)
        print(json.dumps({"profile": r["workload"], "kernel_ms": r["kernel_ms"],
                          "bytes_per_step": r["bytes_per_step"]}), flush=True)
        return
    if args.profile == "fp8":
        from exact_io_aware_29_gb300 import binding, build, synth
        build.build()
        binding.load_library()
        dev = torch.device("cuda", info.local_rank)
        w = synth.C3
        g = torch.Generator(device=dev)
        g.manual_seed(w.seed)
        shape = (w.B, w.H, w.N, w.d)
        q = (torch.randn(shape, device=dev, generator=g) * w.q_sigma).to(torch.bfloat16)
        k = torch.randn(shape, device=dev, generator=g).to(torch.bfloat16)
        v = torch.randn(shape, device=dev, generator=g).to(torch.bfloat16)
        for _ in range(3):
            o, lse, _ = binding.attention_forward_fp8(q, k, v, w.scale, True)
        torch.cuda.synchronize()
        print(json.dumps({"profile": "fp8 forward " + w.name, "status": binding.fa_check_status()}), flush=True)
        return
    if args.profile in ("fwd", "bwd", "bwd_det"):
        profile_attention(args, info)
        return
    if args.profile == "varlen":
        profile_varlen(args, info)
        return
    ours_arm(args, info)
    if info.world_size > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
