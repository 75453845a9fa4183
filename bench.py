#!/usr/bin/env python3
"""Benchmark of exact attention (forward + backward) on GB300.

One step = one pass of the whole path over one batch: fa_fwd (O, LSE) then
fa_bwd (dQ, dK, dV) on the causal, key-padded workload
B=4, H=16, N=4096, d=128 with per-batch key lengths uniform in [1024, 4096]
(seeded synthetic bf16 inputs). Throughput is TFLOP/s with the
causal-adjusted count: 4*d FLOPs per visible (query, key) pair forward and
10*d backward (the five backward products, recompute included).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0). ``--impl reference`` times the fp64 CPU oracle
on the same workload, one (batch, head) slice per step.
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
# capture of `bench.py --steps 3 --warmup 3 --no-cpu-baseline --e2e-steps 1`,
# or None until the current kernel has been captured.
BWD_NCU_DRAM_BYTES = 801877504 + 477092352

# DRAM bytes (read + write) of one fa_decode_kernel launch in an ncu capture
# of the smaller decoding step (synth.D_SMALL, `bench.py --profile decode`),
# and that launch's algorithmic bytes. Traffic grows with the cached bytes, so
# the full workload's traffic is scaled from it. Valid for the current kernel.
DECODE_NCU_DRAM_BYTES = 351338240 + 3934208
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
    ap.add_argument("--profile", choices=["decode", "fp8"], default=None,
                    help="run only a small case of one kernel a few times (for profiler captures); prints one "
                         "line with its mean time")
    ap.add_argument("--fp8", action="store_true",
                    help="also time the FP8 (E4M3) forward on the long causal forward workloads")
    ap.add_argument("--decode", action="store_true",
                    help="also time one decoding step over the paged KV cache workload")
    ap.add_argument("--deterministic", action="store_true",
                    help="also time the deterministic backward on the same inputs")
    ap.add_argument("--varlen", action="store_true",
                    help="also time forward and backward on the packed variable-length batch")
    ap.add_argument("--forward-workloads", action="store_true",
                    help="also time the forward alone on the other forward workloads (extra keys)")
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


def cpu_threads():
    return os.cpu_count() or 1


def run_oracle_sample(w, seconds, max_slices=64):
    """Times oracle slices until ``seconds`` of work (at least 2 slices)."""
    pairs = [(b, h) for b in range(w.B) for h in range(w.H)]
    flops, elapsed, done = 0, 0.0, 0
    for b, h in pairs[:max_slices]:
        inputs = slice_inputs(w, b, h)
        t0 = time.perf_counter()
        flops += oracle_slice_pass(w, b, inputs)
        elapsed += time.perf_counter() - t0
        done += 1
        if done >= 2 and elapsed >= seconds:
            break
    return flops, elapsed, done


def reference_arm(args, info):
    from exact_io_aware_29_gb300 import synth
    if not info.is_root:
        return
    w = synth.C4
    pairs = [(b, h) for b in range(w.B) for h in range(w.H)]
    cache = {}

    def inputs(i):
        key = pairs[i % len(pairs)]
        if key not in cache:
            cache.clear()
            cache[key] = slice_inputs(w, *key)
        return key, cache[key]

    for i in range(args.warmup):
        (b, _), x = inputs(i)
        oracle_slice_pass(w, b, x)
    flops, elapsed = 0, 0.0
    for i in range(args.steps):
        (b, _), x = inputs(i)
        t0 = time.perf_counter()
        flops += oracle_slice_pass(w, b, x)
        elapsed += time.perf_counter() - t0
    value = flops / elapsed / 1e12
    sample = f"one (b,h) slice per step: fp64 oracle forward + backward, N=4096 d=128, {args.steps} slices"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * elapsed / max(args.steps, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded SplitMix64 / Box-Muller, bf16-rounded)",
        "config": {"workload": WORKLOAD, "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_threads(), "kind": "oracle",
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
def ours_arm(args, info):
    import numpy as np
    import torch
    from exact_io_aware_29_gb300 import binding, build, multi, synth

    build.build()
    binding.load_library()
    torch.cuda.set_device(info.local_rank)
    dev = torch.device("cuda", info.local_rank)
    w0 = synth.C4
    w = synth.Workload(w0.name, w0.B, w0.H, w0.N, w0.d, w0.causal, multi.rank_seed(w0.seed, info.rank),
                       q_sigma=w0.q_sigma, kv_len_range=w0.kv_len_range, backward=True)
    fwd_flops, bwd_flops, vis = flops_per_step(w)
    step_flops = fwd_flops + bwd_flops

    def host(bits):
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).pin_memory()

    hq, hk, hv, hdo = host(w.q()), host(w.k()), host(w.v()), host(w.do())
    hkv = torch.from_numpy(w.kv_lens().astype(np.int32)).pin_memory()
    q, k, v, do = (t.to(dev) for t in (hq, hk, hv, hdo))
    kv = hkv.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(binding.fa_bwd_workspace_size(w.B, w.H, w.N, w.d), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        binding.fa_fwd(q, k, v, o, lse, w.scale, True, kv, stream)
        binding.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, w.scale, True, kv, ws, stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    if binding.fa_check_status(stream) != binding.FA_OK:
        raise RuntimeError("device status error during warm-up")

    # ---- device-timed region: inputs resident in HBM
    visible = [x.strip() for x in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if x.strip()]
    sampler = ClockSampler(visible[info.local_rank] if info.local_rank < len(visible) else info.local_rank)
    sampler.start()
    binding.fa_timing_begin(args.steps)
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
    kt = {kind: binding.fa_timing_read(kind) for kind in range(4)}
    binding.fa_timing_end()
    if binding.fa_check_status(stream) != binding.FA_OK:
        raise RuntimeError("device status error in the timed region")
    value, slowest_s = multi.aggregate_throughput(step_flops * args.steps / 1e12, ms_total / 1e3)

    # ---- end to end through the public API: pinned host in, host out. Steps
    # run on three streams (host->device copies, compute, device->host copies)
    # over two sets of device buffers, so step k's results travel back while
    # step k+1's inputs arrive; every step copies its own inputs in and its own
    # results out inside the timed region.
    e2e_steps = max(1, min(args.e2e_steps, args.steps))
    ho = torch.empty_like(hq).pin_memory()
    hlse = torch.empty((w.B, w.H, w.N), dtype=torch.float32).pin_memory()
    hdq, hdk, hdv = (torch.empty_like(hq).pin_memory() for _ in range(3))
    sets = [dict(q=q, k=k, v=v, do=do, kv=kv, o=o, lse=lse, dq=dq, dk=dk, dv=dv, ws=ws)]
    sets.append({name: torch.empty_like(t) for name, t in sets[0].items()})
    s_in, s_run, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_run = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_step(i):
        b, x = sets[i % 2], i % 2
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_run[x])  # step i-2 has finished reading this set's inputs
            for dst, src in ((b["q"], hq), (b["k"], hk), (b["v"], hv), (b["do"], hdo), (b["kv"], hkv)):
                dst.copy_(src, non_blocking=True)
            ev_in[x].record(s_in)
        with torch.cuda.stream(s_run):
            s_run.wait_event(ev_in[x])
            if i >= 2:
                s_run.wait_event(ev_out[x])  # step i-2's results are back on the host
            binding.fa_fwd(b["q"], b["k"], b["v"], b["o"], b["lse"], w.scale, True, b["kv"], s_run)
            binding.fa_bwd(b["q"], b["k"], b["v"], b["o"], b["lse"], b["do"], b["dq"], b["dk"], b["dv"], w.scale,
                           True, b["kv"], b["ws"], s_run)
            ev_run[x].record(s_run)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_run[x])
            for dst, src in ((ho, b["o"]), (hlse, b["lse"]), (hdq, b["dq"]), (hdk, b["dk"]), (hdv, b["dv"])):
                dst.copy_(src, non_blocking=True)
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
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hdo, hkv))
    d2h = sum(t.numel() * t.element_size() for t in (ho, hlse, hdq, hdk, hdv))

    # ---- roofline of the dominant kernel (largest share of device time)
    peaks, peak_src = load_peaks()
    names = {0: "fa_fwd_kernel", 1: "fa_bwd_pre_kernel", 2: "fa_bwd_kernel", 3: "fa_bwd_dq_kernel"}
    kflops = {0: fwd_flops, 2: bwd_flops}
    dom = max(kt, key=lambda kd: kt[kd][0])
    dom_ms = kt[dom][0] / max(kt[dom][1], 1)
    sustained = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    burst = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    achieved = kflops.get(dom, 0) / (dom_ms / 1e3) / 1e12
    fwd_ms = kt[0][0] / max(kt[0][1], 1)
    bwd_ms = sum(kt[i][0] for i in (1, 2, 3)) / max(kt[2][1], 1)

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
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded SplitMix64 / Box-Muller, bf16-rounded), per-rank seed",
        "config": {"workload": WORKLOAD, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": True,
                   "kv_lens": [int(x) for x in w.kv_lens()], "visible_pairs": vis,
                   "flops_fwd": fwd_flops, "flops_bwd": bwd_flops,
                   "flops_fwd_nominal": 4 * w.B * w.H * w.N * w.N * w.d // 2,
                   "flops_note": "headline counts exact visible (query, key) pairs (key lengths included); the "
                                 "nominal count is 4 B H N^2 d / 2 for causal, ignoring key lengths",
                   "l2": "not flushed: the per-step working set (Q,K,V,O,dO,dQ,dK,dV bf16 and the fp32 dQ "
                         "accumulator, 0.73 GB) is larger than the 129 MB L2",
                   "parallelism": f"replicas x{info.world_size} (independent (b,h) problems, no collective)"},
        "pct_of_peak": {"step": 100 * value / info.world_size / burst,
                        "denominator": f"bf16_tflops burst {burst} ({peak_src})"},
        "breakdown": {
            "fwd_ms": fwd_ms, "fwd_tflops": tf(fwd_flops, fwd_ms),
            "fwd_pct_peak_burst": 100 * tf(fwd_flops, fwd_ms) / burst,
            "bwd_ms": bwd_ms, "bwd_tflops": tf(bwd_flops, bwd_ms),
            "bwd_pct_peak_burst": 100 * tf(bwd_flops, bwd_ms) / burst,
            "fwd_exps_per_s": vis / (fwd_ms / 1e3), "bwd_exps_per_s": vis / (bwd_ms / 1e3),
            "bwd_main_ms": kt[2][0] / max(kt[2][1], 1), "bwd_pre_ms": kt[1][0] / max(kt[1][1], 1),
            "bwd_dq_ms": kt[3][0] / max(kt[3][1], 1),
        },
        "roofline": {"kernel": names[dom], "bound": "tensor", "achieved": achieved, "peak": sustained,
                     "unit": "TFLOP/s", "frac": achieved / sustained,
                     "traffic": BWD_NCU_DRAM_BYTES if names[dom] == "fa_bwd_kernel" else None,
                     "peak_source": f"bf16_tflops_sustained ({peak_src})", "frac_of_burst": achieved / burst},
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps,
                "how": "pinned host buffers; host->device, compute and device->host on three streams over two "
                       "device buffer sets (step k's results return while step k+1's inputs arrive)"},
        "gpu_launches": 4 * args.steps,
        "clocks": clocks,
    }
    if args.forward_workloads:
        line["forward_workloads"] = forward_sweep(dev, burst)
    if args.varlen:
        line["varlen"] = varlen_measure(dev, burst, sustained, peak_src)
    if args.decode:
        line["decode"] = decode_measure(dev, peaks, peak_src)
    if args.fp8:
        line["fp8_forward"] = fp8_measure(dev, burst, peak_src)
    if args.deterministic:
        line["deterministic"] = deterministic_measure(q, k, v, o, lse, do, kv, ws, w, bwd_flops, burst, sustained,
                                                      peak_src)
    if info.is_root and info.world_size == 1 and not args.no_cpu_baseline:
        flops, el, n = run_oracle_sample(synth.C4, args.cpu_seconds)
        line["cpu_baseline"] = {"value": flops / el / 1e12, "unit": "TFLOP/s", "cores": cpu_threads(),
                                "kind": "oracle",
                                "sample": f"{n} (b,h) slices of the workload, fp64 oracle forward + backward "
                                          f"({el:.1f} s)"}
    if info.is_root:
        print(json.dumps(line), flush=True)


def forward_sweep(dev, burst, reps=20):
    """Forward-only TFLOP/s on the other forward workloads (device-resident
    random bf16 inputs of the workload's shape and Q spread; CUDA events)."""
    import torch
    from exact_io_aware_29_gb300 import binding, synth
    out = {}
    g = torch.Generator(device=dev)
    for key in ("C2", "C2C", "C3", "C5"):
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
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            binding.fa_fwd(q, k, v, o, lse, w.scale, w.causal)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        tflops = 4 * w.d * w.visible_pairs() / (ms / 1e3) / 1e12
        out[w.name] = {"ms": ms, "tflops": tflops, "pct_of_burst_peak": 100 * tflops / burst}
        del q, k, v, o, lse
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


def deterministic_measure(q, k, v, o, lse, do, kv, ws, w, bwd_flops, burst, sustained, peak_src, reps=50):
    """fa_bwd_deterministic on the step's inputs: per-kernel event times, and
    whether two calls give bitwise identical gradients."""
    import torch
    from exact_io_aware_29_gb300 import binding
    grads = [tuple(torch.empty_like(q) for _ in range(3)) for _ in range(2)]

    def bwd(g):
        binding.fa_bwd_deterministic(q, k, v, o, lse, do, *g, w.scale, True, kv, ws)

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
            "roofline": {"kernel": "fa_bwd_kernel (deterministic order)", "bound": "tensor", "achieved": main_tf,
                         "peak": sustained, "unit": "TFLOP/s", "frac": main_tf / sustained, "traffic": None,
                         "peak_source": f"bf16_tflops_sustained ({peak_src})"}}


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
        out[f"{name}_roofline"] = {"bound": "tensor", "achieved": tflops, "peak": sustained, "unit": "TFLOP/s",
                                   "frac": tflops / sustained, "traffic": None,
                                   "peak_source": f"bf16_tflops_sustained ({peak_src}); whole pass, all kernels"}
    if binding.fa_check_status() != binding.FA_OK:
        raise RuntimeError("device status error in the packed-batch measurement")
    return out


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
    ours_arm(args, info)
    if info.world_size > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
