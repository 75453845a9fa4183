"""Helpers shared by the GPU parity tests: seeded inputs to device tensors,
oracle evaluation on whole slices or sampled rows, and the error metrics."""
from __future__ import annotations

import numpy as np

import oracle
from exact_io_aware_29_gb300 import synth

# Tolerances for bf16 inputs/outputs with fp32 accumulation.
O_ATOL = 1e-2        # forward O: max |gpu - oracle|
LSE_ATOL = 1e-3      # forward LSE: max |gpu - oracle|
GRAD_RTOL = 1e-2     # dQ/dK/dV: max |gpu - oracle| / max |oracle|
ZERO_REF_FLOOR = 1e-3  # denominator floor when a reference gradient is identically 0


def to_device(bits: np.ndarray):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16).cuda()


def bf16_tensor_to_f64(t) -> np.ndarray:
    import torch
    return t.detach().to(torch.float32).cpu().numpy().astype(np.float64)


class Inputs:
    """Seeded bf16 inputs of a workload, as bit patterns, fp64 values and device tensors."""

    def __init__(self, w: synth.Workload, with_do: bool = False):
        import torch
        self.w = w
        self.q_bits, self.k_bits, self.v_bits = w.q(), w.k(), w.v()
        self.do_bits = w.do() if with_do else None
        lens = w.kv_lens()
        self.kv_lens = lens
        self.q, self.k, self.v = (to_device(b) for b in (self.q_bits, self.k_bits, self.v_bits))
        self.do = to_device(self.do_bits) if with_do else None
        self.kv_dev = None if lens is None else torch.from_numpy(lens.astype(np.int32)).cuda()

    def f64(self, name):
        return synth.bf16_bits_to_f64(getattr(self, name + "_bits"))

    def kv_len(self, b):
        return None if self.kv_lens is None else int(self.kv_lens[b])


def max_abs(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    both_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
    with np.errstate(invalid="ignore"):  # inf - inf where both are the same infinity (masked out)
        d = np.where(both_inf, 0.0, np.abs(a - b))
    return float(np.max(d)) if d.size else 0.0


def bf16_half_ulp(x) -> np.ndarray:
    """Half the spacing of bf16 numbers at |x|: the rounding error of handing
    x back in bf16 (2^(e-8) for |x| in [2^e, 2^(e+1)), 8 significant bits;
    the subnormal spacing below 2^-126)."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(ax, 2.0 ** -126)))
    return np.ldexp(1.0, e.astype(np.int64) - 8)


def o_err(gpu, ref) -> float:
    """Forward O error against the oracle: max over elements of |gpu - ref|
    less the bf16 rounding of the reference value itself. O is delivered in
    bf16, so an exact kernel still errs by up to half an ulp of O (0.0156 for
    |O| in [4, 8)); the 1e-2 bound applies to what the computation adds."""
    g = np.asarray(gpu, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    both_inf = np.isinf(g) & np.isinf(r) & (np.sign(g) == np.sign(r))
    with np.errstate(invalid="ignore"):  # inf - inf where both are the same infinity (masked out)
        d = np.where(both_inf, 0.0, np.abs(g - r) - np.where(np.isfinite(r), bf16_half_ulp(r), 0.0))
    return float(np.max(d)) if d.size else 0.0


def oracle_fwd_slice(inp: Inputs, b: int, h: int, rows=None):
    """Oracle O, LSE for one (b, h) slice, for all rows or for ``rows``."""
    q = synth.bf16_bits_to_f64(inp.q_bits[b, h])
    k = synth.bf16_bits_to_f64(inp.k_bits[b, h])
    v = synth.bf16_bits_to_f64(inp.v_bits[b, h])
    w = inp.w
    if rows is None:
        return oracle.attention_forward(q, k, v, w.scale, w.causal, inp.kv_len(b))
    return oracle.attention_forward_rows(q, k, v, rows, w.scale, w.causal, inp.kv_len(b))


def oracle_bwd_slice(inp: Inputs, b: int, h: int):
    q = synth.bf16_bits_to_f64(inp.q_bits[b, h])
    k = synth.bf16_bits_to_f64(inp.k_bits[b, h])
    v = synth.bf16_bits_to_f64(inp.v_bits[b, h])
    do = synth.bf16_bits_to_f64(inp.do_bits[b, h])
    w = inp.w
    return oracle.attention_backward(q, k, v, do, w.scale, w.causal, inp.kv_len(b))


# ---------------------------------------------------------------------------
# Oracle on many slices at once: spawned host processes (no CUDA context is
# inherited), single-threaded BLAS each, one slice (or row chunk) per job.
# ---------------------------------------------------------------------------
def _fwd_job(args):
    q, k, v, scale, causal, kv_len, rows = args
    if rows is None:
        return oracle.attention_forward(q, k, v, scale, causal, kv_len)
    return oracle.attention_forward_rows(q, k, v, rows, scale, causal, kv_len)


def _bwd_job(args):
    q, k, v, do, scale, causal, kv_len = args
    return oracle.attention_backward(q, k, v, do, scale, causal, kv_len)


class OraclePool:
    """``with OraclePool() as pool: pool.fwd(jobs)`` maps the oracle over
    (q, k, v, scale, causal, kv_len, rows) jobs in host processes."""

    def __init__(self, workers=None):
        import multiprocessing as mp
        import os
        try:
            n = len(os.sched_getaffinity(0))
        except AttributeError:
            n = os.cpu_count() or 1
        self.n = workers or max(1, min(n, 32))
        keys = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")
        saved = {k: os.environ.get(k) for k in keys}
        for k in keys:
            os.environ[k] = "1"
        try:
            self.pool = mp.get_context("spawn").Pool(self.n)
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.pool.close()
        self.pool.join()

    def fwd(self, jobs):
        return self.pool.map(_fwd_job, jobs, chunksize=1)

    def bwd(self, jobs):
        return self.pool.map(_bwd_job, jobs, chunksize=1)


def slice_f64(bits, b, h):
    return synth.bf16_bits_to_f64(bits[b, h])
