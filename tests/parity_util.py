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
    d = np.where(both_inf, 0.0, np.abs(a - b))
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
