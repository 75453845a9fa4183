"""GPU tests of the deterministic backward (fa_bwd_deterministic,
fa_bwd_varlen_deterministic): repeated calls on the same inputs give bitwise
identical dQ, dK, dV, and the results meet the oracle tolerances like fa_bwd's.
"""
import numpy as np
import pytest

import oracle
from exact_io_aware_29_gb300 import binding, build, synth
import parity_util as pu

pytestmark = pytest.mark.gpu

RUNS = 3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.load_library()


def bits(t):
    import torch
    return t.view(torch.int16).clone()


def rel_err(g, r):
    return pu.max_abs(g, r) / max(float(np.max(np.abs(r))) if r.size else 0.0, pu.ZERO_REF_FLOOR)


def repeated(fn, runs=RUNS):
    """Calls fn() `runs` times (each returns (dQ, dK, dV)) and asserts the
    results are bitwise equal; returns the first."""
    import torch
    first = None
    for _ in range(runs):
        out = fn()
        torch.cuda.synchronize()
        assert binding.fa_check_status() == binding.FA_OK
        got = tuple(bits(t) for t in out)
        if first is None:
            first = got
        else:
            for name, a, b in zip(("dQ", "dK", "dV"), first, got):
                assert torch.equal(a, b), name + " differs between runs"
    return out


FIXED = []
for d in (64, 128):
    for causal in (False, True):
        FIXED.append((1, 2, 129, d, causal, None))
        FIXED.append((2, 3, 700, d, causal, (1, 700)))
FIXED.append((1, 1, 1, 128, True, None))
FIXED.append((2, 2, 1100, 128, True, (900, 1100)))


@pytest.mark.parametrize("B,H,N,d,causal,kv", FIXED)
def test_fixed_layout_bitwise_repeatable_and_exact(B, H, N, d, causal, kv):
    seed = 7100 + N + d + (1 if causal else 0)
    w = synth.small(f"det N{N}", B, H, N, d, causal, seed, kv_len_range=kv, backward=True)
    inp = pu.Inputs(w, with_do=True)
    o, lse = binding.attention_forward(inp.q, inp.k, inp.v, w.scale, causal, inp.kv_dev)
    out = repeated(lambda: binding.attention_backward(inp.q, inp.k, inp.v, o, lse, inp.do, w.scale, causal,
                                                      inp.kv_dev, deterministic=True))
    got = [pu.bf16_tensor_to_f64(t) for t in out]
    for b in range(B):
        for h in range(H):
            ref = pu.oracle_bwd_slice(inp, b, h)
            for name, g, r in zip(("dQ", "dK", "dV"), (x[b, h] for x in got), ref):
                assert rel_err(g, r) <= pu.GRAD_RTOL, (b, h, name)


VARLEN = [
    ([300, 1, 129, 0, 128], [300, 1, 129, 0, 128]),
    ([17, 250, 64], [400, 250, 700]),
    ([300, 5, 200], [100, 5, 31]),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("case", range(len(VARLEN)))
def test_packed_layout_bitwise_repeatable_and_exact(causal, case):
    import torch
    lens_q, lens_k = VARLEN[case]
    H, d = 2, 128
    cu_q = np.concatenate([[0], np.cumsum(lens_q)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lens_k)]).astype(np.int32)
    seed = 7300 + case
    b = {n: synth.bf16_normal_tensor(seed, st, (int(cu[-1]), H, d))
         for n, st, cu in (("q", synth.STREAM_Q, cu_q), ("k", synth.STREAM_K, cu_k), ("v", synth.STREAM_V, cu_k),
                           ("do", synth.STREAM_DO, cu_q))}
    dev = {n: pu.to_device(x) for n, x in b.items()}
    cq, ck = torch.from_numpy(cu_q).cuda(), torch.from_numpy(cu_k).cuda()
    mq, mk = max(lens_q), max(lens_k)
    scale = 1 / np.sqrt(d)
    o, lse = binding.attention_forward_varlen(dev["q"], dev["k"], dev["v"], cq, ck, mq, mk, scale, causal)
    out = repeated(lambda: binding.attention_backward_varlen(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], cq,
                                                             ck, mq, mk, scale, causal, deterministic=True))
    f = {n: synth.bf16_bits_to_f64(x) for n, x in b.items()}
    ref = oracle.varlen_backward(f["q"], f["k"], f["v"], f["do"], cu_q, cu_k, scale, causal)
    for name, g, r in zip(("dQ", "dK", "dV"), out, ref):
        assert rel_err(pu.bf16_tensor_to_f64(g), r) <= pu.GRAD_RTOL, name


def test_c4_full_size_bitwise_repeatable():
    """B4 H16 N4096 d128 causal with key lengths, in the benchmark's launch
    configuration: two deterministic calls agree bit for bit, agree with the
    default order within rounding, and match the oracle on two whole slices."""
    import torch
    w = synth.C4
    inp = pu.Inputs(w, with_do=True)
    o, lse = binding.attention_forward(inp.q, inp.k, inp.v, w.scale, True, inp.kv_dev)
    ws = torch.empty(binding.fa_bwd_workspace_size(w.B, w.H, w.N, w.d), dtype=torch.uint8, device="cuda")
    det = repeated(lambda: binding.attention_backward(inp.q, inp.k, inp.v, o, lse, inp.do, w.scale, True,
                                                      inp.kv_dev, ws, deterministic=True), runs=2)
    fast = binding.attention_backward(inp.q, inp.k, inp.v, o, lse, inp.do, w.scale, True, inp.kv_dev, ws)
    torch.cuda.synchronize()
    for name, a, b in zip(("dQ", "dK", "dV"), det, fast):
        a, b = a.float(), b.float()
        assert (a - b).abs().max().item() <= 1e-2 * b.abs().max().item(), name
    got = [pu.bf16_tensor_to_f64(t) for t in det]
    for b, h in ((0, 0), (3, 15)):
        ref = pu.oracle_bwd_slice(inp, b, h)
        for name, g, r in zip(("dQ", "dK", "dV"), (x[b, h] for x in got), ref):
            assert rel_err(g, r) <= pu.GRAD_RTOL, (b, h, name)
