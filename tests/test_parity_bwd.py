"""GPU backward parity against the fp64 oracle, through the C ABI.

The GPU forward supplies O and LSE (as in training); the oracle computes the
gradients of sum(O * dO) from Q, K, V, dO alone. Tolerance per tensor:
max |gpu - oracle| / max |oracle| <= 1e-2.
"""
import numpy as np
import pytest

from exact_io_aware_29_gb300 import binding, build, synth
import parity_util as pu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.load_library()


def run_bwd(inp):
    import torch
    w = inp.w
    o, lse = binding.attention_forward(inp.q, inp.k, inp.v, w.scale, w.causal, inp.kv_dev)
    dq, dk, dv = binding.attention_backward(inp.q, inp.k, inp.v, o, lse, inp.do, w.scale, w.causal,
                                            inp.kv_dev)
    torch.cuda.synchronize()
    assert binding.fa_check_status() == binding.FA_OK
    return tuple(pu.bf16_tensor_to_f64(t) for t in (dq, dk, dv))


def rel_err(g, r):
    # A reference that is identically zero (one visible key makes dS = 0, so
    # dQ = dK = 0) leaves the ratio undefined: the denominator is then bounded
    # below by ZERO_REF_FLOOR, i.e. absolute residuals up to 1e-5 are accepted.
    return pu.max_abs(g, r) / max(float(np.max(np.abs(r))), pu.ZERO_REF_FLOOR)


def check(inp, pairs=None):
    w = inp.w
    dq, dk, dv = run_bwd(inp)
    for t in (dq, dk, dv):
        assert np.all(np.isfinite(t))
    pairs = pairs or [(b, h) for b in range(w.B) for h in range(w.H)]
    worst = [0.0, 0.0, 0.0]
    for b, h in pairs:
        ref = pu.oracle_bwd_slice(inp, b, h)
        for n, (g, r) in enumerate(zip((dq[b, h], dk[b, h], dv[b, h]), ref)):
            worst[n] = max(worst[n], rel_err(g, r))
        L = inp.kv_len(b)
        if L is not None and L < w.N:  # keys past the valid length get exactly zero gradient
            assert np.all(dk[b, h][L:] == 0) and np.all(dv[b, h][L:] == 0)
    msg = "relative max errors dQ %.3g dK %.3g dV %.3g" % tuple(worst)
    assert max(worst) <= pu.GRAD_RTOL, msg
    return worst


SMALL = []
for d in (64, 128):
    for causal in (False, True):
        for n in (1, 17, 128, 129, 300, 513):
            SMALL.append((1, 2, n, d, causal, None))
        SMALL.append((3, 2, 700, d, causal, (1, 700)))
        SMALL.append((2, 1, 384, d, causal, (128, 128)))
        SMALL.append((2, 1, 256, d, causal, (0, 0)))


@pytest.mark.parametrize("B,H,N,d,causal,kv", SMALL)
def test_bwd_small_full(B, H, N, d, causal, kv):
    seed = 5000 + N * 7 + d + (1 if causal else 0) + (0 if kv is None else kv[0])
    w = synth.small(f"bwd N{N}", B, H, N, d, causal, seed, kv_len_range=kv, backward=True)
    check(pu.Inputs(w, with_do=True))


def test_bwd_many_query_blocks():
    w = synth.small("bwd N1100", 1, 2, 1100, 128, True, 31, kv_len_range=(900, 1100), backward=True)
    check(pu.Inputs(w, with_do=True))


def test_bwd_deterministic_dk_dv():
    import torch
    w = synth.small("det", 1, 2, 600, 128, True, 12, backward=True)
    inp = pu.Inputs(w, with_do=True)
    o, lse = binding.attention_forward(inp.q, inp.k, inp.v, w.scale, True)
    a = binding.attention_backward(inp.q, inp.k, inp.v, o, lse, inp.do, w.scale, True)
    b = binding.attention_backward(inp.q, inp.k, inp.v, o, lse, inp.do, w.scale, True)
    torch.cuda.synchronize()
    # dK and dV are accumulated in one CTA each: bitwise reproducible.
    assert torch.equal(a[1].view(torch.int16), b[1].view(torch.int16))
    assert torch.equal(a[2].view(torch.int16), b[2].view(torch.int16))


@pytest.mark.slow
def test_bwd_c4_full_size_every_slice():
    """All 64 (b, h) slices of the benchmark's workload (every L2 head group of
    the persistent kernel, the last one included), in the full-size launch
    the benchmark times; the oracle runs on host processes in parallel."""
    w = synth.C4
    inp = pu.Inputs(w, with_do=True)
    dq, dk, dv = run_bwd(inp)
    pairs = [(b, h) for b in range(w.B) for h in range(w.H)]
    jobs = [tuple(pu.slice_f64(x, b, h) for x in (inp.q_bits, inp.k_bits, inp.v_bits, inp.do_bits))
            + (w.scale, True, inp.kv_len(b)) for b, h in pairs]
    with pu.OraclePool() as pool:
        refs = pool.bwd(jobs)
    worst = [0.0, 0.0, 0.0]
    for (b, h), ref in zip(pairs, refs):
        for n, (g, r) in enumerate(zip((dq[b, h], dk[b, h], dv[b, h]), ref)):
            assert np.all(np.isfinite(g))
            worst[n] = max(worst[n], rel_err(g, r))
        L = inp.kv_len(b)
        assert np.all(dk[b, h][L:] == 0) and np.all(dv[b, h][L:] == 0)
    assert max(worst) <= pu.GRAD_RTOL, "relative max errors dQ %.3g dK %.3g dV %.3g" % tuple(worst)


# The main kernel is persistent (one CTA per SM taking work items in turn), so
# shapes with more items than SMs make every CTA run several items: the item
# ring, barrier phases counted across items and accumulators restarted per
# item are only exercised there. 2 x 48 heads x 6 key blocks = 576 items, some
# of them past kv_len (written as zeros without entering the main loop).
MANY_ITEMS = [(128, True), (64, True), (128, False)]
MANY_PAIRS = [(0, 0), (0, 23), (0, 47), (1, 5), (1, 30), (1, 47)]


@pytest.mark.parametrize("d,causal", MANY_ITEMS)
def test_bwd_many_items_per_cta(d, causal):
    w = synth.small(f"bwd items d{d}", 2, 48, 768, d, causal, 77 + d + causal, kv_len_range=(200, 768),
                    backward=True)
    check(pu.Inputs(w, with_do=True), MANY_PAIRS)


def test_bwd_deterministic_many_items_per_cta():
    import torch
    w = synth.small("det items", 2, 48, 768, 128, True, 91, kv_len_range=(200, 768), backward=True)
    inp = pu.Inputs(w, with_do=True)
    o, lse = binding.attention_forward(inp.q, inp.k, inp.v, w.scale, True, inp.kv_dev)
    runs = [binding.attention_backward(inp.q, inp.k, inp.v, o, lse, inp.do, w.scale, True, inp.kv_dev,
                                       deterministic=True) for _ in range(2)]
    torch.cuda.synchronize()
    assert binding.fa_check_status() == binding.FA_OK
    for a, b in zip(*runs):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    dq, dk, dv = (pu.bf16_tensor_to_f64(t) for t in runs[0])
    worst = 0.0
    for b, h in MANY_PAIRS[:3]:
        for g, r in zip((dq[b, h], dk[b, h], dv[b, h]), pu.oracle_bwd_slice(inp, b, h)):
            worst = max(worst, rel_err(g, r))
    assert worst <= pu.GRAD_RTOL, worst
