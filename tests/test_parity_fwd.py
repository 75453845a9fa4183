"""GPU forward parity against the fp64 oracle, through the C ABI.

Small cases compare every element of O and LSE; the full-size workloads
compare seeded sampled rows of every head (the oracle evaluates those rows one
by one from the definition), in the same launch configuration the benchmark
times.
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


def run_fwd(inp):
    import torch
    w = inp.w
    o, lse = binding.attention_forward(inp.q, inp.k, inp.v, w.scale, w.causal, inp.kv_dev)
    torch.cuda.synchronize()
    assert binding.fa_check_status() == binding.FA_OK
    return pu.bf16_tensor_to_f64(o), lse.cpu().numpy().astype(np.float64)


def check_full(inp):
    o, lse = run_fwd(inp)
    w = inp.w
    worst_o = worst_l = 0.0
    for b in range(w.B):
        for h in range(w.H):
            ro, rl = pu.oracle_fwd_slice(inp, b, h)
            worst_o = max(worst_o, pu.o_err(o[b, h], ro))
            worst_l = max(worst_l, pu.max_abs(lse[b, h], rl))
    assert np.all(np.isfinite(o)), "non-finite O"
    assert worst_o <= pu.O_ATOL, f"O max abs err {worst_o}"
    assert worst_l <= pu.LSE_ATOL, f"LSE max abs err {worst_l}"
    return worst_o, worst_l


SMALL = []
for d in (64, 128):
    for causal in (False, True):
        for n in (1, 17, 128, 129, 255, 300, 513):
            SMALL.append((1, 2, n, d, causal, None))
        SMALL.append((3, 2, 700, d, causal, (1, 700)))
        SMALL.append((2, 1, 1000, d, causal, (0, 0)))        # every key masked
        SMALL.append((2, 1, 384, d, causal, (1, 1)))         # a single visible key
        SMALL.append((2, 1, 384, d, causal, (128, 128)))     # block-aligned key limit


@pytest.mark.parametrize("B,H,N,d,causal,kv", SMALL)
def test_fwd_small_full(B, H, N, d, causal, kv):
    seed = 1000 + N * 7 + d + (1 if causal else 0) + (0 if kv is None else kv[0])
    w = synth.small(f"small N{N}", B, H, N, d, causal, seed, kv_len_range=kv)
    check_full(pu.Inputs(w))


def test_fwd_c1_full():
    check_full(pu.Inputs(synth.C1))


def test_fwd_large_logits_force_rescaling():
    # q ~ N(0, 4^2) as in the long causal d=128 workload, at a size the oracle finishes fully.
    w = synth.small("rescale", 1, 4, 1024, 128, True, 77, q_sigma=4.0)
    check_full(pu.Inputs(w))


def test_fwd_kv_len_zero_row_values():
    w = synth.small("empty", 1, 1, 200, 64, False, 5, kv_len_range=(0, 0))
    o, lse = run_fwd(pu.Inputs(w))
    assert np.all(o == 0) and np.all(lse == -np.inf)


def test_fwd_deterministic():
    import torch
    inp = pu.Inputs(synth.small("det", 2, 3, 777, 128, True, 9, kv_len_range=(300, 777)))
    w = inp.w
    o1, l1 = binding.attention_forward(inp.q, inp.k, inp.v, w.scale, w.causal, inp.kv_dev)
    o2, l2 = binding.attention_forward(inp.q, inp.k, inp.v, w.scale, w.causal, inp.kv_dev)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)


def check_sampled(w, rows_per_head, heads=None):
    inp = pu.Inputs(w)
    o, lse = run_fwd(inp)
    worst_o = worst_l = 0.0
    pairs = heads or [(b, h) for b in range(w.B) for h in range(w.H)]
    for b, h in pairs:
        rows = synth.distinct_rows(w.seed, synth.STREAM_ROWS, rows_per_head, w.N, salt=b * w.H + h)
        ro, rl = pu.oracle_fwd_slice(inp, b, h, rows)
        worst_o = max(worst_o, pu.o_err(o[b, h][rows], ro))
        worst_l = max(worst_l, pu.max_abs(lse[b, h][rows], rl))
    assert np.all(np.isfinite(o))
    assert worst_o <= pu.O_ATOL, f"O max abs err {worst_o}"
    assert worst_l <= pu.LSE_ATOL, f"LSE max abs err {worst_l}"


def check_rows_pooled(w, jobs_of):
    """Runs the forward once at full size, then compares the (b, h, rows)
    pieces ``jobs_of`` names against the oracle, evaluated on host processes
    in parallel (rows=None: the whole slice)."""
    inp = pu.Inputs(w)
    o, lse = run_fwd(inp)
    assert np.all(np.isfinite(o))
    pieces = list(jobs_of(w))
    jobs = [tuple(pu.slice_f64(x, b, h) for x in (inp.q_bits, inp.k_bits, inp.v_bits))
            + (w.scale, w.causal, inp.kv_len(b), rows) for b, h, rows in pieces]
    with pu.OraclePool() as pool:
        refs = pool.fwd(jobs)
    worst_o = worst_l = 0.0
    for (b, h, rows), (ro, rl) in zip(pieces, refs):
        sel = slice(None) if rows is None else rows
        worst_o = max(worst_o, pu.o_err(o[b, h][sel], ro))
        worst_l = max(worst_l, pu.max_abs(lse[b, h][sel], rl))
    assert worst_o <= pu.O_ATOL, f"O max abs err {worst_o}"
    assert worst_l <= pu.LSE_ATOL, f"LSE max abs err {worst_l}"


@pytest.mark.slow
@pytest.mark.parametrize("name", ["C2", "C2C"])
def test_fwd_c2_every_row(name):
    """Every row of every head of the d = 64 workload."""
    check_rows_pooled(synth.WORKLOADS[name],
                      lambda w: ((b, h, None) for b in range(w.B) for h in range(w.H)))


@pytest.mark.slow
def test_fwd_c3_every_row_of_two_heads():
    """Every row of one head per batch entry (in 1024-row pieces), plus the
    seeded sampled rows of every other head."""
    def pieces(w):
        full = {(b, (7 * b + 5) % w.H) for b in range(w.B)}
        for b, h in sorted(full):
            for r0 in range(0, w.N, 1024):
                yield b, h, np.arange(r0, min(r0 + 1024, w.N))
        for b in range(w.B):
            for h in range(w.H):
                if (b, h) not in full:
                    yield b, h, synth.distinct_rows(w.seed, synth.STREAM_ROWS, w.sample_rows, w.N,
                                                    salt=b * w.H + h)
    check_rows_pooled(synth.C3, pieces)


@pytest.mark.slow
def test_fwd_c4_every_row():
    """Every row of every head of the benchmark's step workload (key lengths
    per batch entry), in the full-size launch."""
    check_rows_pooled(synth.C4, lambda w: ((b, h, None) for b in range(w.B) for h in range(w.H)))


@pytest.mark.slow
def test_fwd_c5_sampled():
    check_sampled(synth.C5, synth.C5.sample_rows)


@pytest.mark.slow
def test_fwd_l1_sampled():
    """The longest forward the benchmark times (B1 H8 N131072 d128 causal):
    seeded rows of every head, in the full-size launch."""
    check_sampled(synth.L1, synth.L1.sample_rows)


@pytest.mark.slow
def test_fwd_nc_sampled():
    """The benchmark's non-causal d = 128 point (B2 H16 N8192): seeded rows of
    every head."""
    check_sampled(synth.NC, synth.NC.sample_rows)


# More Q-tile pairs than SMs: every SM runs several CTAs in turn, in the
# head-grouped order, with key padding that leaves some CTAs a short key range
# and some second tiles past the query length.
MANY_ITEMS = [(64, False), (64, True), (128, False), (128, True)]


@pytest.mark.parametrize("d,causal", MANY_ITEMS)
def test_fwd_many_items_per_cta(d, causal):
    w = synth.small(f"fwd items d{d}", 2, 24, 1300, d, causal, 401 + d + causal, kv_len_range=(90, 1300))
    check_full(pu.Inputs(w))
