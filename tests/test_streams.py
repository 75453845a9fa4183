"""Several forward + backward problems in flight at once, each on a CUDA
stream of its own with a backward workspace of its own. The library keeps no
device state shared between calls (the backward's counters, ticket and dQ
accumulator live in the caller's workspace), so every result must equal the
same problem run alone: the forward and the deterministic backward bit for
bit, the default backward's dK and dV bit for bit (each is summed inside one
CTA), and its dQ (summed by L2 reductions in any order) within the oracle's
tolerance."""
import numpy as np
import pytest

from exact_io_aware_29_gb300 import binding, build, synth
import parity_util as pu

pytestmark = pytest.mark.gpu

# (B, H, N, d, causal, key-length range, deterministic backward)
JOBS = [
    (2, 3, 700, 128, True, (300, 700), False),
    (1, 4, 513, 64, False, None, True),
    (2, 2, 1000, 128, False, (1, 1000), True),
    (1, 40, 384, 64, True, None, False),  # more backward items than SMs
    (3, 2, 257, 128, True, None, False),
    (1, 2, 900, 64, True, (450, 900), True),
]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.load_library()


def rel_err(g, r):
    return pu.max_abs(g, r) / max(float(np.max(np.abs(r))), pu.ZERO_REF_FLOOR)


def test_problems_on_concurrent_streams_match_each_run_alone():
    import torch
    jobs = []
    for n, (B, H, N, d, causal, kv, det) in enumerate(JOBS):
        w = synth.small(f"streams {n}", B, H, N, d, causal, 5300 + n, kv_len_range=kv, backward=True)
        inp = pu.Inputs(w, with_do=True)
        o, lse = binding.attention_forward(inp.q, inp.k, inp.v, w.scale, causal, inp.kv_dev)
        alone = binding.attention_backward(inp.q, inp.k, inp.v, o, lse, inp.do, w.scale, causal, inp.kv_dev,
                                           deterministic=det)
        out = dict(o=torch.empty_like(o), lse=torch.empty_like(lse),
                   grads=[torch.empty_like(inp.q) for _ in range(3)],
                   ws=torch.empty(binding.fa_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device="cuda"))
        jobs.append((inp, det, (o, lse, alone), out, torch.cuda.Stream()))
    torch.cuda.synchronize()

    # Every job issued three times, interleaved across the streams, with no
    # host synchronisation in between: kernels of different jobs overlap.
    for _ in range(3):
        for inp, det, _, out, s in jobs:
            w = inp.w
            binding.fa_fwd(inp.q, inp.k, inp.v, out["o"], out["lse"], w.scale, w.causal, inp.kv_dev, s)
            fn = binding.fa_bwd_deterministic if det else binding.fa_bwd
            fn(inp.q, inp.k, inp.v, out["o"], out["lse"], inp.do, *out["grads"], w.scale, w.causal, inp.kv_dev,
               out["ws"], s)
    torch.cuda.synchronize()
    for inp, det, (o, lse, alone), out, s in jobs:
        assert binding.fa_check_status(s) == binding.FA_OK
        assert torch.equal(out["o"].view(torch.int16), o.view(torch.int16))
        assert torch.equal(out["lse"], lse)
        dq, dk, dv = out["grads"]
        assert torch.equal(dk.view(torch.int16), alone[1].view(torch.int16))
        assert torch.equal(dv.view(torch.int16), alone[2].view(torch.int16))
        if det:
            assert torch.equal(dq.view(torch.int16), alone[0].view(torch.int16))
        g = pu.bf16_tensor_to_f64(dq)
        w = inp.w
        for b in range(w.B):
            for h in range(w.H):
                ref = pu.oracle_bwd_slice(inp, b, h)
                assert np.all(np.isfinite(g[b, h]))
                assert rel_err(g[b, h], ref[0]) <= pu.GRAD_RTOL, (w.name, b, h)
