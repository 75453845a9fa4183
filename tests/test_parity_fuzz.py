"""Seeded random shapes through the forward and the backward, against the fp64
oracle, through the C ABI.

The hand-picked cases elsewhere cover the named edge cases one at a time; this
sweep draws batch, heads, length, head dim, mask and key lengths at random
(seeded), so that combinations of them (ragged tails in both tiles of a CTA,
non-causal grids whose last partial wave is split into single-tile CTAs, key
lengths of zero next to full ones, lengths of one) meet the kernels together.
Tolerances are the ones every parity test uses (O 1e-2, LSE 1e-3). The gradients
are checked against the oracle's backward with its row term D = rowsum(dO ∘ O)
taken from the oracle's own output rounded to bf16, as the method's backward
forms it from the stored O; against the definition's rowsum(dP ∘ P) too when
the slice has four keys or more. With two or three keys dQ and dK nearly cancel
(every row of dS sums to zero) and O's bf16 rounding, entering through D,
takes the error against the definition to about 1.2 % of max |dQ|.
"""
import numpy as np
import pytest

import oracle
from exact_io_aware_29_gb300 import binding, build, synth
import parity_util as pu

pytestmark = pytest.mark.gpu


def _cases(n=20, seed=20261203):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        B = int(rng.integers(1, 4))
        H = int(rng.integers(1, 4))
        N = int(np.clip(np.exp(rng.uniform(0.0, np.log(900.0))), 1, 900))
        d = int(rng.choice([64, 128]))
        causal = bool(rng.integers(0, 2))
        kv = None
        if rng.uniform() < 0.5:
            lo = int(rng.integers(0, N + 1))
            kv = (lo, int(rng.integers(lo, N + 1)))
        out.append((i, B, H, N, d, causal, kv))
    return out


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.load_library()


def _rel_err(g, r):
    return pu.max_abs(g, r) / max(float(np.max(np.abs(r))), pu.ZERO_REF_FLOOR)


@pytest.mark.parametrize("i,B,H,N,d,causal,kv", _cases())
def test_fuzz_forward_backward(i, B, H, N, d, causal, kv):
    import torch
    w = synth.small(f"fuzz {i}", B, H, N, d, causal, 90000 + i, kv_len_range=kv, backward=True)
    inp = pu.Inputs(w, with_do=True)
    o, lse = binding.attention_forward(inp.q, inp.k, inp.v, w.scale, w.causal, inp.kv_dev)
    grads = [binding.attention_backward(inp.q, inp.k, inp.v, o, lse, inp.do, w.scale, w.causal, inp.kv_dev,
                                        deterministic=det) for det in (False, True)]
    torch.cuda.synchronize()
    assert binding.fa_check_status() == binding.FA_OK
    o, lse = pu.bf16_tensor_to_f64(o), lse.cpu().numpy().astype(np.float64)
    for dq, dk, dv in grads:
        _check_fixed(inp, o, lse, *(pu.bf16_tensor_to_f64(t) for t in (dq, dk, dv)))


def _check_fixed(inp, o, lse, dq, dk, dv):
    w = inp.w
    B, H, N = w.B, w.H, w.N
    worst_o = worst_l = 0.0
    worst_g = [0.0, 0.0, 0.0]
    for b in range(B):
        for h in range(H):
            ro, rl = pu.oracle_fwd_slice(inp, b, h)
            worst_o = max(worst_o, pu.o_err(o[b, h], ro))
            worst_l = max(worst_l, pu.max_abs(lse[b, h], rl))
            o_st = synth.bf16_bits_to_f64(synth.f32_to_bf16_bits(np.asarray(ro, dtype=np.float32)))
            ref = oracle.attention_backward(pu.slice_f64(inp.q_bits, b, h), pu.slice_f64(inp.k_bits, b, h),
                                            pu.slice_f64(inp.v_bits, b, h), pu.slice_f64(inp.do_bits, b, h),
                                            w.scale, w.causal, inp.kv_len(b), o_stored=o_st)
            keys = N if inp.kv_len(b) is None else min(N, inp.kv_len(b))
            refs = [ref] + ([pu.oracle_bwd_slice(inp, b, h)] if keys >= 4 else [])
            for rr in refs:
                for n, (g, r) in enumerate(zip((dq[b, h], dk[b, h], dv[b, h]), rr)):
                    worst_g[n] = max(worst_g[n], _rel_err(g, r))
            L = inp.kv_len(b)
            if L is not None and L < N:  # keys past the valid length get exactly zero gradient
                assert np.all(dk[b, h][L:] == 0) and np.all(dv[b, h][L:] == 0)
    assert np.all(np.isfinite(o)) and all(np.all(np.isfinite(t)) for t in (dq, dk, dv))
    assert worst_o <= pu.O_ATOL, f"O max abs err {worst_o}"
    assert worst_l <= pu.LSE_ATOL, f"LSE max abs err {worst_l}"
    assert max(worst_g) <= pu.GRAD_RTOL, "relative max errors dQ %.3g dK %.3g dV %.3g" % tuple(worst_g)


def _varlen_cases(n=12, seed=20261204):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        S = int(rng.integers(1, 6))

        def draw():  # a fifth of the sequences empty
            return [0 if rng.uniform() < 0.2 else int(rng.integers(1, 601)) for _ in range(S)]

        lq = draw()
        lk = list(lq) if rng.uniform() < 0.5 else draw()
        if sum(lq) == 0:
            lq[0] = 1
        if sum(lk) == 0:
            lk[0] = 1
        out.append((i, lq, lk, int(rng.integers(1, 4)), int(rng.choice([64, 128])), bool(rng.integers(0, 2))))
    return out


@pytest.mark.parametrize("i,lens_q,lens_k,H,d,causal", _varlen_cases())
def test_fuzz_packed_forward_backward(i, lens_q, lens_k, H, d, causal):
    """Packed batches of random query and key lengths (empty sequences and
    Lq != Lk included, bottom-right causal), forward and backward."""
    import torch
    cu_q = np.concatenate([[0], np.cumsum(lens_q)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lens_k)]).astype(np.int32)
    tq, tk = int(cu_q[-1]), int(cu_k[-1])
    seed = 95000 + i
    bits = {"q": synth.bf16_normal_tensor(seed, synth.STREAM_Q, (tq, H, d)),
            "k": synth.bf16_normal_tensor(seed, synth.STREAM_K, (tk, H, d)),
            "v": synth.bf16_normal_tensor(seed, synth.STREAM_V, (tk, H, d)),
            "do": synth.bf16_normal_tensor(seed, synth.STREAM_DO, (tq, H, d))}
    dev = {n: pu.to_device(b) for n, b in bits.items()}
    f64 = {n: synth.bf16_bits_to_f64(b) for n, b in bits.items()}
    cq, ck = torch.from_numpy(cu_q).cuda(), torch.from_numpy(cu_k).cuda()
    scale = 1 / np.sqrt(d)
    mq, mk = max(max(lens_q), 1), max(max(lens_k), 1)
    o, lse = binding.attention_forward_varlen(dev["q"], dev["k"], dev["v"], cq, ck, mq, mk, scale, causal)
    grads = [binding.attention_backward_varlen(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], cq, ck, mq, mk,
                                               scale, causal, deterministic=det) for det in (False, True)]
    torch.cuda.synchronize()
    assert binding.fa_check_status() == binding.FA_OK
    ro, rl = oracle.varlen_forward(f64["q"], f64["k"], f64["v"], cu_q, cu_k, scale, causal)
    go, gl = pu.bf16_tensor_to_f64(o), lse.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(go))
    assert pu.o_err(go, ro) <= pu.O_ATOL
    assert pu.max_abs(gl, rl) <= pu.LSE_ATOL
    # Gradients against the oracle with D from its own output rounded to bf16
    # (see the module docstring), sequence by sequence.
    o_st = synth.bf16_bits_to_f64(synth.f32_to_bf16_bits(np.asarray(ro, dtype=np.float32)))
    rq, rk, rv = np.zeros_like(f64["q"]), np.zeros_like(f64["k"]), np.zeros_like(f64["v"])
    for b in range(len(lens_q)):
        qa, qe, ka, ke = int(cu_q[b]), int(cu_q[b + 1]), int(cu_k[b]), int(cu_k[b + 1])
        for h in range(H):
            rq[qa:qe, h], rk[ka:ke, h], rv[ka:ke, h] = oracle.attention_backward(
                f64["q"][qa:qe, h], f64["k"][ka:ke, h], f64["v"][ka:ke, h], f64["do"][qa:qe, h], scale, causal,
                None, (ke - ka) - (qe - qa), o_stored=o_st[qa:qe, h])
    for det, (dq, dk, dv) in zip((False, True), grads):
        for name, g, r in (("dQ", dq, rq), ("dK", dk, rk), ("dV", dv, rv)):
            g = pu.bf16_tensor_to_f64(g)
            assert np.all(np.isfinite(g)), (det, name)
            assert _rel_err(g, r) <= pu.GRAD_RTOL, (det, name, _rel_err(g, r))


def _fp8_cases(n=10, seed=20261205):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        N = int(np.clip(np.exp(rng.uniform(0.0, np.log(900.0))), 1, 900))
        kv = None
        if rng.uniform() < 0.5:
            lo = int(rng.integers(0, N + 1))
            kv = (lo, int(rng.integers(lo, N + 1)))
        out.append((i, int(rng.integers(1, 4)), int(rng.integers(1, 4)), N, bool(rng.integers(0, 2)), kv))
    return out


@pytest.mark.parametrize("i,B,H,N,causal,kv", _fp8_cases())
def test_fuzz_fp8_forward(i, B, H, N, causal, kv):
    """The FP8 forward (head dim 128) on random shapes, within the bounds of
    rounding P to E4M3 (the FP8 parity tests' criterion)."""
    import torch
    from test_parity_fp8 import _check_rows
    w = synth.small(f"fuzz fp8 {i}", B, H, N, 128, causal, 97000 + i, kv_len_range=kv)
    inp = pu.Inputs(w)
    o, lse, _ = binding.attention_forward_fp8(inp.q, inp.k, inp.v, w.scale, causal, inp.kv_dev)
    torch.cuda.synchronize()
    assert binding.fa_check_status() == binding.FA_OK
    go, gl = pu.bf16_tensor_to_f64(o), lse.cpu().numpy()
    assert np.all(np.isfinite(go))
    for b in range(B):
        for h in range(H):
            _check_rows(go[b, h], gl[b, h], inp.q_bits[b, h], inp.k_bits[b, h], inp.v_bits[b, h], w.scale, causal,
                        inp.kv_len(b))


def _decode_cases(n=8, seed=20261206):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        B = int(rng.integers(1, 7))
        bs = int(rng.choice([64, 128, 256, 512]))
        lens = [0 if rng.uniform() < 0.15 else int(rng.integers(1, 3000)) for _ in range(B)]
        out.append((i, lens, int(rng.integers(1, 4)), int(rng.choice([64, 128])), bs))
    return out


@pytest.mark.parametrize("i,lens,H,d,bs", _decode_cases())
def test_fuzz_paged_decode(i, lens, H, d, bs):
    """Decoding from a paged cache with random lengths (empty ones included),
    heads, head dims and page sizes."""
    from test_parity_decode import run
    top = max(max(lens), 1)
    w = synth.DecodeWorkload(f"fuzz dec {i}", len(lens), H, d, bs, 98000 + i, (top, top), spare_blocks=2)
    run(w, lens=lens)


def _many_head_cases(n=4, seed=20261207):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        B = int(rng.integers(1, 9))
        H = int(rng.integers(8, 49))
        N = int(rng.integers(100, 400))
        kv = None if rng.uniform() < 0.5 else (1, N)
        out.append((i, B, H, N, int(rng.choice([64, 128])), bool(rng.integers(0, 2)), kv))
    return out


@pytest.mark.parametrize("i,B,H,N,d,causal,kv", _many_head_cases())
def test_fuzz_many_heads(i, B, H, N, d, causal, kv):
    """Grids of hundreds of heads (several head groups, many work items per
    persistent backward CTA, non-causal last waves split), on a seeded sample
    of (b, h) slices."""
    import torch
    w = synth.small(f"fuzz heads {i}", B, H, N, d, causal, 99000 + i, kv_len_range=kv, backward=True)
    inp = pu.Inputs(w, with_do=True)
    o, lse = binding.attention_forward(inp.q, inp.k, inp.v, w.scale, w.causal, inp.kv_dev)
    dq, dk, dv = binding.attention_backward(inp.q, inp.k, inp.v, o, lse, inp.do, w.scale, w.causal, inp.kv_dev)
    torch.cuda.synchronize()
    assert binding.fa_check_status() == binding.FA_OK
    o, lse = pu.bf16_tensor_to_f64(o), lse.cpu().numpy().astype(np.float64)
    dq, dk, dv = (pu.bf16_tensor_to_f64(t) for t in (dq, dk, dv))
    rng = np.random.default_rng(1000 + i)
    picks = {(B - 1, H - 1), (0, 0)} | {(int(rng.integers(0, B)), int(rng.integers(0, H))) for _ in range(6)}
    for b, h in sorted(picks):
        ro, rl = pu.oracle_fwd_slice(inp, b, h)
        assert pu.o_err(o[b, h], ro) <= pu.O_ATOL
        assert pu.max_abs(lse[b, h], rl) <= pu.LSE_ATOL
        ref = pu.oracle_bwd_slice(inp, b, h)
        for name, g, r in (("dQ", dq[b, h], ref[0]), ("dK", dk[b, h], ref[1]), ("dV", dv[b, h], ref[2])):
            assert _rel_err(g, r) <= pu.GRAD_RTOL, ((b, h), name, _rel_err(g, r))
