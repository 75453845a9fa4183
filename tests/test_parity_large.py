"""GPU parity on tensors of more than 2^31 elements (2^32 bytes of bf16): every
offset past that point must be formed in 64 bits, in the kernels' stores, the
tensor maps, the backward's workspace and the FP8 codes.

A few seeded source slices are repeated over thousands of heads (fixed
layout) or over a packed batch of about a million tokens, on the device. The
slices on both sides of the 2^31-element boundary, and the last one, are
compared with the fp64 oracle of their source. The number of distinct sources
is odd, so an offset that wrapped at 2^31 or 2^32 bytes would read another
source's values (in the fixed layout both are whole, even numbers of slices;
in the packed batch they fall inside sequences)."""
import numpy as np
import pytest

import oracle
from oracle import fp8 as ofp8
from exact_io_aware_29_gb300 import binding, build, synth
import parity_util as pu
from test_parity_fp8 import _check_rows

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

S = 5            # distinct source slices
N, D = 1024, 128
LIMIT = 2 ** 31  # elements


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.load_library()
    yield
    import torch
    torch.cuda.empty_cache()


def rel_err(g, r):
    return pu.max_abs(g, r) / max(float(np.max(np.abs(r))), pu.ZERO_REF_FLOOR)


def sources(name, seed):
    """S seeded [N, d] slices of Q, K, V, dO (bit patterns)."""
    w = synth.small(name, 1, S, N, D, True, seed, backward=True)
    return {n: getattr(w, n)()[0] for n in ("q", "k", "v", "do")}, w.scale


def test_fixed_layout_beyond_2e31_elements():
    """B4 H4250 N1024 d128 causal (2.23e9 elements per tensor), key lengths
    per batch entry: forward, backward and FP8 forward."""
    import torch
    B, H = 4, 4250
    BH = B * H
    assert BH * N * D > LIMIT
    kv = [N, 777, 1000, 513]
    src, scale = sources("beyond 2^31, fixed layout", 7201)
    idx = torch.arange(BH, device="cuda") % S
    dev = {n: pu.to_device(b).index_select(0, idx).view(B, H, N, D) for n, b in src.items()}
    kv_dev = torch.tensor(kv, dtype=torch.int32, device="cuda")
    first = LIMIT // (N * D)  # first slice at or past 2^31 elements (2^32 bytes)
    half = first // 2         # first slice at or past 2^31 bytes
    check = [0, half - 1, half, first - 1, first, first + 1, BH - 1]
    f64 = {n: synth.bf16_bits_to_f64(b) for n, b in src.items()}

    o, lse = binding.attention_forward(dev["q"], dev["k"], dev["v"], scale, True, kv_dev)
    dq, dk, dv = binding.attention_backward(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], scale, True, kv_dev)
    torch.cuda.synchronize()
    assert binding.fa_check_status() == binding.FA_OK
    for bh in check:
        b, h, s = bh // H, bh % H, bh % S
        ro, rl = oracle.attention_forward(f64["q"][s], f64["k"][s], f64["v"][s], scale, True, kv[b])
        go = pu.bf16_tensor_to_f64(o[b, h])
        assert np.all(np.isfinite(go))
        assert pu.o_err(go, ro) <= pu.O_ATOL, bh
        assert pu.max_abs(lse[b, h].cpu().numpy(), rl) <= pu.LSE_ATOL, bh
        ref = oracle.attention_backward(f64["q"][s], f64["k"][s], f64["v"][s], f64["do"][s], scale, True, kv[b])
        for g, r in zip((dq[b, h], dk[b, h], dv[b, h]), ref):
            g = pu.bf16_tensor_to_f64(g)
            assert np.all(np.isfinite(g))
            assert rel_err(g, r) <= pu.GRAD_RTOL, bh
    del dq, dk, dv, o, lse
    torch.cuda.empty_cache()

    # FP8: 8-bit codes past 2^31 bytes, V^T's padded rows, the forward's stores.
    o, lse, (q8, sq, k8, sk, v8t, sv) = binding.attention_forward_fp8(dev["q"], dev["k"], dev["v"], scale, True,
                                                                      kv_dev)
    torch.cuda.synchronize()
    assert binding.fa_check_status() == binding.FA_OK
    for bh in (first - 1, first, BH - 1):
        b, h, s = bh // H, bh % H, bh % S
        rc, rs = ofp8.quantize_blocks(synth.bf16_bits_to_f32(src["k"][s])[None])
        np.testing.assert_array_equal(k8[b, h].cpu().numpy(), rc[0])
        np.testing.assert_array_equal(sk[b, h].cpu().numpy(), rs[0])
        rows = np.arange(0, N, 7)
        go = pu.bf16_tensor_to_f64(o[b, h])[rows]
        assert np.all(np.isfinite(go))
        _check_rows(go, lse[b, h].cpu().numpy()[rows], src["q"][s], src["k"][s], src["v"][s], scale, True, kv[b],
                    rows)


def test_packed_batch_beyond_2e31_elements():
    """1100 causal sequences of 960-1024 tokens, H16 d128 packed as
    [total, H, d] (about 1.09e6 tokens, 2.2e9 elements): forward and backward
    of the sequences that hold the rows at 2^31 bytes and 2^31 elements, the
    one before the latter, the first and the last."""
    import torch
    H, nseq = 16, 1100
    rng = np.random.default_rng(7202)
    lens = rng.integers(960, N + 1, nseq)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    total = int(cu[-1])
    assert total * H * D > LIMIT
    src, scale = sources("beyond 2^31, packed", 7203)
    # source slice s as [N, H, d]: head h of it is slice (s + h) % S
    per = {n: pu.to_device(b) for n, b in src.items()}
    heads = (torch.arange(S, device="cuda")[:, None] + torch.arange(H, device="cuda")[None, :]) % S
    thd = {n: t[heads].permute(0, 2, 1, 3).contiguous() for n, t in per.items()}  # [S, N, H, d]
    dev = {n: torch.cat([t[i % S, :int(lens[i])] for i in range(nseq)]) for n, t in thd.items()}
    del thd
    cu_dev = torch.tensor(cu, dtype=torch.int32, device="cuda")
    def holding(row):  # the sequence holding packed row `row`
        return int(np.searchsorted(cu, row, side="right")) - 1
    cross = holding(LIMIT // (H * D))      # 2^31 elements
    half = holding(LIMIT // (2 * H * D))   # 2^31 bytes
    check = [0, half, cross - 1, cross, nseq - 1]
    f64 = {n: synth.bf16_bits_to_f64(b) for n, b in src.items()}

    o, lse = binding.attention_forward_varlen(dev["q"], dev["k"], dev["v"], cu_dev, cu_dev, N, N, scale, True)
    dq, dk, dv = binding.attention_backward_varlen(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], cu_dev, cu_dev,
                                                   N, N, scale, True)
    torch.cuda.synchronize()
    assert binding.fa_check_status() == binding.FA_OK
    for i in check:
        a, L = int(cu[i]), int(lens[i])
        for h in (0, H - 1):
            s = (i % S + h) % S
            q, k, v, do = (f64[n][s][:L] for n in ("q", "k", "v", "do"))
            ro, rl = oracle.attention_forward(q, k, v, scale, True)
            go = pu.bf16_tensor_to_f64(o[a:a + L, h])
            assert np.all(np.isfinite(go))
            assert pu.o_err(go, ro) <= pu.O_ATOL, (i, h)
            assert pu.max_abs(lse[h, a:a + L].cpu().numpy(), rl) <= pu.LSE_ATOL, (i, h)
            ref = oracle.attention_backward(q, k, v, do, scale, True)
            for g, r in zip((dq[a:a + L, h], dk[a:a + L, h], dv[a:a + L, h]), ref):
                g = pu.bf16_tensor_to_f64(g)
                assert np.all(np.isfinite(g))
                assert rel_err(g, r) <= pu.GRAD_RTOL, (i, h)


def test_paged_decode_pool_beyond_2e31_elements():
    """A paged cache of 2100 pages of 512 tokens at H16 d128 (2.2e9 elements
    per pool): sequences on the pages at 2^31 bytes and at 2^31 elements, at
    the end of the pool and at its start. Every page no sequence owns holds
    NaN, so a read from a wrong page would show in O."""
    import torch
    H, bs, nb = 16, 512, 2100
    assert nb * bs * H * D > LIMIT
    page = bs * H * D
    p_el, p_by = LIMIT // page, LIMIT // (2 * page)
    lens = np.array([3000, 4097, 1, 2500], np.int32)
    pages = [list(range(nb - 6, nb)), list(range(p_el - 4, p_el + 5)), [0], list(range(p_by - 2, p_by + 3))]
    used = sorted({x for p in pages for x in p})
    at = {x: i for i, x in enumerate(used)}
    table = np.zeros((len(lens), max(len(p) for p in pages)), np.int32)
    compact = np.zeros_like(table)  # the same table over the owned pages only, for the oracle
    for b, p in enumerate(pages):
        assert len(p) == -(-int(lens[b]) // bs)
        table[b, :len(p)] = p
        compact[b, :len(p)] = [at[x] for x in p]
    kc = synth.bf16_normal_tensor(7204, synth.STREAM_K, (len(used), bs, H, D))
    vc = synth.bf16_normal_tensor(7204, synth.STREAM_V, (len(used), bs, H, D))
    q = synth.bf16_normal_tensor(7204, synth.STREAM_Q, (len(lens), H, D))
    owned = torch.tensor(used, device="cuda")
    pools = []
    for bits in (kc, vc):
        p = torch.full((nb, bs, H, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        p[owned] = pu.to_device(bits)
        pools.append(p)
    scale = D ** -0.5
    o, lse = binding.attention_decode_paged(pu.to_device(q), pools[0], pools[1],
                                            torch.from_numpy(table).cuda(), torch.from_numpy(lens).cuda(),
                                            int(lens.max()), scale)
    torch.cuda.synchronize()
    assert binding.fa_check_status() == binding.FA_OK
    ro, rl = oracle.paged_decode_forward(synth.bf16_bits_to_f64(q), synth.bf16_bits_to_f64(kc),
                                         synth.bf16_bits_to_f64(vc), compact, lens, scale)
    go = pu.bf16_tensor_to_f64(o)
    assert np.all(np.isfinite(go))
    assert pu.o_err(go, ro) <= pu.O_ATOL
    assert pu.max_abs(lse.cpu().numpy(), rl) <= pu.LSE_ATOL
