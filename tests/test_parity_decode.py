"""GPU parity of decoding from a paged KV cache (fa_decode_paged) against the
fp64 oracle: pages scattered over the pool by a seeded permutation, lengths
at and around page and tile edges (including empty sequences), one CTA per
head and many splits per head, and the decode workload at full size."""
import numpy as np
import pytest

import oracle
from exact_io_aware_29_gb300 import binding, build, synth
import parity_util as pu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.load_library()


def run(w, lens=None, table=None):
    import torch
    lens = w.seq_lens() if lens is None else np.asarray(lens, np.int32)
    table = w.block_table() if table is None else table
    q_bits = w.q()
    kp, vp = w.pool_bits(synth.STREAM_K), w.pool_bits(synth.STREAM_V)
    q, k, v = pu.to_device(q_bits), pu.to_device(kp), pu.to_device(vp)
    t = torch.from_numpy(np.ascontiguousarray(table, dtype=np.int32)).cuda()
    L = torch.from_numpy(np.asarray(lens, np.int32)).cuda()
    max_len = max(int(np.max(lens)), 1)
    o, lse = binding.attention_decode_paged(q, k, v, t, L, max_len, w.scale)
    torch.cuda.synchronize()
    assert binding.fa_check_status() == binding.FA_OK
    ro, rl = oracle.paged_decode_forward(synth.bf16_bits_to_f64(q_bits), synth.bf16_bits_to_f64(kp),
                                         synth.bf16_bits_to_f64(vp), table, lens, w.scale)
    go = pu.bf16_tensor_to_f64(o)
    assert np.all(np.isfinite(go))
    assert pu.o_err(go, ro) <= pu.O_ATOL
    assert pu.max_abs(lse.cpu().numpy(), rl) <= pu.LSE_ATOL
    return go, lse


CASES = [
    # (B, H, d, block_size, len_range)
    (3, 2, 128, 64, (1, 700)),
    (4, 3, 128, 512, (1000, 3000)),
    (2, 2, 64, 128, (60, 200)),
    (5, 1, 64, 64, (1, 129)),
    (2, 4, 128, 256, (4000, 9000)),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_decode_against_oracle(case):
    B, H, d, bs, rng = CASES[case]
    w = synth.DecodeWorkload(f"dec{case}", B, H, d, bs, 8800 + case, rng, spare_blocks=3)
    run(w)


@pytest.mark.parametrize("d", [64, 128])
def test_decode_edge_lengths(d):
    # empty, one key, one tile, tile +- 1, page +- 1
    lens = [0, 1, 63, 64, 65, 127, 128, 129, 255, 256, 257]
    w = synth.DecodeWorkload("edges", len(lens), 2, d, 128, 8900 + d, (257, 257), spare_blocks=2)
    # the workload's own draw sets the pool up for 257 tokens per sequence; the
    # kernel and the oracle read only the first lens[b] of them
    go, lse = run(w, lens=lens)
    assert np.all(go[0] == 0) and np.all(lse.cpu().numpy()[0] == -np.inf)


def test_decode_many_splits_per_head():
    # one head: about 1024 CTAs wanted, so every 64-key tile gets its own CTA
    w = synth.DecodeWorkload("splits", 1, 1, 128, 64, 8950, (5000, 5000))
    run(w)


def test_decode_block_ids_outside_the_pool_read_as_zeros():
    import torch
    w = synth.DecodeWorkload("oob", 2, 2, 128, 64, 8960, (300, 300), spare_blocks=0)
    table = w.block_table().copy()
    table[1, 2] = w.n_blocks + 5           # page 2 of sequence 1 points past the pool
    table[0, 1] = -3                       # page 1 of sequence 0 is negative
    kp, vp = w.pool_bits(synth.STREAM_K), w.pool_bits(synth.STREAM_V)
    zk, zv = kp.copy(), vp.copy()
    # the oracle sees a pool with an extra all-zero block at the end
    zero = np.zeros((1,) + kp.shape[1:], kp.dtype)
    zk, zv = np.concatenate([zk, zero]), np.concatenate([zv, zero])
    otab = np.where((table < 0) | (table >= w.n_blocks), w.n_blocks, table)
    q = pu.to_device(w.q())
    o, lse = binding.attention_decode_paged(q, pu.to_device(kp), pu.to_device(vp),
                                            torch.from_numpy(table.astype(np.int32)).cuda(),
                                            torch.from_numpy(w.seq_lens()).cuda(), 300, w.scale)
    torch.cuda.synchronize()
    ro, rl = oracle.paged_decode_forward(synth.bf16_bits_to_f64(w.q()), synth.bf16_bits_to_f64(zk),
                                         synth.bf16_bits_to_f64(zv), otab, w.seq_lens(), w.scale)
    assert pu.o_err(pu.bf16_tensor_to_f64(o), ro) <= pu.O_ATOL
    assert pu.max_abs(lse.cpu().numpy(), rl) <= pu.LSE_ATOL


def test_d1_full_size_sampled():
    """The decode workload at full size (16 sequences of 1K..32K cached tokens,
    16 heads, d = 128, pages of 512) in the benchmark's launch configuration:
    three sequences (shortest, a middle one, longest) carry their seeded cache
    and are checked on every head; the rest of the pool holds device random
    values."""
    import torch
    w = synth.D1
    lens = w.seq_lens()
    table = w.block_table()
    order = np.argsort(lens)
    checked = [int(order[0]), int(order[len(order) // 2]), int(order[-1])]
    g = torch.Generator(device="cuda")
    g.manual_seed(9)
    shape = (w.n_blocks, w.block_size, w.H, w.d)
    kp = torch.randn(shape, device="cuda", generator=g).to(torch.bfloat16)
    vp = torch.randn(shape, device="cuda", generator=g).to(torch.bfloat16)
    logical = {}
    for b in checked:
        for name, pool, st in (("k", kp, synth.STREAM_K), ("v", vp, synth.STREAM_V)):
            rows = w.seq_bits(st, b)
            logical[(name, b)] = synth.bf16_bits_to_f64(rows)
            dev = pu.to_device(rows)
            for t in range(int(w.pages()[b])):
                seg = dev[t * w.block_size:(t + 1) * w.block_size]
                pool[int(table[b, t]), :seg.shape[0]] = seg
    q_bits = w.q()
    o, lse = binding.attention_decode_paged(pu.to_device(q_bits), kp, vp, torch.from_numpy(table).cuda(),
                                            torch.from_numpy(lens).cuda(), int(lens.max()), w.scale)
    torch.cuda.synchronize()
    assert binding.fa_check_status() == binding.FA_OK
    go, gl = pu.bf16_tensor_to_f64(o), lse.cpu().numpy()
    qf = synth.bf16_bits_to_f64(q_bits)
    for b in checked:
        for h in range(w.H):
            ro, rl = oracle.attention_forward(qf[b, h][None], logical[("k", b)][:, h], logical[("v", b)][:, h],
                                              w.scale)
            assert pu.o_err(go[b, h], ro[0]) <= pu.O_ATOL, (b, h)
            assert abs(gl[b, h] - rl[0]) <= pu.LSE_ATOL, (b, h)
