"""Seeded input generator: published SplitMix64 vector, bf16 rounding, recipes."""
import numpy as np
import pytest

from exact_io_aware_29_gb300 import synth


def test_splitmix64_published_vector():
    # First outputs of the public reference SplitMix64 seeded with 1234567.
    assert synth.splitmix64_sequential(1234567, 5) == [
        6457827717110365317, 3203168211198807973, 9817491932198370423,
        4593380528125082431, 16408922859458223821]


def test_stream_is_random_access():
    full = synth.splitmix64_stream(42, 3, 0, 1000)
    part = synth.splitmix64_stream(42, 3, 500, 100)
    np.testing.assert_array_equal(full[500:600], part)
    # stream 0 with seed s reproduces the sequential generator
    seq = synth.splitmix64_sequential(42, 10)
    np.testing.assert_array_equal(synth.splitmix64_stream(42, 0, 0, 10), np.array(seq, np.uint64))


def test_bf16_round_to_nearest_even():
    bits = np.array([0x3F800000, 0x3F808000, 0x3F818000, 0x3F80FFFF, 0xBF808001, 0x00000000],
                    dtype=np.uint32)
    got = synth.f32_to_bf16_bits(bits.view(np.float32))
    np.testing.assert_array_equal(got, np.array([0x3F80, 0x3F80, 0x3F82, 0x3F81, 0xBF81, 0x0000],
                                                dtype=np.uint16))
    x = np.random.default_rng(0).normal(size=10000).astype(np.float32)
    back = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(x))
    assert np.max(np.abs(back - x) / np.abs(x)) <= 2.0 ** -8  # unit roundoff of an 8-bit significand


def test_normals_moments():
    x = synth.normals(7, 0, 200000, sigma=4.0)
    assert abs(x.mean()) < 0.05
    assert abs(x.std() - 4.0) < 0.05


def test_workload_recipes():
    lens = synth.C4.kv_lens()
    assert lens.shape == (4,) and np.all((lens >= 1024) & (lens <= 4096))
    rows = synth.C5.rows(3)
    assert len(rows) == 512 and len(set(rows.tolist())) == 512
    assert rows.min() >= 0 and rows.max() < 65536
    assert synth.C1.visible_pairs() == 256 * 256
    assert synth.C2C.visible_pairs() == 4 * 16 * 2048 * 2049 // 2
    w = synth.small("t", 1, 1, 10, 4, True, 1, kv_len_range=(3, 3))
    # rows 0..2 see 1,2,3 keys; rows 3..9 see 3 keys
    assert w.visible_pairs() == 1 + 2 + 3 + 7 * 3


def test_bf16_tensor_deterministic():
    a = synth.bf16_normal_tensor(5, 1, (2, 3, 16, 8))
    b = synth.bf16_normal_tensor(5, 1, (2, 3, 16, 8))
    np.testing.assert_array_equal(a, b)
    assert a.dtype == np.uint16


def test_slice_draw_matches_full_tensor():
    w = synth.small("s", 2, 3, 40, 8, True, 99, q_sigma=4.0)
    full_q, full_k = w.q(), w.k()
    for b, h in ((0, 0), (1, 2), (0, 1)):
        np.testing.assert_array_equal(w.slice_bits(synth.STREAM_Q, b, h), full_q[b, h])
        np.testing.assert_array_equal(w.slice_bits(synth.STREAM_K, b, h), full_k[b, h])


def test_packed_workload_slices_and_pairs():
    w = synth.PackedWorkload("p", 5, 3, 8, True, 123, (1, 9))
    cu = w.cu_seqlens()
    assert cu[0] == 0 and np.all(np.diff(cu) >= 1) and np.all(np.diff(cu) <= 9)
    full = synth.bf16_normal_tensor(w.seed, synth.STREAM_K, (w.total, w.H, w.d))
    for b in range(w.n_seq):
        np.testing.assert_array_equal(w.seq_bits(synth.STREAM_K, b), full[cu[b]:cu[b + 1]])
    brute = sum(int(np.sum(np.arange(L)[:, None] >= np.arange(L)[None, :])) for L in np.diff(cu)) * w.H
    assert w.visible_pairs() == brute
    lens = synth.V1.lens()
    assert len(lens) == 16 and lens.min() >= 512 and lens.max() <= 8192


def test_decode_workload_pages():
    import oracle
    w = synth.DecodeWorkload("t", 3, 2, 8, 4, 321, (1, 13), spare_blocks=2)
    table, lens = w.block_table(), w.seq_lens()
    used = [int(table[b, t]) for b in range(w.B) for t in range(int(w.pages()[b]))]
    assert len(set(used)) == len(used) and all(0 <= x < w.n_blocks for x in used)
    pool = w.pool_bits(synth.STREAM_K)
    for b in range(w.B):   # reading the pages back through the table gives the sequence's draw
        np.testing.assert_array_equal(oracle.gather_pages(pool, table[b], int(lens[b]), w.block_size),
                                      w.seq_bits(synth.STREAM_K, b))
    lens1 = synth.D1.seq_lens()
    assert lens1.min() >= 1024 and lens1.max() <= 32768 and synth.D1.block_table().shape[0] == 16
