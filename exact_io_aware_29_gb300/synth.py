"""Seeded synthetic workloads for the attention path.

This module draws the inputs that both the CUDA path and the CPU oracle are
fed. It holds none of the attention arithmetic: only a counter-based random
generator, Box-Muller normals, round-to-nearest-even bf16 encoding and the
per-workload recipes (shapes, value distributions, key lengths, sampled rows).

Generator: SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014; constants as in Vigna's public reference
implementation). Draw ``i`` (0-based) of stream ``t`` under seed ``s`` is
``mix(s + (t * 2**40 + i + 1) * 0x9E3779B97F4A7C15)``, so any slice of any
tensor can be regenerated on its own.

Streams: 0 = Q, 1 = K, 2 = V, 3 = dO, 4 = key lengths, 5 = sampled rows.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
STREAM_STRIDE = 1 << 40

STREAM_Q, STREAM_K, STREAM_V, STREAM_DO, STREAM_KVLEN, STREAM_ROWS = range(6)


def splitmix64_mix(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output function on a uint64 array (wrapping arithmetic)."""
    z = z.astype(np.uint64, copy=True)
    with np.errstate(over="ignore"):
        z ^= z >> np.uint64(30)
        z *= _M1
        z ^= z >> np.uint64(27)
        z *= _M2
        z ^= z >> np.uint64(31)
    return z


def splitmix64_stream(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Draws ``start .. start+count-1`` of one stream, as uint64."""
    idx = np.arange(start + 1, start + 1 + count, dtype=np.uint64)
    idx += np.uint64(stream * STREAM_STRIDE)
    with np.errstate(over="ignore"):
        state = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + idx * GOLDEN
    return splitmix64_mix(state)


def splitmix64_sequential(seed: int, count: int) -> list[int]:
    """Plain sequential SplitMix64 (state advanced by the golden gamma before
    each output), for checking against the published test vector."""
    out = []
    s = seed & 0xFFFFFFFFFFFFFFFF
    for _ in range(count):
        s = (s + 0x9E3779B97F4A7C15) & 0xFFFFFFFFFFFFFFFF
        out.append(int(splitmix64_mix(np.array([s], dtype=np.uint64))[0]))
    return out


def uniform01(bits: np.ndarray) -> np.ndarray:
    """Top 53 bits -> double in (0, 1] (never 0, so log() is finite)."""
    return ((bits >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)


def normals(seed: int, stream: int, count: int, sigma: float = 1.0) -> np.ndarray:
    """``count`` N(0, sigma^2) doubles by Box-Muller over pairs of draws
    (draws 2i, 2i+1 give elements 2i = r cos t and 2i+1 = r sin t)."""
    return normals_slice(seed, stream, 0, count, sigma)


def normals_slice(seed: int, stream: int, start: int, count: int, sigma: float = 1.0) -> np.ndarray:
    """Elements ``start .. start+count-1`` of :func:`normals` (``start`` even)."""
    if start % 2:
        raise ValueError("start must be even (Box-Muller pairs)")
    npairs = (count + 1) // 2
    bits = splitmix64_stream(seed, stream, start, 2 * npairs)
    u1 = uniform01(bits[0::2])
    u2 = uniform01(bits[1::2])
    r = np.sqrt(-2.0 * np.log(u1))
    th = 2.0 * math.pi * u2
    out = np.empty(2 * npairs, dtype=np.float64)
    out[0::2] = r * np.cos(th)
    out[1::2] = r * np.sin(th)
    return out[:count] * sigma


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest, ties to even (finite input)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    with np.errstate(over="ignore"):
        return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> fp32 values (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> fp64 values (exact widening)."""
    return bf16_bits_to_f32(b).astype(np.float64)


def bf16_normal_tensor(seed: int, stream: int, shape, sigma: float = 1.0) -> np.ndarray:
    """Seeded N(0, sigma^2) tensor: fp64 draw -> fp32 -> bf16 (RNE); bit patterns."""
    n = int(np.prod(shape))
    x = normals(seed, stream, n, sigma).astype(np.float32)
    return f32_to_bf16_bits(x).reshape(shape)


def uniform_ints(seed: int, stream: int, count: int, lo: int, hi: int) -> np.ndarray:
    """``count`` integers uniform in [lo, hi] (inclusive)."""
    u = uniform01(splitmix64_stream(seed, stream, 0, count))  # (0, 1]
    span = hi - lo + 1
    v = np.floor((1.0 - u) * span).astype(np.int64)  # [0, span)
    return (lo + np.minimum(v, span - 1)).astype(np.int32)


def distinct_rows(seed: int, stream: int, count: int, n: int, salt: int = 0) -> np.ndarray:
    """``count`` distinct row indices uniform in [0, n), sorted."""
    count = min(count, n)
    chosen: list[int] = []
    seen = set()
    start = salt * (1 << 24)
    while len(chosen) < count:
        u = uniform01(splitmix64_stream(seed, stream, start, 4 * count))
        start += 4 * count
        for r in np.minimum(np.floor((1.0 - u) * n).astype(np.int64), n - 1):
            r = int(r)
            if r not in seen:
                seen.add(r)
                chosen.append(r)
                if len(chosen) == count:
                    break
    return np.array(sorted(chosen), dtype=np.int64)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One attention problem: shapes, mask, distributions and seed."""
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    seed: int
    q_sigma: float = 1.0
    kv_len_range: Optional[tuple[int, int]] = None
    backward: bool = False
    sample_rows: int = 0  # >0: parity on that many seeded rows per head

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def kv_lens(self) -> Optional[np.ndarray]:
        if self.kv_len_range is None:
            return None
        lo, hi = self.kv_len_range
        return uniform_ints(self.seed, STREAM_KVLEN, self.B, lo, hi)

    def q(self) -> np.ndarray:
        return bf16_normal_tensor(self.seed, STREAM_Q, (self.B, self.H, self.N, self.d), self.q_sigma)

    def k(self) -> np.ndarray:
        return bf16_normal_tensor(self.seed, STREAM_K, (self.B, self.H, self.N, self.d))

    def v(self) -> np.ndarray:
        return bf16_normal_tensor(self.seed, STREAM_V, (self.B, self.H, self.N, self.d))

    def do(self) -> np.ndarray:
        return bf16_normal_tensor(self.seed, STREAM_DO, (self.B, self.H, self.N, self.d))

    def slice_bits(self, stream: int, b: int, h: int) -> np.ndarray:
        """The [N, d] slice (b, h) of one input tensor, drawn on its own."""
        n = self.N * self.d
        sigma = self.q_sigma if stream == STREAM_Q else 1.0
        x = normals_slice(self.seed, stream, (b * self.H + h) * n, n, sigma).astype(np.float32)
        return f32_to_bf16_bits(x).reshape(self.N, self.d)

    def rows(self, head_index: int) -> np.ndarray:
        """Seeded distinct query rows for (flattened) head ``head_index``."""
        return distinct_rows(self.seed, STREAM_ROWS, self.sample_rows, self.N, salt=head_index)

    def visible_pairs(self) -> int:
        """Exact number of visible (query, key) pairs over the whole batch."""
        lens = self.kv_lens()
        total = 0
        for b in range(self.B):
            L = self.N if lens is None else int(min(lens[b], self.N))
            if self.causal:
                # rows r < L see r+1 keys; rows r >= L see L keys
                total += L * (L + 1) // 2 + (self.N - L) * L
            else:
                total += self.N * L
        return total * self.H


SEED_BASE = 0xFA000000

# The five workloads the path is specified and measured on.
C1 = Workload("C1 fwd B1 H1 N256 d64 non-causal", 1, 1, 256, 64, False, SEED_BASE + 0)
C2 = Workload("C2 fwd B4 H16 N2048 d64 non-causal", 4, 16, 2048, 64, False, SEED_BASE + 1)
C2C = Workload("C2 fwd B4 H16 N2048 d64 causal", 4, 16, 2048, 64, True, SEED_BASE + 1)
C3 = Workload("C3 fwd B2 H32 N8192 d128 causal q~N(0,16)", 2, 32, 8192, 128, True, SEED_BASE + 2,
              q_sigma=4.0, sample_rows=512)
C4 = Workload("C4 fwd+bwd B4 H16 N4096 d128 causal kv_lens U[1024,4096]", 4, 16, 4096, 128, True,
              SEED_BASE + 3, kv_len_range=(1024, 4096), backward=True)
C5 = Workload("C5 fwd B1 H8 N65536 d128 causal", 1, 8, 65536, 128, True, SEED_BASE + 4, sample_rows=512)

# Two more forward shapes from the pages' sweeps (head dim 128, 8 or 16
# heads): the longest causal context and a non-causal point.
L1 = Workload("L1 fwd B1 H8 N131072 d128 causal", 1, 8, 131072, 128, True, SEED_BASE + 8, sample_rows=128)
NC = Workload("NC fwd B2 H16 N8192 d128 non-causal", 2, 16, 8192, 128, False, SEED_BASE + 9, sample_rows=256)

WORKLOADS = {"C1": C1, "C2": C2, "C2C": C2C, "C3": C3, "C4": C4, "C5": C5, "L1": L1, "NC": NC}

# Forward-only workloads the benchmark times beside the forward + backward step.
FORWARD_SWEEP = ("C2", "C2C", "C3", "C5", "L1", "NC")


@dataclasses.dataclass(frozen=True)
class PackedWorkload:
    """Variable-length sequences packed as [total, H, d]: sequence b holds rows
    cu[b] .. cu[b+1]-1 of Q, K, V and dO (query and key lengths equal), with
    lengths uniform in ``len_range`` (inclusive)."""
    name: str
    n_seq: int
    H: int
    d: int
    causal: bool
    seed: int
    len_range: tuple[int, int]

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def lens(self) -> np.ndarray:
        lo, hi = self.len_range
        return uniform_ints(self.seed, STREAM_KVLEN, self.n_seq, lo, hi)

    def cu_seqlens(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.lens())]).astype(np.int32)

    @property
    def total(self) -> int:
        return int(self.cu_seqlens()[-1])

    def seq_bits(self, stream: int, b: int) -> np.ndarray:
        """Rows of sequence b ([L, H, d] bf16 bits) of the packed tensor drawn
        from ``stream``; the packed tensor is one draw in [total, H, d] order."""
        cu = self.cu_seqlens()
        per_row = self.H * self.d
        n = int(cu[b + 1] - cu[b])
        x = normals_slice(self.seed, stream, int(cu[b]) * per_row, n * per_row).astype(np.float32)
        return f32_to_bf16_bits(x).reshape(n, self.H, self.d)

    def visible_pairs(self) -> int:
        total = 0
        for L in self.lens():
            L = int(L)
            total += L * (L + 1) // 2 if self.causal else L * L
        return total * self.H


@dataclasses.dataclass(frozen=True)
class DecodeWorkload:
    """One decoding step over a paged KV cache: query [B, H, d]; sequence b's
    cache (``seq_len[b]`` tokens, lengths uniform in ``len_range``) is one
    contiguous draw in [token, H, d] order per sequence (as in a packed batch),
    cut into pages of ``block_size`` tokens scattered over a pool of
    ``n_blocks`` physical blocks by a seeded permutation."""
    name: str
    B: int
    H: int
    d: int
    block_size: int
    seed: int
    len_range: tuple[int, int]
    spare_blocks: int = 8

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def seq_lens(self) -> np.ndarray:
        lo, hi = self.len_range
        return uniform_ints(self.seed, STREAM_KVLEN, self.B, lo, hi)

    def cu_seqlens(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.seq_lens())]).astype(np.int64)

    def pages(self) -> np.ndarray:
        return -(-self.seq_lens().astype(np.int64) // self.block_size)

    @property
    def n_blocks(self) -> int:
        return int(self.pages().sum()) + self.spare_blocks

    @property
    def max_blocks(self) -> int:
        return int(self.pages().max())

    def block_table(self) -> np.ndarray:
        """int32 [B, max_blocks]; entries past a sequence's pages are 0."""
        order = np.argsort(splitmix64_stream(self.seed, STREAM_ROWS, 0, self.n_blocks), kind="stable")
        table = np.zeros((self.B, self.max_blocks), dtype=np.int32)
        at = 0
        for b, n in enumerate(self.pages()):
            table[b, :n] = order[at:at + n]
            at += int(n)
        return table

    def q(self) -> np.ndarray:
        return bf16_normal_tensor(self.seed, STREAM_Q, (self.B, self.H, self.d))

    def seq_bits(self, stream: int, b: int) -> np.ndarray:
        """Cache rows of sequence b ([L, H, d] bf16 bits) drawn from ``stream``."""
        cu = self.cu_seqlens()
        per_row = self.H * self.d
        n = int(cu[b + 1] - cu[b])
        x = normals_slice(self.seed, stream, int(cu[b]) * per_row, n * per_row).astype(np.float32)
        return f32_to_bf16_bits(x).reshape(n, self.H, self.d)

    def pool_bits(self, stream: int) -> np.ndarray:
        """The whole pool [n_blocks, block_size, H, d] (small workloads only);
        slots no sequence owns hold 0."""
        pool = np.zeros((self.n_blocks, self.block_size, self.H, self.d), dtype=np.uint16)
        table = self.block_table()
        for b, L in enumerate(self.seq_lens()):
            rows = self.seq_bits(stream, b)
            for t in range(int(self.pages()[b])):
                seg = rows[t * self.block_size:(t + 1) * self.block_size]
                pool[table[b, t], :len(seg)] = seg
        return pool

    def cache_bytes(self) -> int:
        """K and V bytes one decoding step must read (bf16)."""
        return int(self.seq_lens().sum()) * self.H * self.d * 2 * 2


# One decoding step: 16 sequences with 1K..32K cached tokens, 16 heads of 128,
# pages of 512 tokens.
D1 = DecodeWorkload("D1 decode B16 H16 d128 paged bs512 L~U[1024,32768]", 16, 16, 128, 512, SEED_BASE + 6,
                    (1024, 32768))
# A smaller decoding step for profiler captures (its cache, ~0.4 GB, is still
# larger than the L2).
D_SMALL = DecodeWorkload("decode B4 H16 d128 paged bs512 L~U[8192,16384]", 4, 16, 128, 512, SEED_BASE + 7,
                         (8192, 16384))


# Packed training batch: 16 sequences of 512..8192 tokens, 16 heads of 128.
V1 = PackedWorkload("V1 fwd+bwd packed 16 seqs L~U[512,8192] H16 d128 causal", 16, 16, 128, True,
                    SEED_BASE + 5, (512, 8192))


def small(name: str, B: int, H: int, N: int, d: int, causal: bool, seed: int,
          kv_len_range=None, backward=False, q_sigma=1.0) -> Workload:
    """A reduced workload for parity tests the oracle finishes in seconds."""
    return Workload(name, B, H, N, d, causal, seed, q_sigma=q_sigma,
                    kv_len_range=kv_len_range, backward=backward)
