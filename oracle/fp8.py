"""FP8 (E4M3) block quantisation and the FP8 attention forward, in plain numpy.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

Sources: youngju.dev "flash_attention.zh" §9.2 (FP8 with block quantisation:
every block keeps its own scale factor to preserve dynamic range);
"FlashAttention 完整解析" §5.5 (E4M3 inputs, range +-448; scaling before the
softmax products to avoid underflow).

Readings taken where the pages leave the step open:
  * A block is 128 consecutive rows (tokens) of one (batch, head) slice of Q, K
    or V, all d columns. Its scale is s = amax / 448 (fp32) and each value is
    coded as e4m3(x * (448 / amax)) with the fp32 product rounded to nearest
    even and saturated to +-448 (the E4M3 "fn" format: no infinities, 448 the
    largest finite value). An all-zero block has s = 0 and codes 0.
  * The FP8 forward computes the attention of the dequantised inputs
    (code * s): that is the oracle's result. The kernel additionally rounds the
    probabilities to e4m3 before the P.V product; the oracle bounds the effect
    of that rounding instead of reproducing it (it depends on the kernel's
    running maximum): see p_rounding_bounds.
"""
from __future__ import annotations

import numpy as np

from .attention import attention_forward

E4M3_MAX = 448.0
BLOCK = 128


# ----------------------------------------------------------------------------
# The E4M3 format: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits;
# exponent field 0 holds subnormals m/8 * 2^-6; code 0x7F / 0xFF is NaN.
# ----------------------------------------------------------------------------
def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """uint8 codes -> fp64 values (NaN for the two NaN codes)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return sign * val


def e4m3_round(y: np.ndarray) -> np.ndarray:
    """Round fp64 values (here: exact fp32 values) to the nearest E4M3 value,
    ties to even, saturating at +-448."""
    y = np.asarray(y, dtype=np.float64)
    a = np.abs(y)
    _, e = np.frexp(a)                       # a = f * 2^e with f in [0.5, 1)
    E = np.maximum(e - 1, -6)                # binade exponent; subnormals share 2^-6's quantum
    quantum = np.ldexp(1.0, E - 3)           # 3 mantissa bits
    r = np.round(a / quantum) * quantum      # a / quantum is exact; np.round ties to even
    r = np.minimum(r, E4M3_MAX)
    return np.copysign(r, y)


def e4m3_encode(values: np.ndarray) -> np.ndarray:
    """Exactly representable E4M3 values -> uint8 codes. The format has two
    zeros: -0 (a negative value rounded to zero keeps its sign) is 0x80."""
    v = np.asarray(values, dtype=np.float64)
    a = np.abs(v)
    sign = np.where(np.signbit(v), 0x80, 0)
    _, e = np.frexp(a)
    E = e - 1
    sub = a < 2.0 ** -6
    mant_sub = np.round(a / 2.0 ** -9).astype(np.int64)
    Es = np.where(sub, 0, E)
    frac = np.where(sub, 0.0, a / np.ldexp(1.0, Es) - 1.0)
    mant_norm = np.round(frac * 8).astype(np.int64)
    field_e = np.where(sub, 0, Es + 7)
    mant = np.where(sub, mant_sub, mant_norm)
    code = np.where(a == 0, 0, (field_e << 3) | mant)
    return (code | sign).astype(np.uint8)


# ----------------------------------------------------------------------------
# Block quantisation ([P2] §9.2): one scale per 128 rows of a (batch, head)
# slice, computed and applied in fp32 as stated in the module docstring.
# ----------------------------------------------------------------------------
def quantize_blocks(x: np.ndarray, block: int = BLOCK):
    """x: [S, N, d] (fp32-representable values, e.g. bf16 widened). Returns
    codes uint8 [S, N, d] and scales fp32 [S, ceil(N / block)]."""
    x = np.asarray(x, dtype=np.float32)
    S, N, d = x.shape
    nb = -(-N // block)
    codes = np.zeros((S, N, d), dtype=np.uint8)
    scales = np.zeros((S, nb), dtype=np.float32)
    for s in range(S):
        for i in range(nb):
            blk = x[s, i * block:(i + 1) * block]
            amax = np.float32(np.max(np.abs(blk))) if blk.size else np.float32(0)
            if amax == 0:
                continue
            inv = np.float32(E4M3_MAX) / amax                    # fp32 division, round to nearest
            scales[s, i] = amax / np.float32(E4M3_MAX)
            y = (blk * inv).astype(np.float32)                   # fp32 products, round to nearest
            codes[s, i * block:(i + 1) * block] = e4m3_encode(e4m3_round(y.astype(np.float64)))
    return codes, scales


def dequantize_blocks(codes: np.ndarray, scales: np.ndarray, block: int = BLOCK) -> np.ndarray:
    """codes [S, N, d], scales [S, nb] -> fp64 values code * scale."""
    vals = e4m3_decode(codes)
    rows = np.arange(codes.shape[1]) // block
    return vals * np.asarray(scales, np.float64)[:, rows][:, :, None]


def fp8_attention_forward(q_codes, q_scales, k_codes, k_scales, v_codes, v_scales, scale, causal=False,
                          kv_len=None, rows=None):
    """One (batch, head) slice ([N, d] codes, [nb] scales): attention of the
    dequantised inputs. Returns O [N, d], LSE [N] (the query rows ``rows``
    only, when given)."""
    from .attention import attention_forward_rows
    q = dequantize_blocks(q_codes[None], q_scales[None])[0]
    k = dequantize_blocks(k_codes[None], k_scales[None])[0]
    v = dequantize_blocks(v_codes[None], v_scales[None])[0]
    if rows is not None:
        return attention_forward_rows(q, k, v, rows, scale, causal, kv_len)
    return attention_forward(q, k, v, scale, causal, kv_len)


# ----------------------------------------------------------------------------
# What rounding P to e4m3 can do to O. The kernel feeds the P.V product with
# P'_j = e4m3(p_j * 2^7 * sV_b(j) / max_b sV_b), where p_j = 2^(x_j - m) <= 2^1.75
# is taken against its running maximum m (at most 1.75 binades below the row
# maximum, so P' stays below 2^8.75 < 448 and never saturates), and divides by
# l = sum_j p_j (unrounded) at the end. Neither term below depends on that
# threshold. For a P' in
# E4M3's normal range the rounding error is at most 2^-4 of it; below 2^-6 it
# is at most 2^-10 absolute, i.e. at most 2^-17 * max sV / sV_b(j) in units of
# p, and l >= 1. In units of the normalised probabilities P_rj = p_j / l:
#   |dO_rc| <= sum_j (2^-4 P_rj + 2^-17 max sV / sV_b(j)) |V_jc|       (bound)
# and, taking the roundings as independent and uniform over their interval,
#   E[dO_rc^2] <= sum_j ((2^-4)^2 / 3) P_rj^2 V_jc^2 + (subnormal terms),
# which gives the root-mean-square bound used by the tests.
# ----------------------------------------------------------------------------
def p_rounding_bounds(q_codes, q_scales, k_codes, k_scales, v_codes, v_scales, scale, causal=False,
                      kv_len=None, rows=None):
    """Per-element worst-case bound [N, d] and per-element variance bound
    [N, d] of the error the e4m3 rounding of P adds to O (see above); for the
    query rows ``rows`` only when given."""
    from .attention import NEG_INF, logits, safe_softmax, visible_rows
    q = dequantize_blocks(q_codes[None], q_scales[None])[0]
    k = dequantize_blocks(k_codes[None], k_scales[None])[0]
    v = dequantize_blocks(v_codes[None], v_scales[None])[0]
    rows = np.arange(q.shape[0]) if rows is None else np.asarray(rows)
    s = logits(q[rows], k, scale)
    s = np.where(visible_rows(rows, k.shape[0], causal, kv_len), s, NEG_INF)
    p, _, _ = safe_softmax(s)                                   # normalised, [rows, Nk]
    sv = np.asarray(v_scales, np.float64)
    smax = float(np.max(sv)) if sv.size else 0.0
    blk = np.arange(k.shape[0]) // BLOCK
    with np.errstate(divide="ignore"):
        sub = np.where(sv[blk] > 0, 2.0 ** -17 * smax / sv[blk], 0.0)   # [Nk]
    av = np.abs(v)
    bound = 2.0 ** -4 * (p @ av) + (p > 0).astype(np.float64) @ (sub[:, None] * av)
    var = (2.0 ** -8 / 3.0) * ((p * p) @ (av * av)) + (p > 0).astype(np.float64) @ ((sub[:, None] * av) ** 2 / 3.0)
    return bound, var
