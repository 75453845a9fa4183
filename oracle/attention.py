"""Plain fp64 CPU oracle for exact scaled dot-product attention.

TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this module. It shares no code with the CUDA path
and imports nothing from it.

Sources (the three pages on IO-aware exact attention):
  [P1] "FlashAttention算法详解：从IO瓶颈到Triton实现" (gentlecold.top):
       §先说结论 (the definition O = softmax(QK^T/sqrt(d) + M) V),
       §Online Softmax, §一个小数值例子 (worked example), §FlashAttention Forward流程
       (the forward loop), §Causal Mask怎么处理, §Backward为什么更复杂 (gradient
       formulas and LSE = m + log l).
  [P2] youngju.dev "flash_attention.zh": §6.1-6.3 (safe softmax, online merge,
       rescaling property), §7.2 (recompute from saved statistics).
  [P3] "FlashAttention 完整解析：从原理到 CUDA/Triton 实现" (blog.freezetheflame.cc):
       §1.1 (the definition), §2.3 (online merge), §7.2-7.4 (KV cache pages
       addressed through a block table).

What is computed is the definition, written out: logits are materialised in
fp64, the mask is applied, a two-pass safe softmax forms P, O = P V and
LSE = m + ln l. Inputs are bf16 values widened exactly to fp64. The blocked
online-softmax routines below follow the pages' algorithm step by step; they
exist so the tests can show that the algorithm the kernels run reaches the
definition for every block split.

Readings taken where the pages are silent:
  * The mask M is -inf where (causal and c > r + offset) or c >= kv_len
    (keys only). offset = 0 (top-left alignment) for the fixed-length layout;
    for packed variable-length sequences with n_q queries and n_k keys it is
    n_k - n_q, so the last query sees every key (bottom-right alignment).
  * A row with no visible key has O = 0 and LSE = -inf; it contributes nothing
    to the backward.
  * LSE is in natural-log units of the scaled logits S = scale * Q K^T.
  * dS is the gradient with respect to the scaled logits, so dQ and dK carry
    the factor ``scale`` (chain rule).
  * Decoding from a paged KV cache: the one new query of a sequence comes
    after its L cached tokens (its own K/V already appended), so it sees all
    L keys; token t lives in slot t mod block_size of physical block
    block_table[b][t // block_size].
"""
from __future__ import annotations

import numpy as np

NEG_INF = -np.inf


# ----------------------------------------------------------------------------
# Mask  ([P1] §Causal Mask怎么处理; key padding per the forward loop's
# "apply mask if causal or padding")
# ----------------------------------------------------------------------------
def visible(n_q: int, n_k: int, causal: bool, kv_len: int | None, offset: int = 0) -> np.ndarray:
    """Boolean [n_q, n_k]: True where key c is visible to query r."""
    r = np.arange(n_q)[:, None]
    c = np.arange(n_k)[None, :]
    vis = np.ones((n_q, n_k), dtype=bool)
    if causal:
        vis &= c <= r + offset
    if kv_len is not None:
        vis &= c < kv_len
    return vis


def visible_rows(rows: np.ndarray, n_k: int, causal: bool, kv_len: int | None, offset: int = 0) -> np.ndarray:
    """Same as :func:`visible`, for a subset of query rows."""
    r = np.asarray(rows)[:, None]
    c = np.arange(n_k)[None, :]
    vis = np.ones((len(rows), n_k), dtype=bool)
    if causal:
        vis &= c <= r + offset
    if kv_len is not None:
        vis &= c < kv_len
    return vis


# ----------------------------------------------------------------------------
# Safe softmax of a materialised logit matrix ([P2] §6.1; [P1] §Online Softmax
# first three equations)
# ----------------------------------------------------------------------------
def row_max(s: np.ndarray) -> np.ndarray:
    """m_r = max_c S_rc (−inf for an all-masked row or a row with no keys)."""
    if s.shape[-1] == 0:
        return np.full(s.shape[:-1], NEG_INF)
    return np.max(s, axis=-1)


def safe_softmax(s: np.ndarray):
    """Returns (P, m, l) with m = rowmax, l = sum exp(S - m), P = exp(S - m)/l.

    Rows that are entirely -inf give P = 0, m = -inf, l = 0.
    """
    m = row_max(s)
    empty = ~np.isfinite(m)
    m_safe = np.where(empty, 0.0, m)
    e = np.exp(s - m_safe[..., None])          # exp(-inf) = 0 on masked entries
    l = np.sum(e, axis=-1)
    l_safe = np.where(empty, 1.0, l)
    p = e / l_safe[..., None]
    p[empty] = 0.0
    return p, m, l


def logits(q: np.ndarray, k: np.ndarray, scale: float) -> np.ndarray:
    """S = scale * Q K^T (fp64; the matmul is a library primitive)."""
    return scale * (q @ k.T)


# ----------------------------------------------------------------------------
# Forward: the definition ([P1] §先说结论; [P3] §1.1; LSE per [P1] §Backward)
# ----------------------------------------------------------------------------
def attention_forward(q, k, v, scale, causal=False, kv_len=None, offset=0):
    """One (batch, head) slice. q: [n_q, d], k, v: [n_k, d] fp64.
    Returns (O [n_q, d], LSE [n_q])."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    s = logits(q, k, scale)
    s = np.where(visible(q.shape[0], k.shape[0], causal, kv_len, offset), s, NEG_INF)
    p, m, l = safe_softmax(s)
    o = p @ v
    with np.errstate(divide="ignore"):
        lse = np.where(l > 0, m + np.log(np.where(l > 0, l, 1.0)), NEG_INF)
    return o, lse


def attention_forward_rows(q, k, v, rows, scale, causal=False, kv_len=None, offset=0):
    """Definition evaluated for selected query rows only. Returns (O[rows], LSE[rows])."""
    rows = np.asarray(rows)
    q = np.asarray(q, dtype=np.float64)[rows]
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    s = logits(q, k, scale)
    s = np.where(visible_rows(rows, k.shape[0], causal, kv_len, offset), s, NEG_INF)
    p, m, l = safe_softmax(s)
    o = p @ v
    with np.errstate(divide="ignore"):
        lse = np.where(l > 0, m + np.log(np.where(l > 0, l, 1.0)), NEG_INF)
    return o, lse


def probabilities(q, k, scale, causal=False, kv_len=None, offset=0):
    """Materialised P for one slice (used by the backward and by invariant tests)."""
    s = logits(np.asarray(q, np.float64), np.asarray(k, np.float64), scale)
    s = np.where(visible(s.shape[0], s.shape[1], causal, kv_len, offset), s, NEG_INF)
    p, _, _ = safe_softmax(s)
    return p


# ----------------------------------------------------------------------------
# Backward: the gradient formulas of [P1] §Backward为什么更复杂, with the scale
# made explicit (dS is taken w.r.t. the scaled logits).
# ----------------------------------------------------------------------------
def softmax_grad(p: np.ndarray, dp: np.ndarray) -> np.ndarray:
    """dS = P ∘ (dP − rowsum(dP ∘ P))."""
    return p * (dp - np.sum(dp * p, axis=-1, keepdims=True))


def attention_backward(q, k, v, do, scale, causal=False, kv_len=None, offset=0, o_stored=None):
    """One slice. Returns (dQ, dK, dV) of L = sum(O ∘ dO).

    By default the row term of dS is rowsum(dP ∘ P), from the materialised P.
    With ``o_stored`` (the forward's output as stored, e.g. rounded to bf16)
    it is D = rowsum(dO ∘ O) of that O, the form the method's backward uses
    ([P1] §Backward为什么更复杂: the row term equals rowsum(dO ∘ O) because O = P V);
    with the exact O both give the same dS."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    p = probabilities(q, k, scale, causal, kv_len, offset)
    dv = p.T @ do                      # dV = P^T dO
    dp = do @ v.T                      # dP = dO V^T
    if o_stored is None:
        ds = softmax_grad(p, dp)       # dS = P ∘ (dP − rowsum(dP ∘ P))
    else:                              # dS = P ∘ (dP − rowsum(dO ∘ O_stored))
        ds = p * (dp - np.sum(do * np.asarray(o_stored, dtype=np.float64), axis=-1, keepdims=True))
    dq = scale * (ds @ k)              # dQ = dS K   (times d(S)/d(QK^T) = scale)
    dk = scale * (ds.T @ q)            # dK = dS^T Q (same factor)
    return dq, dk, dv


def attention_backward_rows(q, k, v, do, rows, scale, causal=False, kv_len=None):
    """dQ for selected query rows (each needs only its own row of P)."""
    rows = np.asarray(rows)
    qf = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do_r = np.asarray(do, dtype=np.float64)[rows]
    s = logits(qf[rows], k, scale)
    s = np.where(visible_rows(rows, k.shape[0], causal, kv_len), s, NEG_INF)
    p, _, _ = safe_softmax(s)
    dp = do_r @ v.T
    ds = softmax_grad(p, dp)
    return scale * (ds @ k)


# ----------------------------------------------------------------------------
# Online softmax, in the pages' steps ([P1] §Online Softmax; [P2] §6.2)
# ----------------------------------------------------------------------------
def online_softmax_state(x: np.ndarray, bounds) -> tuple[float, float]:
    """Scan one logit row block by block; return the running (m, l) at the end.

    ``bounds`` are the block edges, e.g. [0, 2, 4] splits a length-4 row in two.
    Per block: m_blk = max(block); m_new = max(m, m_blk);
    l = l * e^(m - m_new) + sum(e^(x_blk - m_new)); m = m_new.
    """
    m, l = NEG_INF, 0.0
    for a, b in zip(bounds[:-1], bounds[1:]):
        blk = np.asarray(x[a:b], dtype=np.float64)
        if blk.size == 0:
            continue
        m_new = max(m, float(np.max(blk)))
        if m_new == NEG_INF:          # nothing visible yet
            continue
        l = l * np.exp(m - m_new) + float(np.sum(np.exp(blk - m_new)))
        m = m_new
    return m, l


def merge_states(m1, l1, m2, l2):
    """Merge two partial (m, l) states: the rescaling rule of [P2] §6.2."""
    m = max(m1, m2)
    if m == NEG_INF:
        return NEG_INF, 0.0
    return m, l1 * np.exp(m1 - m) + l2 * np.exp(m2 - m)


def _rescale_factor(m_old: np.ndarray, m_new: np.ndarray) -> np.ndarray:
    """alpha = e^(m_old − m_new); 0 where nothing was seen before (m_old = −inf)."""
    with np.errstate(invalid="ignore"):
        a = np.exp(m_old - np.where(np.isfinite(m_new), m_new, 0.0))
    return np.where(np.isfinite(m_old), a, 0.0)


def _block_probs(qk: np.ndarray, m_new: np.ndarray) -> np.ndarray:
    """p = e^(qk − m_new) for the current block (0 on masked entries)."""
    return np.exp(qk - np.where(np.isfinite(m_new), m_new, 0.0)[:, None])


def _accumulate(acc, alpha, p, v_blk):
    """acc_new = alpha * acc_old + p @ V_blk ([P1] §Online Softmax)."""
    return acc * alpha[:, None] + p @ v_blk


def blocked_attention_forward(q, k, v, scale, causal=False, kv_len=None, block_m=64, block_n=64):
    """The forward loop of [P1] §FlashAttention Forward流程, in fp64.

    For each query block: m = −inf, l = 0, acc = 0; for each key/value block:
    qk = Q_i K_j^T * scale, masked; m_new = max(m, rowmax(qk)); p = e^(qk − m_new);
    alpha = e^(m − m_new); acc = acc*alpha + p V_j; l = l*alpha + rowsum(p);
    m = m_new. Finally O = acc / l and LSE = m + ln l.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    n, d = q.shape
    nk = k.shape[0]
    o = np.zeros((n, v.shape[1]))
    lse = np.full(n, NEG_INF)
    for i0 in range(0, n, block_m):
        rows = np.arange(i0, min(i0 + block_m, n))
        m = np.full(len(rows), NEG_INF)
        l = np.zeros(len(rows))
        acc = np.zeros((len(rows), v.shape[1]))
        for j0 in range(0, nk, block_n):
            cols = slice(j0, min(j0 + block_n, nk))
            qk = (q[rows] @ k[cols].T) * scale
            vis = visible_rows(rows, nk, causal, kv_len)[:, cols]
            qk = np.where(vis, qk, NEG_INF)
            m_new = np.maximum(m, np.max(qk, axis=1))
            p = _block_probs(qk, m_new)
            alpha = _rescale_factor(m, m_new)
            acc = _accumulate(acc, alpha, p, v[cols])
            l = l * alpha + np.sum(p, axis=1)
            m = m_new
        seen = l > 0
        o[rows[seen]] = acc[seen] / l[seen][:, None]
        lse[rows[seen]] = m[seen] + np.log(l[seen])
    return o, lse


# ----------------------------------------------------------------------------
# Batched wrappers over [B, H, N, d]
# ----------------------------------------------------------------------------
def batched_forward(q, k, v, scale, causal=False, kv_lens=None, heads=None):
    """q, k, v: [B, H, N, d]. Returns O [B, H, N, d] and LSE [B, H, N].

    ``heads`` optionally restricts the work to a list of (b, h) pairs; the
    other slices are left as NaN.
    """
    B, H, N, d = q.shape
    o = np.full((B, H, N, v.shape[-1]), np.nan)
    lse = np.full((B, H, N), np.nan)
    pairs = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    for b, h in pairs:
        L = None if kv_lens is None else int(kv_lens[b])
        o[b, h], lse[b, h] = attention_forward(q[b, h], k[b, h], v[b, h], scale, causal, L)
    return o, lse


def batched_backward(q, k, v, do, scale, causal=False, kv_lens=None, heads=None):
    """Returns dQ, dK, dV [B, H, N, d] (NaN outside ``heads`` when given)."""
    B, H, N, d = q.shape
    dq = np.full(q.shape, np.nan)
    dk = np.full(k.shape, np.nan)
    dv = np.full(v.shape, np.nan)
    pairs = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    for b, h in pairs:
        L = None if kv_lens is None else int(kv_lens[b])
        dq[b, h], dk[b, h], dv[b, h] = attention_backward(q[b, h], k[b, h], v[b, h], do[b, h],
                                                          scale, causal, L)
    return dq, dk, dv


# ----------------------------------------------------------------------------
# Packed variable-length batches: tokens of all sequences concatenated,
# arrays [total, H, d]; sequence b owns rows cu[b]:cu[b+1]. Causal masking is
# bottom-right aligned (offset n_k - n_q per sequence).
# ----------------------------------------------------------------------------
def varlen_forward(q, k, v, cu_q, cu_k, scale, causal=False):
    """Returns O [total_q, H, d] and LSE [H, total_q]."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    tq, H, d = q.shape
    o = np.zeros((tq, H, v.shape[2]))
    lse = np.full((H, tq), NEG_INF)
    for b in range(len(cu_q) - 1):
        qa, qe, ka, ke = int(cu_q[b]), int(cu_q[b + 1]), int(cu_k[b]), int(cu_k[b + 1])
        for h in range(H):
            o[qa:qe, h], lse[h, qa:qe] = attention_forward(q[qa:qe, h], k[ka:ke, h], v[ka:ke, h], scale, causal,
                                                           None, (ke - ka) - (qe - qa))
    return o, lse


def varlen_backward(q, k, v, do, cu_q, cu_k, scale, causal=False):
    """Returns dQ [total_q, H, d], dK, dV [total_k, H, d]."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    do = np.asarray(do, np.float64)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for b in range(len(cu_q) - 1):
        qa, qe, ka, ke = int(cu_q[b]), int(cu_q[b + 1]), int(cu_k[b]), int(cu_k[b + 1])
        for h in range(q.shape[1]):
            dq[qa:qe, h], dk[ka:ke, h], dv[ka:ke, h] = attention_backward(
                q[qa:qe, h], k[ka:ke, h], v[ka:ke, h], do[qa:qe, h], scale, causal, None, (ke - ka) - (qe - qa))
    return dq, dk, dv


# ----------------------------------------------------------------------------
# Decoding from a paged KV cache ([P3] §7.2-7.4): K/V live in a pool of
# fixed-size physical blocks [num_blocks, block_size, H, d]; a per-sequence
# block table maps logical block t // block_size to a physical block.
# ----------------------------------------------------------------------------
def gather_pages(pool, table_row, length, block_size):
    """The logical [length, H, d] cache of one sequence, read through its
    block table row (plain indexing, token by token)."""
    pool = np.asarray(pool)
    rows = [pool[int(table_row[t // block_size]), t % block_size] for t in range(length)]
    if not rows:
        return np.zeros((0,) + pool.shape[2:], dtype=pool.dtype)
    return np.stack(rows)


def paged_decode_forward(q, k_pool, v_pool, block_table, seq_lens, scale):
    """q: [B, H, d]; pools [num_blocks, block_size, H, d]; block_table
    [B, max_blocks]; seq_lens [B]. Returns O [B, H, d] and LSE [B, H]: each
    query attends to all seq_lens[b] keys of its sequence."""
    q = np.asarray(q, np.float64)
    B, H, d = q.shape
    bs = np.asarray(k_pool).shape[1]
    o = np.zeros((B, H, np.asarray(v_pool).shape[3]))
    lse = np.full((B, H), NEG_INF)
    for b in range(B):
        L = int(seq_lens[b])
        k = np.asarray(gather_pages(k_pool, block_table[b], L, bs), np.float64)
        v = np.asarray(gather_pages(v_pool, block_table[b], L, bs), np.float64)
        for h in range(H):
            ob, lb = attention_forward(q[b, h][None, :], k[:, h], v[:, h], scale)
            o[b, h], lse[b, h] = ob[0], lb[0]
    return o, lse
