"""Pins of the fp64 oracle to facts the pages and the mathematics fix.

Every check here is independent of the oracle's own code: the pages' worked
example, closed forms, library routines (scipy, torch autograd), invariants and
brute-force finite differences. The mutation tests at the end plant the
mistakes the pages' own sketches contain (and a few plausible others) into the
oracle on the CPU and show that at least one pin catches each.
"""
import itertools
import math
import os

import numpy as np
import pytest
import scipy.special

import oracle
import oracle.attention as oa

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_example.txt")


def _read_golden():
    vals = {}
    with open(GOLDEN, encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, rest = line.split("=", 1)
            key = key.strip()
            if ":" in rest:
                expr, num = rest.rsplit(":", 1)
                vals[key] = (expr.strip(), [float(t) for t in num.split()])
            else:
                vals[key] = (None, [float(t) for t in rest.split()])
    return vals


def _rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------------------
# Worked example (page 1, section 一个小数值例子)
# ---------------------------------------------------------------------------
def test_golden_values_match_page_closed_forms():
    g = _read_golden()
    e = math.exp
    assert g["l1"][1][0] == pytest.approx(e(-1) + 1, rel=1e-15)
    assert g["l2"][1][0] == pytest.approx(e(-2) + e(-1) + 1 + e(-3), rel=1e-15)
    assert g["l_oneshot"][1][0] == pytest.approx(sum(e(x - 3) for x in (1, 2, 3, 0)), rel=1e-15)
    l2 = g["l2"][1][0]
    for x, p in zip((1, 2, 3, 0), g["p"][1]):
        assert p == pytest.approx(e(x - 3) / l2, rel=1e-15)
    assert g["lse"][1][0] == pytest.approx(3 + math.log(l2), rel=1e-15)


def test_worked_example_online_states():
    g = _read_golden()
    row = np.array(g["row"][1])
    m1, l1 = oracle.online_softmax_state(row, [0, 2])
    assert m1 == g["m1"][1][0]
    assert l1 == pytest.approx(g["l1"][1][0], rel=1e-15)
    m2, l2 = oracle.online_softmax_state(row, [int(b) for b in g["blocks"][1]])
    assert m2 == g["m2"][1][0]
    assert l2 == pytest.approx(g["l2"][1][0], rel=1e-15)


def test_worked_example_one_shot_definition():
    g = _read_golden()
    row = np.array([g["row"][1]])
    p, m, l = oracle.safe_softmax(row)
    assert m[0] == 3.0
    assert l[0] == pytest.approx(g["l_oneshot"][1][0], rel=1e-15)
    np.testing.assert_allclose(p[0], g["p"][1], rtol=1e-14)
    # LSE through the attention definition: one query, four keys, d = 1,
    # logits scale*q*k = the row when q = 1, scale = 1.
    q = np.ones((1, 1))
    k = np.array(g["row"][1])[:, None]
    v = np.eye(4)
    o, lse = oracle.attention_forward(q, k, v, 1.0)
    assert lse[0] == pytest.approx(g["lse"][1][0], rel=1e-15)
    np.testing.assert_allclose(o[0], g["p"][1], rtol=1e-14)


# ---------------------------------------------------------------------------
# Exactness of the blocked algorithm (page 2 §6.2-6.3; page 1 §Online Softmax)
# ---------------------------------------------------------------------------
def test_online_softmax_every_split_of_short_rows():
    rng = _rng(1)
    for _ in range(20):
        x = rng.normal(scale=5.0, size=8)
        _, m_ref, l_ref = oracle.safe_softmax(x[None, :])
        for cuts in itertools.chain.from_iterable(
                itertools.combinations(range(1, 8), r) for r in range(0, 8)):
            bounds = [0, *cuts, 8]
            m, l = oracle.online_softmax_state(x, bounds)
            assert m == m_ref[0]
            assert abs(l - l_ref[0]) <= 1e-14 * l_ref[0]


def test_online_softmax_random_splits_and_orders():
    rng = _rng(2)
    for _ in range(50):
        n = int(rng.integers(2, 400))
        x = rng.normal(scale=8.0, size=n)
        lse_ref = scipy.special.logsumexp(x)
        cuts = np.sort(rng.choice(np.arange(1, n), size=min(n - 1, int(rng.integers(1, 12))),
                                  replace=False))
        bounds = [0, *cuts.tolist(), n]
        m, l = oracle.online_softmax_state(x, bounds)
        assert abs((m + math.log(l)) - lse_ref) <= 1e-13 * max(1.0, abs(lse_ref))
        # merging the same blocks in a random order gives the same state
        states = [oracle.online_softmax_state(x[a:b], [0, b - a]) for a, b in
                  zip(bounds[:-1], bounds[1:])]
        order = rng.permutation(len(states))
        mm, ll = -np.inf, 0.0
        for i in order:
            mm, ll = oracle.merge_states(mm, ll, *states[i])
        assert mm == m
        assert abs(ll - l) <= 1e-13 * l


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("kv_len", [None, 1, 37, 100])
@pytest.mark.parametrize("blocks", [(16, 16), (64, 32), (7, 13), (128, 128)])
def test_blocked_forward_equals_definition(causal, kv_len, blocks):
    rng = _rng(3)
    n, d = 100, 16
    q, k, v = (rng.normal(size=(n, d)) for _ in range(3))
    o_ref, lse_ref = oracle.attention_forward(q, k, v, 0.25, causal, kv_len)
    o, lse = oracle.blocked_attention_forward(q, k, v, 0.25, causal, kv_len, *blocks)
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------------------
# Library special cases
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("causal,kv_len", [(False, None), (True, None), (False, 50), (True, 20)])
def test_forward_against_scipy_softmax(causal, kv_len):
    rng = _rng(4)
    n, d = 70, 12
    q, k, v = (rng.normal(size=(n, d)) for _ in range(3))
    scale = 1 / math.sqrt(d)
    o, lse = oracle.attention_forward(q, k, v, scale, causal, kv_len)
    for r in range(n):
        cols = [c for c in range(n) if (not causal or c <= r) and (kv_len is None or c < kv_len)]
        s = np.array([scale * float(np.dot(q[r], k[c])) for c in cols])
        p = scipy.special.softmax(s)
        np.testing.assert_allclose(o[r], p @ v[cols], rtol=1e-12, atol=1e-13)
        assert lse[r] == pytest.approx(scipy.special.logsumexp(s), rel=1e-13, abs=1e-13)


def test_backward_against_torch_autograd():
    torch = pytest.importorskip("torch")
    rng = _rng(5)
    n, d = 33, 8
    q, k, v, do = (rng.normal(size=(n, d)) for _ in range(4))
    for causal, kv_len in [(False, None), (True, None), (True, 20), (False, 7)]:
        tq, tk, tv = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q, k, v))
        s = (tq @ tk.T) * 0.3
        mask = torch.ones(n, n, dtype=torch.bool)
        if causal:
            mask &= torch.tril(torch.ones(n, n, dtype=torch.bool))
        if kv_len is not None:
            mask[:, kv_len:] = False
        s = s.masked_fill(~mask, float("-inf"))
        o = torch.softmax(s, dim=-1) @ tv
        (o * torch.tensor(do)).sum().backward()
        dq, dk, dv = oracle.attention_backward(q, k, v, do, 0.3, causal, kv_len)
        np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------------------
# Closed forms and invariants of the definition
# ---------------------------------------------------------------------------
def test_rows_of_p_sum_to_one():
    rng = _rng(6)
    q, k = rng.normal(size=(50, 8)), rng.normal(size=(50, 8))
    for causal, kv_len in [(False, None), (True, None), (True, 9)]:
        p = oracle.probabilities(q, k, 0.5, causal, kv_len)
        np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=1e-14)
        assert np.all(p[~oracle.visible(50, 50, causal, kv_len)] == 0)


def test_constant_v_gives_constant_o():
    rng = _rng(7)
    q, k = rng.normal(size=(40, 8)), rng.normal(size=(40, 8))
    row = rng.normal(size=5)
    v = np.tile(row, (40, 1))
    o, _ = oracle.attention_forward(q, k, v, 0.7, True, 31)
    np.testing.assert_allclose(o, np.tile(row, (40, 1)), rtol=1e-13)


def test_single_visible_key():
    rng = _rng(8)
    q, k, v = (rng.normal(size=(20, 4)) for _ in range(3))
    o, lse = oracle.attention_forward(q, k, v, 0.5, causal=True)
    np.testing.assert_array_equal(o[0], v[0])
    assert lse[0] == pytest.approx(0.5 * float(q[0] @ k[0]), rel=1e-14)
    o, lse = oracle.attention_forward(q, k, v, 0.5, causal=False, kv_len=1)
    np.testing.assert_allclose(o, np.tile(v[0], (20, 1)), rtol=1e-14)
    np.testing.assert_allclose(lse, 0.5 * (q @ k[0]), rtol=1e-14)


def test_zero_query_gives_mean_of_visible_values():
    rng = _rng(9)
    k, v = rng.normal(size=(30, 6)), rng.normal(size=(30, 6))
    q = np.zeros((30, 6))
    o, lse = oracle.attention_forward(q, k, v, 1.0, causal=True, kv_len=25)
    for r in range(30):
        cnt = min(r + 1, 25)
        np.testing.assert_allclose(o[r], v[:cnt].mean(axis=0), rtol=1e-13, atol=1e-15)
        assert lse[r] == pytest.approx(math.log(cnt), rel=1e-14)


def test_key_shift_invariance():
    # page 2 §6.3: a common additive shift of a row's logits leaves P unchanged.
    rng = _rng(10)
    q, k, v = (rng.normal(size=(25, 6)) for _ in range(3))
    u = rng.normal(size=6)
    o1, l1 = oracle.attention_forward(q, k, v, 0.4, True, None)
    o2, l2 = oracle.attention_forward(q, k + u, v, 0.4, True, None)
    np.testing.assert_allclose(o2, o1, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l2, l1 + 0.4 * (q @ u), rtol=1e-12, atol=1e-12)


def test_joint_key_permutation_invariance():
    rng = _rng(11)
    q, k, v = (rng.normal(size=(25, 6)) for _ in range(3))
    perm = rng.permutation(25)
    o1, l1 = oracle.attention_forward(q, k, v, 0.4)
    o2, l2 = oracle.attention_forward(q, k[perm], v[perm], 0.4)
    np.testing.assert_allclose(o2, o1, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l2, l1, rtol=1e-13)


def test_fully_masked_row_reading():
    rng = _rng(12)
    q, k, v = (rng.normal(size=(5, 4)) for _ in range(3))
    o, lse = oracle.attention_forward(q, k, v, 1.0, kv_len=0)
    assert np.all(o == 0) and np.all(lse == -np.inf)
    dq, dk, dv = oracle.attention_backward(q, k, v, rng.normal(size=(5, 4)), 1.0, kv_len=0)
    assert np.all(dq == 0) and np.all(dk == 0) and np.all(dv == 0)


def test_sampled_rows_equal_full():
    rng = _rng(13)
    q, k, v, do = (rng.normal(size=(64, 8)) for _ in range(4))
    rows = np.array([0, 5, 17, 63])
    o, lse = oracle.attention_forward(q, k, v, 0.3, True, 40)
    o_r, lse_r = oracle.attention_forward_rows(q, k, v, rows, 0.3, True, 40)
    np.testing.assert_allclose(o_r, o[rows], rtol=1e-13)
    np.testing.assert_allclose(lse_r, lse[rows], rtol=1e-13)
    dq, _, _ = oracle.attention_backward(q, k, v, do, 0.3, True, 40)
    np.testing.assert_allclose(oracle.attention_backward_rows(q, k, v, do, rows, 0.3, True, 40),
                               dq[rows], rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------------------
# Backward: brute-force central finite differences of L = sum(O ∘ dO)
# ---------------------------------------------------------------------------
def _fd_grads(q, k, v, do, scale, causal, kv_len, h=1e-6):
    def loss(qq, kk, vv):
        o, _ = oracle.attention_forward(qq, kk, vv, scale, causal, kv_len)
        return float(np.sum(o * do))

    grads = []
    for which in range(3):
        base = [q.copy(), k.copy(), v.copy()]
        g = np.zeros_like(base[which])
        for idx in np.ndindex(*g.shape):
            plus = [a.copy() for a in base]
            minus = [a.copy() for a in base]
            plus[which][idx] += h
            minus[which][idx] -= h
            g[idx] = (loss(*plus) - loss(*minus)) / (2 * h)
        grads.append(g)
    return grads


@pytest.mark.parametrize("n,d,causal,kv_len", [
    (1, 4, False, None), (3, 4, True, None), (8, 8, False, None), (8, 4, True, 5),
    (17, 4, True, None), (17, 8, False, 9),
])
def test_backward_finite_differences(n, d, causal, kv_len):
    rng = _rng(100 + n * 10 + d)
    q, k, v, do = (rng.normal(size=(n, d)) for _ in range(4))
    scale = 1 / math.sqrt(d) * 1.3
    dq, dk, dv = oracle.attention_backward(q, k, v, do, scale, causal, kv_len)
    fq, fk, fv = _fd_grads(q, k, v, do, scale, causal, kv_len)
    for a, f in ((dq, fq), (dk, fk), (dv, fv)):
        err = np.max(np.abs(a - f))
        ref = max(np.max(np.abs(f)), 1e-3)
        assert err <= 1e-6 * ref + 1e-9, (err, ref)


def test_backward_sum_identities():
    rng = _rng(14)
    n, d = 40, 8
    q, k, v, do = (rng.normal(size=(n, d)) for _ in range(4))
    for causal, kv_len in [(False, None), (True, None), (True, 30)]:
        dq, dk, dv = oracle.attention_backward(q, k, v, do, 0.35, causal, kv_len)
        # sum_c dS_rc = 0 for every row => sum_c dK_c = 0
        np.testing.assert_allclose(dk.sum(axis=0), 0.0, atol=1e-12)
        # sum_c dV_c = sum over rows with a visible key of dO_r
        np.testing.assert_allclose(dv.sum(axis=0), do.sum(axis=0), rtol=1e-12, atol=1e-12)
        p = oracle.probabilities(q, k, 0.35, causal, kv_len)
        ds = oracle.softmax_grad(p, do @ v.T)
        np.testing.assert_allclose(ds.sum(axis=1), 0.0, atol=1e-12)


def test_backward_with_stored_output():
    # The row term from the stored output, D = rowsum(dO ∘ O): with the exact
    # O (= P V) it is rowsum(dP ∘ P) and the gradients are the definition's;
    # a perturbed O moves dS by exactly -P * rowsum(dO ∘ perturbation).
    rng = _rng(15)
    n, d, scale = 33, 8, 0.35
    q, k, v, do = (rng.normal(size=(n, d)) for _ in range(4))
    for causal, kv_len in [(False, None), (True, None), (True, 20)]:
        o, _ = oracle.attention_forward(q, k, v, scale, causal, kv_len)
        ref = oracle.attention_backward(q, k, v, do, scale, causal, kv_len)
        same = oracle.attention_backward(q, k, v, do, scale, causal, kv_len, o_stored=o)
        for a, b in zip(ref, same):
            np.testing.assert_allclose(b, a, rtol=1e-10, atol=1e-12)
        eps = rng.normal(size=o.shape) * 1e-3
        moved = oracle.attention_backward(q, k, v, do, scale, causal, kv_len, o_stored=o + eps)
        p = oracle.probabilities(q, k, scale, causal, kv_len)
        dds = -p * np.sum(do * eps, axis=1, keepdims=True)
        np.testing.assert_allclose(moved[0], ref[0] + scale * dds @ k, rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(moved[1], ref[1] + scale * dds.T @ q, rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(moved[2], ref[2], rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# Mutation tests: plant a mistake in the oracle (CPU) and show a pin fails.
# ---------------------------------------------------------------------------
def _pins_hold():
    """A compact subset of the pins above; True when all hold."""
    ok = True
    try:
        test_worked_example_online_states()
        test_worked_example_one_shot_definition()
        test_blocked_forward_equals_definition(True, 37, (16, 16))
        test_forward_against_scipy_softmax(True, 20)
        test_backward_finite_differences(8, 4, True, 5)
        test_backward_against_torch_autograd()
    except AssertionError:
        ok = False
    return ok


def test_pins_hold_unmutated():
    assert _pins_hold()


def _overwrite_instead_of_accumulate(acc, alpha, p, v_blk):
    return p @ v_blk                                   # page 3 §6.2 sketch's slip


def _rescale_per_column(acc, alpha, p, v_blk):
    return acc * (alpha ** p.shape[1])[:, None] + p @ v_blk   # page 3 §3.3 sketch's slip


def _dropped_rescale_in_l(m_old, m_new):
    return np.where(np.isfinite(m_old), 1.0, 0.0)      # alpha forgotten


def _wrong_sign_softmax_grad(p, dp):
    return p * (dp + np.sum(dp * p, axis=-1, keepdims=True))


def _no_rowsum_softmax_grad(p, dp):
    return p * dp


def _max_over_wrong_axis(s):
    return np.max(s, axis=0) if s.ndim == 2 and s.shape[0] == s.shape[1] else np.max(s, axis=-1)


@pytest.mark.parametrize("name,target,mutant", [
    ("overwrite acc", "_accumulate", _overwrite_instead_of_accumulate),
    ("rescale per column", "_accumulate", _rescale_per_column),
    ("alpha dropped", "_rescale_factor", _dropped_rescale_in_l),
    ("dS sign", "softmax_grad", _wrong_sign_softmax_grad),
    ("dS rowsum dropped", "softmax_grad", _no_rowsum_softmax_grad),
    ("max over keys' axis", "row_max", _max_over_wrong_axis),
])
def test_mutations_are_caught(monkeypatch, name, target, mutant):
    monkeypatch.setattr(oa, target, mutant)
    assert not _pins_hold(), f"mutation '{name}' slipped past every pin"


def test_mutation_dropped_backward_scale(monkeypatch):
    orig = oa.attention_backward

    def mutant(q, k, v, do, scale, causal=False, kv_len=None):
        dq, dk, dv = orig(q, k, v, do, scale, causal, kv_len)
        return dq / scale, dk / scale, dv
    monkeypatch.setattr(oa, "attention_backward", mutant)
    monkeypatch.setattr(oracle, "attention_backward", mutant)
    assert not _pins_hold()


def test_mutation_transposed_dk(monkeypatch):
    orig = oa.attention_backward

    def mutant(q, k, v, do, scale, causal=False, kv_len=None):
        dq, dk, dv = orig(q, k, v, do, scale, causal, kv_len)
        p = oa.probabilities(q, k, scale, causal, kv_len)
        ds = oa.softmax_grad(p, np.asarray(do) @ np.asarray(v).T)
        return dq, scale * (ds @ np.asarray(q)), dv     # dS Q instead of dS^T Q
    monkeypatch.setattr(oa, "attention_backward", mutant)
    monkeypatch.setattr(oracle, "attention_backward", mutant)
    assert not _pins_hold()


# ---------------------------------------------------------------------------
# Packed variable-length batches with bottom-right causal alignment
# ---------------------------------------------------------------------------
def test_bottom_right_equals_tail_of_square_causal():
    # n_q queries placed at the end of an n_k-long sequence: bottom-right causal
    # on (n_q, n_k) is the last n_q rows of ordinary causal attention on a
    # square problem whose first n_k - n_q queries are arbitrary.
    rng = _rng(20)
    for n_q, n_k in ((1, 9), (5, 12), (12, 12), (3, 40)):
        q = rng.normal(size=(n_q, 8))
        k, v = rng.normal(size=(n_k, 8)), rng.normal(size=(n_k, 8))
        o, lse = oracle.attention_forward(q, k, v, 0.4, True, None, n_k - n_q)
        qsq = np.concatenate([rng.normal(size=(n_k - n_q, 8)), q])
        osq, lsesq = oracle.attention_forward(qsq, k, v, 0.4, True)
        np.testing.assert_allclose(o, osq[n_k - n_q:], rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(lse, lsesq[n_k - n_q:], rtol=1e-13)


def test_single_query_sees_every_key():
    rng = _rng(21)
    k, v = rng.normal(size=(30, 6)), rng.normal(size=(30, 6))
    q = rng.normal(size=(1, 6))
    o, lse = oracle.attention_forward(q, k, v, 0.5, True, None, 29)
    s = 0.5 * (k @ q[0])
    np.testing.assert_allclose(o[0], scipy.special.softmax(s) @ v, rtol=1e-12)
    assert lse[0] == pytest.approx(scipy.special.logsumexp(s), rel=1e-13)


def test_more_queries_than_keys_leaves_early_rows_empty():
    rng = _rng(22)
    q, k, v = rng.normal(size=(10, 4)), rng.normal(size=(4, 4)), rng.normal(size=(4, 4))
    o, lse = oracle.attention_forward(q, k, v, 1.0, True, None, 4 - 10)
    assert np.all(o[:6] == 0) and np.all(lse[:6] == -np.inf)
    assert np.all(np.isfinite(lse[6:]))


def test_varlen_is_per_sequence_attention():
    rng = _rng(23)
    cu_q = np.array([0, 5, 5, 17, 40])
    cu_k = np.array([0, 7, 10, 22, 45])
    H, d = 2, 8
    q = rng.normal(size=(cu_q[-1], H, d))
    k, v = rng.normal(size=(cu_k[-1], H, d)), rng.normal(size=(cu_k[-1], H, d))
    for causal in (False, True):
        o, lse = oracle.varlen_forward(q, k, v, cu_q, cu_k, 0.35, causal)
        # against brute force over the whole packed batch with a block mask
        for h in range(H):
            s = 0.35 * q[:, h] @ k[:, h].T
            for r in range(cu_q[-1]):
                b = np.searchsorted(cu_q, r, side="right") - 1
                lq, lk = cu_q[b + 1] - cu_q[b], cu_k[b + 1] - cu_k[b]
                i = r - cu_q[b]
                cols = [c for c in range(cu_k[b], cu_k[b + 1])
                        if not causal or (c - cu_k[b]) <= i + lk - lq]
                if not cols:
                    assert np.all(o[r, h] == 0) and lse[h, r] == -np.inf
                    continue
                np.testing.assert_allclose(o[r, h], scipy.special.softmax(s[r, cols]) @ v[cols, h],
                                           rtol=1e-12, atol=1e-13)
                assert lse[h, r] == pytest.approx(scipy.special.logsumexp(s[r, cols]), rel=1e-13)


def test_varlen_backward_finite_differences():
    rng = _rng(24)
    cu_q, cu_k = np.array([0, 3, 7]), np.array([0, 5, 9])
    H, d = 1, 4
    q = rng.normal(size=(7, H, d))
    k, v = rng.normal(size=(9, H, d)), rng.normal(size=(9, H, d))
    do = rng.normal(size=(7, H, d))
    dq, dk, dv = oracle.varlen_backward(q, k, v, do, cu_q, cu_k, 0.6, True)

    def loss(qq, kk, vv):
        o, _ = oracle.varlen_forward(qq, kk, vv, cu_q, cu_k, 0.6, True)
        return float(np.sum(o * do))

    h = 1e-6
    for arr, grad in ((q, dq), (k, dk), (v, dv)):
        fd = np.zeros_like(arr)
        for idx in np.ndindex(*arr.shape):
            a = arr.copy(); a[idx] += h
            b = arr.copy(); b[idx] -= h
            args_p = [a if x is arr else x for x in (q, k, v)]
            args_m = [b if x is arr else x for x in (q, k, v)]
            fd[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        assert np.max(np.abs(fd - grad)) <= 1e-6 * max(np.max(np.abs(fd)), 1e-3)


def test_sequences_without_keys_or_queries():
    rng = _rng(25)
    q = rng.normal(size=(4, 3))
    o, lse = oracle.attention_forward(q, np.zeros((0, 3)), np.zeros((0, 3)), 1.0, True)
    assert o.shape == (4, 3) and np.all(o == 0) and np.all(lse == -np.inf)
    o, lse = oracle.attention_forward(np.zeros((0, 3)), q, q, 1.0, False)
    assert o.shape == (0, 3) and lse.shape == (0,)
    cu_q, cu_k = np.array([0, 0, 4]), np.array([0, 2, 2])
    k = rng.normal(size=(2, 1, 3))
    o, lse = oracle.varlen_forward(q[:, None, :], k, k, cu_q, cu_k, 1.0, True)
    assert np.all(o == 0) and np.all(lse == -np.inf)   # sequence 1 has four queries and no keys


# ---------------------------------------------------------------------------
# Decoding from a paged KV cache ([P3] §7.2-7.4)
# ---------------------------------------------------------------------------
def _paged_case(seed, lens, bs, H=2, d=4, spare=3):
    """Random pool with scattered physical blocks; returns the pieces and the
    logical per-sequence caches built independently of the block table."""
    rng = _rng(seed)
    B = len(lens)
    need = [-(-L // bs) for L in lens]
    n_blocks = sum(need) + spare
    perm = rng.permutation(n_blocks)
    table = np.full((B, max(max(need), 1) + 1), -7)   # unused entries hold junk
    logical_k, logical_v = [], []
    k_pool = rng.normal(size=(n_blocks, bs, H, d))       # junk everywhere first
    v_pool = rng.normal(size=(n_blocks, bs, H, d))
    at = 0
    for b, L in enumerate(lens):
        kb, vb = rng.normal(size=(L, H, d)), rng.normal(size=(L, H, d))
        logical_k.append(kb)
        logical_v.append(vb)
        for t in range(need[b]):
            phys = int(perm[at]); at += 1
            table[b, t] = phys
            seg = slice(t * bs, min(L, (t + 1) * bs))
            k_pool[phys, :seg.stop - seg.start] = kb[seg]
            v_pool[phys, :seg.stop - seg.start] = vb[seg]
    q = rng.normal(size=(B, H, d))
    return q, k_pool, v_pool, table, np.array(lens), logical_k, logical_v


def test_paged_decode_brute_force():
    q, kp, vp, table, lens, lk, lv = _paged_case(30, [5, 1, 9], bs=4)
    o, lse = oracle.paged_decode_forward(q, kp, vp, table, lens, 0.45)
    for b, L in enumerate(lens):
        for h in range(q.shape[1]):
            s = np.array([0.45 * float(np.dot(q[b, h], lk[b][t, h])) for t in range(L)])
            p = scipy.special.softmax(s)
            want = sum(p[t] * lv[b][t, h] for t in range(L))
            np.testing.assert_allclose(o[b, h], want, rtol=1e-12, atol=1e-14)
            assert lse[b, h] == pytest.approx(scipy.special.logsumexp(s), rel=1e-13)


def test_paged_decode_equals_packed_single_queries():
    # paging is a pure re-indexing: one query per sequence over the contiguous
    # (packed) caches gives the same result through the independently pinned
    # packed-batch function
    q, kp, vp, table, lens, lk, lv = _paged_case(31, [7, 16, 3, 12], bs=8)
    o, lse = oracle.paged_decode_forward(q, kp, vp, table, lens, 0.3)
    cu_q = np.arange(len(lens) + 1)
    cu_k = np.concatenate([[0], np.cumsum(lens)])
    for causal in (False, True):
        ov, lsev = oracle.varlen_forward(q, np.concatenate(lk), np.concatenate(lv), cu_q, cu_k, 0.3, causal)
        np.testing.assert_allclose(o, ov, rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(lse, lsev.T, rtol=1e-13)


def test_paged_decode_block_permutation_and_junk_invariance():
    q, kp, vp, table, lens, _, _ = _paged_case(32, [6, 11], bs=4)
    o, lse = oracle.paged_decode_forward(q, kp, vp, table, lens, 0.7)
    rng = _rng(33)
    perm = rng.permutation(kp.shape[0])            # physical block p moves to perm[p]
    kp2, vp2 = np.empty_like(kp), np.empty_like(vp)
    kp2[perm], vp2[perm] = kp, vp
    table2 = np.where(table >= 0, perm[np.clip(table, 0, None)], table)
    o2, lse2 = oracle.paged_decode_forward(q, kp2, vp2, table2, lens, 0.7)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)
    # slots past each sequence's length and blocks it does not own are never read
    kp3, vp3 = kp.copy(), vp.copy()
    used = {(int(table[b, t // 4]), t % 4) for b in range(2) for t in range(lens[b])}
    for blk in range(kp.shape[0]):
        for slot in range(4):
            if (blk, slot) not in used:
                kp3[blk, slot] = 1e6
                vp3[blk, slot] = -1e6
    o3, lse3 = oracle.paged_decode_forward(q, kp3, vp3, table, lens, 0.7)
    np.testing.assert_array_equal(o, o3)
    np.testing.assert_array_equal(lse, lse3)


def test_paged_decode_degenerate_lengths():
    q, kp, vp, table, lens, lk, lv = _paged_case(34, [0, 1], bs=4)
    o, lse = oracle.paged_decode_forward(q, kp, vp, table, lens, 0.5)
    assert np.all(o[0] == 0) and np.all(lse[0] == -np.inf)        # no keys: empty row
    np.testing.assert_allclose(o[1], lv[1][0], rtol=1e-15)          # one key: O = V_0
    np.testing.assert_allclose(lse[1], 0.5 * np.einsum("hd,hd->h", q[1], lk[1][0]), rtol=1e-14)


def test_paged_decode_pins_catch_a_slot_off_by_one(monkeypatch):
    import oracle.attention as oa

    def shifted(pool, table_row, length, block_size):
        pool = np.asarray(pool)
        rows = [pool[int(table_row[t // block_size]), (t + 1) % block_size] for t in range(length)]
        return np.stack(rows) if rows else np.zeros((0,) + pool.shape[2:])

    monkeypatch.setattr(oa, "gather_pages", shifted)
    with pytest.raises(AssertionError):
        test_paged_decode_brute_force()
    with pytest.raises(AssertionError):
        test_paged_decode_equals_packed_single_queries()
