"""Closed forms and invariances of attention checked on the GPU path, within
the parity tolerances (O 1e-2, LSE 1e-3; gradient sums relative to the sum
of magnitudes). The same properties pin the oracle on the CPU; here they hold
the kernels to the definition without the oracle in between ("FlashAttention
算法详解" §先说结论 for O = softmax(scale QK^T + M) V, §Backward为什么更复杂 for the
gradients; the key-shift invariance is the max-subtraction argument of
"flash_attention.zh" §6.3)."""
import numpy as np
import pytest

from exact_io_aware_29_gb300 import binding, build, synth
import parity_util as pu

pytestmark = pytest.mark.gpu

SHAPES = [(2, 2, 300, 64), (2, 2, 517, 128)]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.load_library()


def bf16(x):
    """fp64 array -> (bf16 bit patterns, the fp64 values they hold)."""
    bits = synth.f32_to_bf16_bits(np.asarray(x, np.float32))
    return bits, synth.bf16_bits_to_f64(bits)


def normal(rng, shape, sigma=1.0):
    return bf16(rng.standard_normal(shape) * sigma)


def fwd(q, k, v, scale, causal, kv=None):
    import torch
    kv_dev = None if kv is None else torch.tensor(kv, dtype=torch.int32, device="cuda")
    o, lse = binding.attention_forward(pu.to_device(q), pu.to_device(k), pu.to_device(v), scale, causal, kv_dev)
    torch.cuda.synchronize()
    assert binding.fa_check_status() == binding.FA_OK
    return pu.bf16_tensor_to_f64(o), lse.cpu().numpy().astype(np.float64)


def visible_count(N, causal, kv):
    """[B, N] number of keys each query row sees."""
    B = len(kv)
    r = np.arange(N)
    lim = np.minimum(r + 1, N) if causal else np.full(N, N)
    return np.stack([np.minimum(lim, kv[b]) for b in range(B)])


@pytest.mark.parametrize("B,H,N,d", SHAPES)
@pytest.mark.parametrize("causal", [False, True])
def test_constant_value_rows_give_that_row(B, H, N, d, causal):
    """Every key carries the same value row v: each row with a visible key
    outputs v, whatever its weights."""
    rng = np.random.default_rng(41 + N + causal)
    q, _ = normal(rng, (B, H, N, d), 2.0)
    k, _ = normal(rng, (B, H, N, d))
    vrow_bits, vrow = normal(rng, (B, H, 1, d))
    v = np.ascontiguousarray(np.broadcast_to(vrow_bits, (B, H, N, d)))
    kv = [N, N // 3]
    o, _ = fwd(q, k, v, d ** -0.5, causal, kv)
    want = np.broadcast_to(vrow, (B, H, N, d))
    assert pu.o_err(o, want) <= pu.O_ATOL


@pytest.mark.parametrize("B,H,N,d", SHAPES)
def test_single_visible_key(B, H, N, d):
    """Key length 1: every row sees key 0 alone, so O_r = V_0 and
    LSE_r = scale q_r . k_0; causal row 0 likewise sees only key 0."""
    rng = np.random.default_rng(43 + N)
    (q, qf), (k, kf), (v, vf) = (normal(rng, (B, H, N, d)) for _ in range(3))
    scale = d ** -0.5
    o, lse = fwd(q, k, v, scale, False, [1] * B)
    assert pu.o_err(o, np.broadcast_to(vf[:, :, :1], o.shape)) <= pu.O_ATOL
    assert pu.max_abs(lse, scale * np.einsum("bhrd,bhd->bhr", qf, kf[:, :, 0])) <= pu.LSE_ATOL
    o, lse = fwd(q, k, v, scale, True)
    assert pu.o_err(o[:, :, 0], vf[:, :, 0]) <= pu.O_ATOL
    assert pu.max_abs(lse[:, :, 0], scale * np.einsum("bhd,bhd->bh", qf[:, :, 0], kf[:, :, 0])) <= pu.LSE_ATOL


@pytest.mark.parametrize("B,H,N,d", SHAPES)
@pytest.mark.parametrize("causal", [False, True])
def test_zero_query_averages_the_visible_values(B, H, N, d, causal):
    """Q = 0 makes every visible logit 0: P is uniform over the visible keys,
    O_r is the mean of their value rows and LSE_r = ln(their count)."""
    rng = np.random.default_rng(47 + N + causal)
    q = np.zeros((B, H, N, d), np.uint16)
    (k, _), (v, vf) = (normal(rng, (B, H, N, d)) for _ in range(2))
    kv = [N - 7, 129]
    o, lse = fwd(q, k, v, d ** -0.5, causal, kv)
    cnt = visible_count(N, causal, kv)                                     # [B, N]
    csum = np.cumsum(vf, axis=2)                                           # prefix sums over keys
    want = np.empty_like(vf)
    for b in range(B):
        want[b] = csum[b][:, cnt[b] - 1] / cnt[b][None, :, None]
    assert pu.o_err(o, want) <= pu.O_ATOL
    assert pu.max_abs(lse, np.broadcast_to(np.log(cnt)[:, None, :], lse.shape)) <= pu.LSE_ATOL


@pytest.mark.parametrize("B,H,N,d", SHAPES)
@pytest.mark.parametrize("causal", [False, True])
def test_adding_one_vector_to_every_key(B, H, N, d, causal):
    """K + u (the same u for every key row) adds scale q_r . u to every logit
    of row r: O is unchanged and LSE_r moves by that amount. Keys and u are
    multiples of 1/16 below 4 in magnitude, so K + u is exact in bf16."""
    rng = np.random.default_rng(53 + N + causal)
    q, qf = normal(rng, (B, H, N, d))
    v, _ = normal(rng, (B, H, N, d))
    kq = np.clip(np.round(rng.standard_normal((B, H, N, d)) * 16) / 16, -2, 2)
    u = np.round(rng.uniform(-1, 1, (B, H, 1, d)) * 16) / 16
    k0, _ = bf16(kq)
    k1, k1f = bf16(kq + u)
    assert np.array_equal(k1f, kq + u)
    scale = d ** -0.5
    kv = [N, N - 100]
    o0, l0 = fwd(q, k0, v, scale, causal, kv)
    o1, l1 = fwd(q, k1, v, scale, causal, kv)
    assert pu.max_abs(o1, o0) <= pu.O_ATOL
    assert pu.max_abs(l1 - l0, scale * np.einsum("bhrd,bhd->bhr", qf, u[:, :, 0])) <= pu.LSE_ATOL


@pytest.mark.parametrize("B,H,N,d", SHAPES)
def test_permuting_keys_with_their_values(B, H, N, d):
    """Without a mask, reordering the (key, value) pairs leaves O and LSE
    unchanged (only the kernels' summation order changes)."""
    rng = np.random.default_rng(59 + N)
    (q, _), (k, _), (v, _) = (normal(rng, (B, H, N, d)) for _ in range(3))
    perm = rng.permutation(N)
    o0, l0 = fwd(q, k, v, d ** -0.5, False)
    o1, l1 = fwd(q, np.ascontiguousarray(k[:, :, perm]), np.ascontiguousarray(v[:, :, perm]), d ** -0.5, False)
    assert pu.max_abs(o1, o0) <= pu.O_ATOL
    assert pu.max_abs(l1, l0) <= pu.LSE_ATOL


@pytest.mark.parametrize("B,H,N,d", SHAPES)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("deterministic", [False, True])
def test_gradient_sums(B, H, N, d, causal, deterministic):
    """Each row of dS sums to zero, so the dK rows sum to zero; each row of P
    sums to one, so the dV rows sum to the dO rows of the rows that see a
    key. Held per column to 1e-2 of the sum of magnitudes."""
    import torch
    rng = np.random.default_rng(61 + N + causal)
    (q, _), (k, _), (v, _), (do, dof) = (normal(rng, (B, H, N, d)) for _ in range(4))
    kv = [N, N // 2]
    kv_dev = torch.tensor(kv, dtype=torch.int32, device="cuda")
    t = [pu.to_device(x) for x in (q, k, v, do)]
    o, lse = binding.attention_forward(t[0], t[1], t[2], d ** -0.5, causal, kv_dev)
    dq, dk, dv = binding.attention_backward(t[0], t[1], t[2], o, lse, t[3], d ** -0.5, causal, kv_dev,
                                            deterministic=deterministic)
    torch.cuda.synchronize()
    assert binding.fa_check_status() == binding.FA_OK
    dk, dv = pu.bf16_tensor_to_f64(dk), pu.bf16_tensor_to_f64(dv)
    sees = visible_count(N, causal, kv) > 0                                 # [B, N]
    want_dv = np.einsum("bhrd,br->bhd", dof, sees.astype(np.float64))
    for got, want, mag in ((dk.sum(axis=2), 0.0, np.abs(dk).sum(axis=2)),
                           (dv.sum(axis=2), want_dv, np.abs(dv).sum(axis=2))):
        assert np.all(np.abs(got - want) <= 1e-2 * mag + 1e-6)
