"""GPU forward parity for V values anywhere in bf16's range, through the C ABI.

The forward runs P V in f16 when a CTA's V values fit f16 and repeats the scan
with bf16 operands and V scaled by a power of two when they do not. These
tests put V entries far outside f16's range (1e5, 3e38, 2^124) and far below
it (1e-30, bf16 subnormals), in whole tensors, sprinkled into N(0,1) data,
per head, and only in masked padding keys, and compare every element with the
fp64 oracle.

Tolerance. The parity bound on O (max-abs error 1e-2) holds for unit-variance V.
O is linear in V, so a V scaled by s gets the bound 1e-2 * s (plus bf16's
subnormal spacing 2^-133 for outputs that small). For V with a few extreme
entries the bound is taken per element as 1e-2 * max(u, A), with u the unit
of the slice's V and A_rc = sum_c P_rc |V_c,col| the size of the terms that
make up O_rc (the usual error bound of a weighted sum); A <= 1 for the
unit-variance entries, so those keep the plain bound. As everywhere, the bf16
rounding of the result itself (half an ulp of O) comes on top.
"""
import numpy as np
import pytest

import oracle
from exact_io_aware_29_gb300 import binding, build, synth
import parity_util as pu

pytestmark = pytest.mark.gpu

BF16_SUBNORMAL_STEP = 2.0 ** -133


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.load_library()


def bf16_bits(x64: np.ndarray) -> np.ndarray:
    return synth.f32_to_bf16_bits(np.asarray(x64, dtype=np.float32))


def run_fwd(q_bits, k_bits, v_bits, scale, causal, kv_lens=None):
    import torch
    q, k, v = (pu.to_device(b) for b in (q_bits, k_bits, v_bits))
    kv = None if kv_lens is None else torch.from_numpy(np.asarray(kv_lens, np.int32)).cuda()
    o, lse = binding.attention_forward(q, k, v, scale, causal, kv)
    torch.cuda.synchronize()
    assert binding.fa_check_status() == binding.FA_OK
    return pu.bf16_tensor_to_f64(o), lse.cpu().numpy().astype(np.float64)


def oracle_slice(q_bits, k_bits, v_bits, b, h, scale, causal, kv_len=None, rows=None):
    """Oracle O, LSE and A = P |V| for one (b, h) slice (all rows or ``rows``)."""
    q, k, v = (synth.bf16_bits_to_f64(x[b, h]) for x in (q_bits, k_bits, v_bits))
    if rows is None:
        o, lse = oracle.attention_forward(q, k, v, scale, causal, kv_len)
        a, _ = oracle.attention_forward(q, k, np.abs(v), scale, causal, kv_len)
    else:
        o, lse = oracle.attention_forward_rows(q, k, v, rows, scale, causal, kv_len)
        a, _ = oracle.attention_forward_rows(q, k, np.abs(v), rows, scale, causal, kv_len)
    return o, lse, a


def base_inputs(B, H, N, d, causal, seed, q_sigma=1.0):
    w = synth.small(f"vrange N{N} d{d}", B, H, N, d, causal, seed, q_sigma=q_sigma)
    return w, w.q(), w.k(), synth.bf16_bits_to_f64(w.v())


def check_weighted(o, lse, q_bits, k_bits, v_bits, w, kv_lens=None, rows_of=None, unit_of=None):
    """Every element within 1e-2 * max(u, A) + 2^-133, u the unit of the slice's
    V (1, or the factor a whole head was scaled by); LSE within the usual 1e-3."""
    worst = 0.0
    for b in range(w.B):
        for h in range(w.H):
            L = None if kv_lens is None else int(kv_lens[b])
            rows = None if rows_of is None else rows_of(b, h)
            u = 1.0 if unit_of is None else unit_of(b, h)
            ro, rl, a = oracle_slice(q_bits, k_bits, v_bits, b, h, w.scale, w.causal, L, rows)
            go = o[b, h] if rows is None else o[b, h][rows]
            gl = lse[b, h] if rows is None else lse[b, h][rows]
            assert np.all(np.isfinite(go)), f"non-finite O at (b={b}, h={h})"
            err = (np.abs(go - ro) - pu.bf16_half_ulp(ro)) / (pu.O_ATOL * np.maximum(u, a) + BF16_SUBNORMAL_STEP)
            worst = max(worst, float(err.max()))
            assert pu.max_abs(gl, rl) <= pu.LSE_ATOL
    assert worst <= 1.0, f"O error {worst:.3f} x the allowed bound"
    return worst


SCALES = [2.0 ** 17, 1e5, 2.0 ** 124, 2.0 ** -100, 1e-30, 2.0 ** -135]


@pytest.mark.parametrize("s", SCALES, ids=lambda s: f"{s:.3g}")
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_whole_v_scaled(s, d, causal):
    """V = bf16(s * N(0,1)): O within 1e-2 * s of the oracle on the same bf16 input."""
    w, qb, kb, v = base_inputs(1, 2, 300, d, causal, 31 + d + int(causal))
    vb = bf16_bits(s * v)
    o, lse = run_fwd(qb, kb, vb, w.scale, causal)
    for h in range(w.H):
        ro, rl, _ = oracle_slice(qb, kb, vb, 0, h, w.scale, causal)
        assert np.all(np.isfinite(o[0, h]))
        err = pu.o_err(o[0, h], ro)
        assert err <= pu.O_ATOL * s + BF16_SUBNORMAL_STEP, f"O error {err:.3g} against scale {s:.3g}"
        assert pu.max_abs(lse[0, h], rl) <= pu.LSE_ATOL


@pytest.mark.parametrize("s", [2.0 ** 20, 2.0 ** 110, 2.0 ** -110])
def test_scaled_v_is_scaled_o(s):
    """An exact power-of-two scaling of V scales O exactly (up to bf16 rounding of O)."""
    w, qb, kb, v = base_inputs(1, 3, 513, 128, True, 57)
    vb = bf16_bits(v)
    o1, l1 = run_fwd(qb, kb, vb, w.scale, True)
    o2, l2 = run_fwd(qb, kb, bf16_bits(s * v), w.scale, True)
    assert np.array_equal(l1, l2)
    # Both passes round P differently (f16 vs bf16), so compare against the
    # oracle-scale bound rather than bit for bit.
    assert float(np.max(np.abs(o2 / s - o1) - 2 * pu.bf16_half_ulp(o1))) <= 2 * pu.O_ATOL


@pytest.mark.parametrize("extreme", [1e5, 3e38, 1e-30, "mixed"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_sprinkled_extremes(extreme, d, causal):
    """N(0,1) V with 1 % of its entries set to +-extreme (random signs and places)."""
    w, qb, kb, v = base_inputs(2, 2, 700, d, causal, 101 + d + int(causal))
    rng = np.random.default_rng(7 + d)
    mask = rng.random(v.shape) < 0.01
    if extreme == "mixed":
        vals = rng.choice([1e5, 3e38, 1e-30, 2.0 ** -140], size=v.shape)
    else:
        vals = np.full(v.shape, float(extreme))
    v = np.where(mask, vals * rng.choice([-1.0, 1.0], size=v.shape), v)
    vb = bf16_bits(v)
    o, lse = run_fwd(qb, kb, vb, w.scale, causal)
    check_weighted(o, lse, qb, kb, vb, w)


def test_heads_on_different_scales():
    """Each head takes its own pass decision: normal, huge, tiny and mixed heads in one call."""
    w, qb, kb, v = base_inputs(1, 4, 640, 128, True, 211)
    v = v.copy()
    v[0, 1] *= 2.0 ** 100
    v[0, 2] *= 2.0 ** -115
    v[0, 3, ::97, 5] = 3e38
    vb = bf16_bits(v)
    o, lse = run_fwd(qb, kb, vb, w.scale, True)
    units = {1: 2.0 ** 100, 2: 2.0 ** -115}
    check_weighted(o, lse, qb, kb, vb, w, unit_of=lambda b, h: units.get(h, 1.0))


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_huge_values_only_in_masked_keys(d, causal):
    """Keys at or past kv_len are masked: 3e38 stored there must not touch O."""
    w, qb, kb, v = base_inputs(2, 2, 512, d, causal, 303 + d)
    kv = [300, 129]
    v = v.copy()
    for b, L in enumerate(kv):
        v[b, :, L:, :] = 3e38
    vb = bf16_bits(v)
    o, lse = run_fwd(qb, kb, vb, w.scale, causal, kv)
    for b in range(w.B):
        for h in range(w.H):
            ro, rl, _ = oracle_slice(qb, kb, vb, b, h, w.scale, causal, kv[b])
            assert pu.o_err(o[b, h], ro) <= pu.O_ATOL
            assert pu.max_abs(lse[b, h], rl) <= pu.LSE_ATOL


@pytest.mark.parametrize("d", [64, 128])
def test_tiny_values_with_normal_padding(d):
    """V of 2^-120 * N(0,1) below kv_len, unit-scale values past it: the
    masked keys must not hide the tiny range from the pass decision."""
    w, qb, kb, v = base_inputs(2, 2, 512, d, True, 313 + d)
    kv = [300, 129]
    s = 2.0 ** -120
    v = v.copy()
    for b, L in enumerate(kv):
        v[b, :, :L, :] *= s
    vb = bf16_bits(v)
    o, lse = run_fwd(qb, kb, vb, w.scale, True, kv)
    for b in range(w.B):
        for h in range(w.H):
            ro, rl, _ = oracle_slice(qb, kb, vb, b, h, w.scale, True, kv[b])
            assert pu.o_err(o[b, h], ro) <= pu.O_ATOL * s + BF16_SUBNORMAL_STEP
            assert pu.max_abs(lse[b, h], rl) <= pu.LSE_ATOL


def test_varlen_extremes():
    """The packed layout shares the kernel: one sequence with huge V, one tiny, one normal."""
    import torch
    H, d = 2, 128
    lens = [300, 513, 77]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    total = int(cu[-1])
    g = synth.small("vrange varlen", 1, 1, total * H, d, False, 409)
    q = g.q().reshape(total, H, d)
    k = g.k().reshape(total, H, d)
    v = synth.bf16_bits_to_f64(g.v()).reshape(total, H, d)
    units = [2.0 ** 90, 2.0 ** -120, 1.0]
    for i, u in enumerate(units):
        v[cu[i]:cu[i + 1]] *= u
    vb = bf16_bits(v)
    scale = 1.0 / np.sqrt(d)
    qt, kt, vt = (pu.to_device(x) for x in (q, k, vb))
    cud = torch.from_numpy(cu).cuda()
    o, lse = binding.attention_forward_varlen(qt, kt, vt, cud, cud, max(lens), max(lens), scale, True)
    torch.cuda.synchronize()
    assert binding.fa_check_status() == binding.FA_OK
    o = pu.bf16_tensor_to_f64(o)
    lse = lse.cpu().numpy().astype(np.float64)
    for i, L in enumerate(lens):
        a0, a1 = int(cu[i]), int(cu[i + 1])
        for h in range(H):
            qs, ks, vs = (synth.bf16_bits_to_f64(x[a0:a1, h]) for x in (q, k, vb))
            ro, rl = oracle.attention_forward(qs, ks, vs, scale, True)
            assert np.all(np.isfinite(o[a0:a1, h]))
            assert pu.o_err(o[a0:a1, h], ro) <= pu.O_ATOL * units[i] + BF16_SUBNORMAL_STEP
            assert pu.max_abs(lse[h, a0:a1], rl) <= pu.LSE_ATOL


@pytest.mark.slow
def test_c3_shape_with_extremes():
    """B2 H32 N8192 d128 causal, Q ~ N(0, 4^2): a quarter of the heads get V entries
    of 3e38 and 1e5, a quarter are scaled by 2^-120; sampled rows of every head."""
    import torch
    w = synth.C3
    gen = torch.Generator(device="cuda")
    gen.manual_seed(w.seed)
    shape = (w.B, w.H, w.N, w.d)
    q = (torch.randn(shape, device="cuda", generator=gen) * w.q_sigma).to(torch.bfloat16)
    k = torch.randn(shape, device="cuda", generator=gen).to(torch.bfloat16)
    v = torch.randn(shape, device="cuda", generator=gen)
    heads = torch.arange(w.H, device="cuda")
    big = (heads % 4 == 1).view(1, -1, 1, 1)
    tiny = (heads % 4 == 2).view(1, -1, 1, 1)
    spots = torch.rand(shape, device="cuda", generator=gen) < 0.002
    signs = torch.where(torch.rand(shape, device="cuda", generator=gen) < 0.5, -1.0, 1.0)
    huge = torch.where(torch.rand(shape, device="cuda", generator=gen) < 0.5, 3e38, 1e5) * signs
    v = torch.where(big & spots, huge, v)
    v = torch.where(tiny, v * 2.0 ** -120, v).to(torch.bfloat16)
    o, lse = binding.attention_forward(q, k, v, w.scale, True)
    torch.cuda.synchronize()
    assert binding.fa_check_status() == binding.FA_OK
    qb, kb, vb = (t.view(torch.int16).cpu().numpy().view(np.uint16) for t in (q, k, v))
    o = pu.bf16_tensor_to_f64(o)
    lse = lse.cpu().numpy().astype(np.float64)

    def rows_of(b, h):
        return synth.distinct_rows(w.seed, synth.STREAM_ROWS, 48, w.N, salt=b * w.H + h)

    check_weighted(o, lse, qb, kb, vb, w, rows_of=rows_of,
                   unit_of=lambda b, h: 2.0 ** -120 if h % 4 == 2 else 1.0)


def test_extremes_across_items_of_one_cta():
    """More Q-tile pairs than SMs, with heads of all four kinds interleaved:
    CTAs that take the bf16 pass run next to and after CTAs that do not."""
    w, qb, kb, v = base_inputs(2, 40, 1024, 128, True, 521)
    v = v.copy()
    units = {}
    for b in range(w.B):
        for h in range(w.H):
            if h % 4 == 1:
                v[b, h] *= 2.0 ** 100
                units[(b, h)] = 2.0 ** 100
            elif h % 4 == 2:
                v[b, h] *= 2.0 ** -115
                units[(b, h)] = 2.0 ** -115
            elif h % 4 == 3:
                v[b, h, ::61, 7] = 3e38
    vb = bf16_bits(v)
    o, lse = run_fwd(qb, kb, vb, w.scale, True)
    worst = 0.0
    for b, h in [(0, h) for h in range(8)] + [(1, h) for h in range(32, 40)]:
        ro, rl, a = oracle_slice(qb, kb, vb, b, h, w.scale, True)
        assert np.all(np.isfinite(o[b, h])), f"non-finite O at (b={b}, h={h})"
        u = units.get((b, h), 1.0)
        err = (np.abs(o[b, h] - ro) - pu.bf16_half_ulp(ro)) / (pu.O_ATOL * np.maximum(u, a) + BF16_SUBNORMAL_STEP)
        worst = max(worst, float(err.max()))
        assert pu.max_abs(lse[b, h], rl) <= pu.LSE_ATOL
    assert worst <= 1.0, f"O error {worst:.3f} x the allowed bound"


def test_many_heads_extremes_at_grid_end():
    """40000 (b, h) of one 256-row Q pair each (40000 CTAs, several head
    groups): heads with 3e38 entries at the start, middle and very end of the
    grid; sampled heads, every row."""
    import torch
    B, H, N, d = 8, 5000, 256, 64
    gen = torch.Generator(device="cuda")
    gen.manual_seed(9901)
    shape = (B, H, N, d)
    q = torch.randn(shape, device="cuda", generator=gen).to(torch.bfloat16)
    k = torch.randn(shape, device="cuda", generator=gen).to(torch.bfloat16)
    v = torch.randn(shape, device="cuda", generator=gen).to(torch.bfloat16)
    flat = v.view(B * H, N, d)
    huge = [0, 997, 20011, 39990, 39998, B * H - 1]
    for bh in huge:
        flat[bh, ::37, 3] = 3e38
    kv = torch.randint(1, N + 1, (B,), device="cuda", generator=gen, dtype=torch.int32)
    scale = 1.0 / np.sqrt(d)
    o, lse = binding.attention_forward(q, k, v, scale, True, kv)
    torch.cuda.synchronize()
    assert binding.fa_check_status() == binding.FA_OK
    kvl = kv.cpu().numpy()
    for bh in huge + [1, 5000, 23456, 39997]:
        b, h = divmod(bh, H)

        def bits(t):
            return t[b, h].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)

        qs, ks, vs = (synth.bf16_bits_to_f64(bits(t)) for t in (q, k, v))
        ro, rl = oracle.attention_forward(qs, ks, vs, scale, True, int(kvl[b]))
        a, _ = oracle.attention_forward(qs, ks, np.abs(vs), scale, True, int(kvl[b]))
        go = pu.bf16_tensor_to_f64(o[b, h])
        gl = lse[b, h].cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(go)), f"non-finite O at bh={bh}"
        err = (np.abs(go - ro) - pu.bf16_half_ulp(ro)) / (pu.O_ATOL * np.maximum(1.0, a) + BF16_SUBNORMAL_STEP)
        assert float(err.max()) <= 1.0, f"bh={bh}: O error {float(err.max()):.3f} x the allowed bound"
        assert pu.max_abs(gl, rl) <= pu.LSE_ATOL
