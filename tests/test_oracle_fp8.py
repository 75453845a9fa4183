"""Pins of the FP8 oracle (oracle/fp8.py) on the CPU: the E4M3 format against
PyTorch's own float8_e4m3fn type, the block quantiser's stated properties,
lossless cases, and the P-rounding bounds against an emulation of the
rounding the kernel applies."""
import numpy as np
import pytest

from oracle import fp8
import oracle


def _rng(seed):
    return np.random.default_rng(seed)


def test_decode_known_codes():
    assert fp8.e4m3_decode(np.array([0x7E]))[0] == 448.0
    assert fp8.e4m3_decode(np.array([0x01]))[0] == 2.0 ** -9        # smallest subnormal
    assert fp8.e4m3_decode(np.array([0x08]))[0] == 2.0 ** -6        # smallest normal
    assert fp8.e4m3_decode(np.array([0x38]))[0] == 1.0
    assert fp8.e4m3_decode(np.array([0xB8]))[0] == -1.0
    assert np.isnan(fp8.e4m3_decode(np.array([0x7F, 0xFF]))).all()


def test_decode_matches_torch_for_every_code():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("no float8_e4m3fn in this torch")
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = fp8.e4m3_decode(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan], ref[~nan])


def test_round_matches_torch_in_range():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("no float8_e4m3fn in this torch")
    rng = _rng(1)
    x = np.concatenate([
        rng.uniform(-448, 448, 20000), rng.normal(0, 1, 20000), rng.normal(0, 2.0 ** -7, 20000),
        # exact midpoints between neighbouring codes (ties go to the even code)
        (fp8.e4m3_decode(np.arange(0, 0x7D)) + fp8.e4m3_decode(np.arange(1, 0x7E))) / 2,
    ]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn)
    got = fp8.e4m3_round(x.astype(np.float64))
    np.testing.assert_array_equal(got, ref.to(torch.float64).numpy())
    # bit for bit, signed zeros included (tiny negative values round to -0)
    np.testing.assert_array_equal(fp8.e4m3_encode(got), ref.view(torch.uint8).numpy())
    tiny = np.array([-1e-6, -2.0 ** -11, 1e-6], dtype=np.float32)
    np.testing.assert_array_equal(fp8.e4m3_encode(fp8.e4m3_round(tiny.astype(np.float64))),
                                  torch.from_numpy(tiny).to(torch.float8_e4m3fn).view(torch.uint8).numpy())


def test_round_saturates_and_encode_inverts_decode():
    assert fp8.e4m3_round(np.array([449.0, 470.0, 1e9, -1e9])).tolist() == [448.0, 448.0, 448.0, -448.0]
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    np.testing.assert_array_equal(fp8.e4m3_encode(fp8.e4m3_decode(codes)), codes)


def test_quantize_blocks_properties():
    rng = _rng(2)
    x = rng.normal(0, 3, size=(2, 300, 16)).astype(np.float32)
    x[1, 128:256] = 0                                          # an all-zero block
    codes, scales = fp8.quantize_blocks(x)
    assert scales.shape == (2, 3) and scales[1, 1] == 0 and not codes[1, 128:256].any()
    for s in range(2):
        for i in range(3):
            blk = x[s, i * 128:(i + 1) * 128]
            amax = np.max(np.abs(blk))
            if amax == 0:
                continue
            assert scales[s, i] == np.float32(amax / np.float32(448))
            # the largest magnitude maps to the largest code
            at = np.unravel_index(np.argmax(np.abs(blk)), blk.shape)
            assert fp8.e4m3_decode(codes[s, i * 128:(i + 1) * 128][at])[()] in (448.0, -448.0)
    deq = fp8.dequantize_blocks(codes, scales)
    err = np.abs(deq - x)
    rows = np.arange(300) // 128
    sc = scales[:, rows][:, :, None].astype(np.float64)
    # rounding error: half an ulp (2^-4 relative) or, below the normal range,
    # half the subnormal spacing; plus the fp32 scaling steps
    assert np.all(err <= np.maximum(2.0 ** -4 * np.abs(x), 2.0 ** -10 * sc) * (1 + 1e-6) + 1e-30)
    # blocks are independent: changing block 2 leaves blocks 0 and 1 alone
    x2 = x.copy()
    x2[0, 256:] *= 10
    c2, s2 = fp8.quantize_blocks(x2)
    np.testing.assert_array_equal(c2[0, :256], codes[0, :256])
    np.testing.assert_array_equal(s2[0, :2], scales[0, :2])


def test_lossless_inputs_give_the_exact_attention():
    # values that are e4m3 numbers times 2^k with the block maximum at 448 * 2^k
    # quantise exactly (scale 2^k), so the FP8 forward's oracle is the plain one
    rng = _rng(3)
    n, d = 200, 8
    mk = lambda: fp8.e4m3_decode(rng.integers(0, 0x7E, size=(n, d)).astype(np.uint8)) * \
        np.where(rng.random((n, d)) < 0.5, -1, 1)
    q, k, v = mk() * 2.0 ** -6, mk() * 2.0 ** -6, mk() * 2.0 ** -5
    for t, step in ((q, 2.0 ** -6), (k, 2.0 ** -6), (v, 2.0 ** -5)):
        t[0, 0], t[128, 0] = 448.0 * step, -448.0 * step      # each block's maximum: 448 * 2^k
    cq, sq = fp8.quantize_blocks(q[None])
    ck, sk = fp8.quantize_blocks(k[None])
    cv, sv = fp8.quantize_blocks(v[None])
    np.testing.assert_array_equal(fp8.dequantize_blocks(cq, sq)[0], q)
    o, lse = fp8.fp8_attention_forward(cq[0], sq[0], ck[0], sk[0], cv[0], sv[0], 0.3, True)
    o2, lse2 = oracle.attention_forward(q, k, v, 0.3, True)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)


def _emulate_p_rounding(q, k, v8, sv, scale, causal):
    """The P rounding the FP8 kernel applies, written out on its own: key blocks
    of 128 in order, a running maximum raised only when a block's maximum
    exceeds it by more than one binade, P' = e4m3(p * 2^7 * sV_b / max sV),
    l summed from the unrounded p, O = sum_j P'_j V8_j * (max sV / 2^7) / l
    with V8 the codes' values (the block scale rides on P')."""
    n, nk = q.shape[0], k.shape[0]
    x = scale * np.log2(np.e) * (q @ k.T)
    if causal:
        x = np.where(np.arange(nk)[None, :] <= np.arange(n)[:, None], x, -np.inf)
    smax = np.max(sv)
    o = np.zeros((n, v8.shape[1]))
    for r in range(n):
        m, l, acc = -np.inf, 0.0, np.zeros(v8.shape[1])
        for b in range(-(-nk // 128)):
            seg = x[r, b * 128:(b + 1) * 128]
            mb = np.max(seg)
            if mb == -np.inf:
                continue
            if mb > m + 1:
                if m > -np.inf:
                    alpha = 2.0 ** (m - mb)
                    l *= alpha
                    acc *= alpha
                m = mb
            p = 2.0 ** (seg - m)
            l += np.sum(p)
            pq = fp8.e4m3_round(p * 2.0 ** 7 * sv[b] / smax)
            acc += pq @ v8[b * 128:(b + 1) * 128]
        o[r] = acc * (smax / 2.0 ** 7) / l
    return o


@pytest.mark.parametrize("causal", [False, True])
def test_p_rounding_bounds_hold_for_an_emulation(causal):
    rng = _rng(4 + causal)
    n, d = 300, 16
    x = rng.normal(size=(3, n, d)).astype(np.float32)
    x[0] *= 2.0
    (cq, sq), (ck, sk), (cv, sv) = (fp8.quantize_blocks(x[i:i + 1]) for i in range(3))
    q, k, v = (fp8.dequantize_blocks(c, s)[0] for c, s in ((cq, sq), (ck, sk), (cv, sv)))
    exact, _ = fp8.fp8_attention_forward(cq[0], sq[0], ck[0], sk[0], cv[0], sv[0], 0.25, causal)
    emul = _emulate_p_rounding(q, k, fp8.e4m3_decode(cv[0]), sv[0].astype(np.float64), 0.25, causal)
    bound, var = fp8.p_rounding_bounds(cq[0], sq[0], ck[0], sk[0], cv[0], sv[0], 0.25, causal)
    err = np.abs(emul - exact)
    assert np.all(err <= bound * (1 + 1e-9) + 1e-12)
    assert np.sqrt(np.mean(err ** 2)) <= 1.5 * np.sqrt(np.mean(var))
    assert np.max(err) > 0  # the rounding does something


def test_row_subsets_match_the_full_slice():
    rng = _rng(6)
    x = rng.normal(size=(3, 260, 8)).astype(np.float32)
    (cq, sq), (ck, sk), (cv, sv) = (fp8.quantize_blocks(x[i:i + 1]) for i in range(3))
    args = (cq[0], sq[0], ck[0], sk[0], cv[0], sv[0], 0.4, True, 200)
    rows = np.array([0, 5, 127, 128, 259])
    o, lse = fp8.fp8_attention_forward(*args)
    o_r, lse_r = fp8.fp8_attention_forward(*args, rows=rows)
    np.testing.assert_allclose(o_r, o[rows], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(lse_r, lse[rows], rtol=1e-12)
    b, v = fp8.p_rounding_bounds(*args)
    b_r, v_r = fp8.p_rounding_bounds(*args, rows=rows)
    np.testing.assert_allclose(b_r, b[rows], rtol=1e-12, atol=1e-18)
    np.testing.assert_allclose(v_r, v[rows], rtol=1e-12, atol=1e-24)
