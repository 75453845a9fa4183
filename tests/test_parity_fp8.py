"""GPU parity of the FP8 path: the block quantiser bit for bit against the
oracle's, and the FP8 forward against the attention of the dequantised inputs
within the bounds the e4m3 rounding of P allows (per element and in root mean
square; see oracle/fp8.py), LSE within 1e-3."""
import numpy as np
import pytest

from oracle import fp8 as ofp8
from exact_io_aware_29_gb300 import binding, build, synth
import parity_util as pu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.load_library()


def bits_f32(bits):
    return synth.bf16_bits_to_f32(bits)


@pytest.mark.parametrize("B,H,N,d", [(1, 2, 300, 128), (2, 1, 129, 64), (1, 1, 1, 128), (1, 3, 256, 128)])
@pytest.mark.parametrize("transpose", [False, True])
def test_quantizer_bit_exact(B, H, N, d, transpose):
    import torch
    x = synth.bf16_normal_tensor(9000 + N + d, synth.STREAM_Q, (B, H, N, d), sigma=3.0)
    if N > 128:
        x[0, 0, 128:256] = 0                                   # an all-zero block
    codes, scales = binding.quantize_fp8(pu.to_device(x), transpose)
    torch.cuda.synchronize()
    assert binding.fa_check_status() == binding.FA_OK
    rc, rs = ofp8.quantize_blocks(bits_f32(x).reshape(B * H, N, d))
    np.testing.assert_array_equal(scales.cpu().numpy().reshape(B * H, -1), rs)
    got = codes.cpu().numpy()
    if transpose:
        Np = got.shape[-1]
        got = got.reshape(B * H, d, Np)
        assert not got[:, :, N:].any()                          # padding columns are zero codes
        np.testing.assert_array_equal(got[:, :, :N].transpose(0, 2, 1), rc)
    else:
        np.testing.assert_array_equal(got.reshape(B * H, N, d), rc)


def _check_rows(o, lse, qb, kb, vb, scale, causal, kv_len, rows=None):
    """Compare O, LSE of one (b, h) slice (rows of it) with the oracle."""
    (cq, sq), (ck, sk), (cv, sv) = (ofp8.quantize_blocks(bits_f32(t)[None]) for t in (qb, kb, vb))
    args = (cq[0], sq[0], ck[0], sk[0], cv[0], sv[0], scale, causal, kv_len)
    ro, rl = ofp8.fp8_attention_forward(*args, rows=rows)
    bound, var = ofp8.p_rounding_bounds(*args, rows=rows)
    err = np.abs(o - ro)
    # bound: the P rounding, plus bf16 rounding of O (2^-8 relative) and fp32
    # accumulation order (small absolute slack)
    lim = 1.05 * bound + 2.0 ** -8 * np.abs(ro) + 1e-3
    assert np.all(err <= lim), float(np.max(err - lim))
    rms = float(np.sqrt(np.mean(err ** 2)))
    assert rms <= 1.5 * float(np.sqrt(np.mean(var))) + 2.0 ** -9 * float(np.sqrt(np.mean(ro ** 2))) + 1e-4, rms
    assert pu.max_abs(lse, rl) <= pu.LSE_ATOL
    return rms


CASES = []
for causal in (False, True):
    for N in (1, 129, 300, 700):
        CASES.append((1, 2, N, causal, None))
    CASES.append((2, 2, 500, causal, (1, 500)))


@pytest.mark.parametrize("B,H,N,causal,kv", CASES)
def test_fp8_forward_small(B, H, N, causal, kv):
    import torch
    d = 128
    w = synth.small(f"fp8 N{N}", B, H, N, d, causal, 9100 + N + (7 if causal else 0), kv_len_range=kv)
    inp = pu.Inputs(w)
    o, lse, _ = binding.attention_forward_fp8(inp.q, inp.k, inp.v, w.scale, causal, inp.kv_dev)
    torch.cuda.synchronize()
    assert binding.fa_check_status() == binding.FA_OK
    go, gl = pu.bf16_tensor_to_f64(o), lse.cpu().numpy()
    assert np.all(np.isfinite(go))
    for b in range(B):
        for h in range(H):
            _check_rows(go[b, h], gl[b, h], inp.q_bits[b, h], inp.k_bits[b, h], inp.v_bits[b, h], w.scale, causal,
                        inp.kv_len(b))


def test_fp8_forward_c3_full_size_sampled():
    """B2 H32 N8192 d128 causal with Q ~ N(0, 4^2) at full size: the codes of
    two heads checked bit for bit, and 96 seeded rows of those heads against
    the oracle."""
    import torch
    w = synth.C3
    inp = pu.Inputs(w)
    o, lse, (q8, sq, k8, sk, v8t, sv) = binding.attention_forward_fp8(inp.q, inp.k, inp.v, w.scale, True)
    torch.cuda.synchronize()
    assert binding.fa_check_status() == binding.FA_OK
    for b, h in ((0, 0), (1, 31)):
        rows = w.rows(b * w.H + h)[::5]
        rc, rs = ofp8.quantize_blocks(bits_f32(inp.k_bits[b, h])[None])
        np.testing.assert_array_equal(k8[b, h].cpu().numpy(), rc[0])
        np.testing.assert_array_equal(sk[b, h].cpu().numpy(), rs[0])
        go = pu.bf16_tensor_to_f64(o[b, h])[rows]
        gl = lse[b, h].cpu().numpy()[rows]
        _check_rows(go, gl, inp.q_bits[b, h], inp.k_bits[b, h], inp.v_bits[b, h], w.scale, True, None, rows)


@pytest.mark.slow
@pytest.mark.parametrize("name,heads", [("C5", ((0, 0), (0, 7))), ("C4", ((0, 3), (1, 9), (3, 15)))])
def test_fp8_forward_full_size_sampled(name, heads):
    """The FP8 forward's other benchmark shapes at full size: C5 (N65536) and
    C4 (key lengths per batch entry); 64 seeded rows of a few heads."""
    import torch
    w = synth.WORKLOADS[name]
    inp = pu.Inputs(w)
    o, lse, _ = binding.attention_forward_fp8(inp.q, inp.k, inp.v, w.scale, True, inp.kv_dev)
    torch.cuda.synchronize()
    assert binding.fa_check_status() == binding.FA_OK
    for b, h in heads:
        rows = np.sort(synth.distinct_rows(w.seed, synth.STREAM_ROWS, 64, w.N, salt=b * w.H + h))
        go = pu.bf16_tensor_to_f64(o[b, h])[rows]
        assert np.all(np.isfinite(go))
        _check_rows(go, lse[b, h].cpu().numpy()[rows], inp.q_bits[b, h], inp.k_bits[b, h], inp.v_bits[b, h],
                    w.scale, True, inp.kv_len(b), rows)


@pytest.mark.parametrize("hot", [(0, 4), (60, 64), (124, 128)])
def test_fp8_forward_row_maximum_at_every_block_position(hot):
    """Keys [hot) of every 128-key block carry far larger logits than the rest,
    so the row maximum sits at that position of each block: a maximum that
    missed any key of the block would leave P' far out of range."""
    import torch
    B, H, N, d = 1, 1, 512, 128
    rng = np.random.default_rng(9300 + hot[0])
    q = np.full((N, d), 0.5, np.float32) + rng.normal(0, 0.05, (N, d)).astype(np.float32)
    k = rng.normal(0, 0.1, (N, d)).astype(np.float32)
    pos = np.arange(N) % 128
    k[(pos >= hot[0]) & (pos < hot[1])] = 1.0
    v = rng.normal(0, 1, (N, d)).astype(np.float32)
    bits = [synth.f32_to_bf16_bits(x).reshape(B, H, N, d) for x in (q, k, v)]
    qd, kd, vd = (pu.to_device(b) for b in bits)
    scale = 1 / np.sqrt(d)
    for causal in (False, True):
        o, lse, _ = binding.attention_forward_fp8(qd, kd, vd, scale, causal)
        torch.cuda.synchronize()
        assert binding.fa_check_status() == binding.FA_OK
        _check_rows(pu.bf16_tensor_to_f64(o)[0, 0], lse.cpu().numpy()[0, 0], bits[0][0, 0], bits[1][0, 0],
                    bits[2][0, 0], scale, causal, None)
