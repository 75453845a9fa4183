"""The bounded-wait path, made to run out on purpose without faulting anything.

FA_TEST_DROP_LOADS=1 makes the kernels' TMA producers issue no loads, so every
wait that depends on them can only end by running out; FA_TEST_WAIT_LIMIT_NS
shortens the bound from 2 s to 2 ms. The kernels then record FA_ERR_TIMEOUT,
give up their remaining waits, free TMEM and return. The test checks that the
host reads that status and that the same context afterwards computes correct
results again.
"""
import numpy as np
import pytest

from exact_io_aware_29_gb300 import binding, build, synth
import parity_util as pu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.load_library()


def _case():
    w = synth.small("timeout", 1, 2, 300, 128, True, 99, kv_len_range=(250, 250), backward=True)
    return w, pu.Inputs(w, with_do=True)


def test_waits_run_out_then_context_recovers(monkeypatch):
    import torch
    w, inp = _case()
    assert binding.fa_check_status() == binding.FA_OK
    monkeypatch.setenv("FA_TEST_WAIT_LIMIT_NS", "2000000")
    monkeypatch.setenv("FA_TEST_DROP_LOADS", "1")
    o, lse = binding.attention_forward(inp.q, inp.k, inp.v, w.scale, True, inp.kv_dev)
    torch.cuda.synchronize()
    assert binding.fa_check_status() == binding.FA_ERR_TIMEOUT
    binding.attention_backward(inp.q, inp.k, inp.v, o, lse, inp.do, w.scale, True, inp.kv_dev)
    torch.cuda.synchronize()
    assert binding.fa_check_status() == binding.FA_ERR_TIMEOUT
    assert binding.fa_check_status() == binding.FA_OK  # reading the status clears it

    monkeypatch.delenv("FA_TEST_WAIT_LIMIT_NS")
    monkeypatch.delenv("FA_TEST_DROP_LOADS")
    o, lse = binding.attention_forward(inp.q, inp.k, inp.v, w.scale, True, inp.kv_dev)
    dq, dk, dv = binding.attention_backward(inp.q, inp.k, inp.v, o, lse, inp.do, w.scale, True, inp.kv_dev)
    torch.cuda.synchronize()
    assert binding.fa_check_status() == binding.FA_OK
    ro, rl = pu.oracle_fwd_slice(inp, 0, 1)
    assert pu.max_abs(pu.bf16_tensor_to_f64(o)[0, 1], ro) <= pu.O_ATOL
    assert pu.max_abs(lse.cpu().numpy()[0, 1], rl) <= pu.LSE_ATOL
    rq, rk, rv = pu.oracle_bwd_slice(inp, 0, 1)
    for g, r in ((dq, rq), (dk, rk), (dv, rv)):
        err = pu.max_abs(pu.bf16_tensor_to_f64(g)[0, 1], r) / max(float(np.max(np.abs(r))), pu.ZERO_REF_FLOOR)
        assert err <= pu.GRAD_RTOL


def test_waits_run_out_in_decode_fp8_and_deterministic_kernels(monkeypatch):
    """The same for the paged decode, the FP8 forward and the deterministic
    backward: every wait that depends on a dropped load runs out, the status
    reads FA_ERR_TIMEOUT, and the context afterwards computes correct results."""
    import torch
    w, inp = _case()
    o, lse = binding.attention_forward(inp.q, inp.k, inp.v, w.scale, True, inp.kv_dev)
    dw = synth.DecodeWorkload("timeout decode", 2, 2, 128, 64, 98, (100, 300), spare_blocks=1)
    kp, vp = (pu.to_device(dw.pool_bits(st)) for st in (synth.STREAM_K, synth.STREAM_V))
    qd = pu.to_device(dw.q())
    table = torch.from_numpy(dw.block_table()).cuda()
    lens = torch.from_numpy(dw.seq_lens()).cuda()
    L = int(dw.seq_lens().max())
    torch.cuda.synchronize()
    assert binding.fa_check_status() == binding.FA_OK
    monkeypatch.setenv("FA_TEST_WAIT_LIMIT_NS", "2000000")
    monkeypatch.setenv("FA_TEST_DROP_LOADS", "1")
    for run in (lambda: binding.attention_decode_paged(qd, kp, vp, table, lens, L, dw.scale),
                lambda: binding.attention_forward_fp8(inp.q, inp.k, inp.v, w.scale, True, inp.kv_dev),
                lambda: binding.attention_backward(inp.q, inp.k, inp.v, o, lse, inp.do, w.scale, True, inp.kv_dev,
                                                   deterministic=True)):
        run()
        torch.cuda.synchronize()
        assert binding.fa_check_status() == binding.FA_ERR_TIMEOUT
    monkeypatch.delenv("FA_TEST_WAIT_LIMIT_NS")
    monkeypatch.delenv("FA_TEST_DROP_LOADS")
    od, _ = binding.attention_decode_paged(qd, kp, vp, table, lens, L, dw.scale)
    dq, dk, dv = binding.attention_backward(inp.q, inp.k, inp.v, o, lse, inp.do, w.scale, True, inp.kv_dev,
                                            deterministic=True)
    torch.cuda.synchronize()
    assert binding.fa_check_status() == binding.FA_OK
    import oracle
    ro, _ = oracle.paged_decode_forward(synth.bf16_bits_to_f64(dw.q()), synth.bf16_bits_to_f64(dw.pool_bits(synth.STREAM_K)),
                                        synth.bf16_bits_to_f64(dw.pool_bits(synth.STREAM_V)), dw.block_table(),
                                        dw.seq_lens(), dw.scale)
    assert pu.max_abs(pu.bf16_tensor_to_f64(od), ro) <= pu.O_ATOL
    rq, rk, rv = pu.oracle_bwd_slice(inp, 0, 1)
    for g, r in ((dq, rq), (dk, rk), (dv, rv)):
        err = pu.max_abs(pu.bf16_tensor_to_f64(g)[0, 1], r) / max(float(np.max(np.abs(r))), pu.ZERO_REF_FLOOR)
        assert err <= pu.GRAD_RTOL
