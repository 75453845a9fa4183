"""The library allocates no device memory: with every buffer (and workspace)
provided by the caller, repeated calls of each entry point leave the device's
free memory unchanged (driver-level cudaMemGetInfo, which any cudaMalloc of
the library would move by at least one 2 MB page)."""
import numpy as np
import pytest

from exact_io_aware_29_gb300 import binding, build, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.load_library()


def _unchanged(fn, calls=10):
    import torch
    for _ in range(3):  # first calls load modules and set kernel attributes
        fn()
    torch.cuda.synchronize()
    before = torch.cuda.mem_get_info()[0]
    for _ in range(calls):
        fn()
    torch.cuda.synchronize()
    after = torch.cuda.mem_get_info()[0]
    assert binding.fa_check_status() == binding.FA_OK
    assert after == before, (before, after)


def test_forward_and_backward_allocate_nothing():
    import torch
    B, H, N, d = 2, 4, 1000, 128
    q, k, v, do = (torch.randn(B, H, N, d, device="cuda").to(torch.bfloat16) for _ in range(4))
    o, dq, dk, dv = (torch.empty_like(q) for _ in range(4))
    lse = torch.empty(B, H, N, device="cuda")
    kv = torch.tensor([700, 1000], dtype=torch.int32, device="cuda")
    ws = torch.empty(binding.fa_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device="cuda")
    _unchanged(lambda: binding.fa_fwd(q, k, v, o, lse, 0.1, True, kv))
    _unchanged(lambda: binding.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, 0.1, True, kv, ws))
    _unchanged(lambda: binding.fa_bwd_deterministic(q, k, v, o, lse, do, dq, dk, dv, 0.1, True, kv, ws))
    _unchanged(lambda: binding.fa_bwd_noalloc(q, k, v, o, lse, do, dq, dk, dv, 0.1, True, kv))


def test_packed_paged_and_fp8_paths_allocate_nothing():
    import torch
    H, d = 2, 128
    lens = [300, 1, 700]
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device="cuda")
    T = int(sum(lens))
    q, k, v, do = (torch.randn(T, H, d, device="cuda").to(torch.bfloat16) for _ in range(4))
    o, dq, dk, dv = (torch.empty_like(q) for _ in range(4))
    lse = torch.empty(H, T, device="cuda")
    ws = torch.empty(binding.fa_bwd_workspace_size(3, H, 700, d), dtype=torch.uint8, device="cuda")
    _unchanged(lambda: binding.fa_fwd_varlen(q, k, v, o, lse, cu, cu, 700, 700, 0.1, True))
    _unchanged(lambda: binding.fa_bwd_varlen(q, k, v, o, lse, do, dq, dk, dv, cu, cu, 700, 700, 0.1, True, ws))

    w = synth.DecodeWorkload("mem", 3, H, d, 128, 5, (100, 900))
    kp = torch.randn((w.n_blocks, w.block_size, H, d), device="cuda").to(torch.bfloat16)
    vp = torch.randn_like(kp)
    qd = torch.randn((3, H, d), device="cuda").to(torch.bfloat16)
    od, lsed = torch.empty_like(qd), torch.empty(3, H, device="cuda")
    table = torch.from_numpy(w.block_table()).cuda()
    sl = torch.from_numpy(w.seq_lens()).cuda()
    L = int(w.seq_lens().max())
    wsd = torch.empty(max(binding.fa_decode_workspace_size(3, H, d, L), 1), dtype=torch.uint8, device="cuda")
    _unchanged(lambda: binding.fa_decode_paged(qd, kp, vp, od, lsed, table, sl, L, 0.1, wsd))

    B, N = 1, 500
    x = torch.randn(B, H, N, d, device="cuda").to(torch.bfloat16)
    q8, sq = binding.quantize_fp8(x, False)
    v8, sv = binding.quantize_fp8(x, True)
    o8, lse8 = torch.empty_like(x), torch.empty(B, H, N, device="cuda")
    _unchanged(lambda: binding.fa_quantize_fp8(x, q8, sq, False))
    _unchanged(lambda: binding.fa_fwd_fp8(q8, q8, v8, sq, sq, sv, o8, lse8, 0.1, True))
