"""fa_bwd_noalloc: the backward for callers that cannot allocate device memory.

Callers such as allocator or memory-pool callbacks, or frameworks whose device
memory belongs to another component, may not call cudaMalloc (or a caching
allocator) when they run the backward. fa_bwd_noalloc gives them the same
gradients as fa_bwd using a fixed scratch array that the library keeps in its
own static device memory. This file is collected last on purpose: it checks,
through the C ABI, that two calls in a row both match the workspace-taking
entry point within the parity tolerance, that both also match the fp64
oracle on every (b, h) slice, that the second call leaves the device's free
memory unchanged (the first call on a device may still load the library's
kernels, which reserves the fixed array), and that a problem too large for
the fixed scratch is refused with FA_ERR_SCRATCH_LIMIT before anything runs.
"""
import ctypes

import numpy as np
import pytest

from exact_io_aware_29_gb300 import binding, build, synth
import parity_util as pu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load_library()


def _rel(g, r):
    return pu.max_abs(g, r) / max(float(np.max(np.abs(r))), pu.ZERO_REF_FLOOR)


@pytest.mark.parametrize("B,H,N,d,causal,kv", [
    (2, 3, 700, 128, True, (300, 700)),
    (1, 4, 513, 64, False, None),
])
def test_noalloc_matches_fa_bwd_twice(lib, B, H, N, d, causal, kv):
    import torch
    w = synth.small("noalloc", B, H, N, d, causal, 4321 + N + d, kv_len_range=kv, backward=True)
    inp = pu.Inputs(w, with_do=True)
    o, lse = binding.attention_forward(inp.q, inp.k, inp.v, w.scale, causal, inp.kv_dev)
    ref = binding.attention_backward(inp.q, inp.k, inp.v, o, lse, inp.do, w.scale, causal, inp.kv_dev)
    torch.cuda.synchronize()
    ref = [pu.bf16_tensor_to_f64(t) for t in ref]
    # the fp64 oracle's gradients on the same inputs, slice by slice
    exact = [[pu.oracle_bwd_slice(inp, b, h) for h in range(H)] for b in range(B)]
    stream = torch.cuda.current_stream().cuda_stream
    kvp = None if inp.kv_dev is None else inp.kv_dev.data_ptr()
    for call in range(2):  # the second call starts from the first call's scratch contents
        dq, dk, dv = (torch.full_like(inp.q, float("nan")) for _ in range(3))
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        st = lib.fa_bwd_noalloc(inp.q.data_ptr(), inp.k.data_ptr(), inp.v.data_ptr(), o.data_ptr(),
                                lse.data_ptr(), inp.do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                B, H, N, d, ctypes.c_float(w.scale), int(causal), kvp, stream)
        assert st == binding.FA_OK, binding.fa_status_string(st)
        torch.cuda.synchronize()
        if call == 1:
            assert torch.cuda.mem_get_info()[0] == free_before
        assert lib.fa_check_status(stream) == binding.FA_OK
        got = [pu.bf16_tensor_to_f64(g) for g in (dq, dk, dv)]
        for g, r in zip(got, ref):
            assert np.all(np.isfinite(g))
            assert _rel(g, r) <= pu.GRAD_RTOL
        for b in range(B):
            for h in range(H):
                for i in range(3):
                    assert _rel(got[i][b, h], exact[b][h][i]) <= pu.GRAD_RTOL


def test_noalloc_rejects_problems_beyond_the_scratch(lib):
    import torch
    B, H, N, d = 64, 64, 4096, 128       # needs ~8.5 GB of workspace
    assert lib.fa_bwd_workspace_size(B, H, N, d) > binding.NOALLOC_SCRATCH_BYTES
    t = torch.zeros(16, dtype=torch.bfloat16, device="cuda")  # never read: refused on the host
    p = t.data_ptr()
    st = lib.fa_bwd_noalloc(p, p, p, p, p, p, p, p, p, B, H, N, d, ctypes.c_float(0.088), 1, None,
                            torch.cuda.current_stream().cuda_stream)
    assert st == binding.FA_ERR_SCRATCH_LIMIT
    assert b"fixed scratch" in lib.fa_status_string(st)
