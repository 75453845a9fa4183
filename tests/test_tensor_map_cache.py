"""The library caches its TMA tensor maps on the host, keyed by address, type,
extents, strides, box and swizzle. These tests reuse one allocation for
problems of different shapes (a stale map would read the wrong extents) and
call the library from several host threads at once (the cache is shared
behind a mutex). The forward is deterministic, so every result must equal,
bit for bit, the same problem run on buffers of its own."""
import threading

import pytest

from exact_io_aware_29_gb300 import binding, build

pytestmark = pytest.mark.gpu

SHAPES = [(1, 2, 300, 128), (2, 1, 200, 64), (2, 3, 129, 128), (1, 1, 1000, 64)]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.load_library()


def _inputs(shape, seed):
    import torch
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return [torch.randn(shape, device="cuda", generator=g).to(torch.bfloat16) for _ in range(3)]


def _reference(shape, seed, causal):
    q, k, v = _inputs(shape, seed)
    o, lse = binding.attention_forward(q, k, v, shape[3] ** -0.5, causal)
    return o, lse


def test_same_storage_different_shapes():
    import torch
    n_max = max(b * h * n * d for b, h, n, d in SHAPES)
    store = [torch.empty(n_max, dtype=torch.bfloat16, device="cuda") for _ in range(4)]
    lse_store = torch.empty(max(b * h * n for b, h, n, _ in SHAPES), dtype=torch.float32, device="cuda")
    for rnd in range(2):  # the second round finds every map in the cache
        for i, shape in enumerate(SHAPES):
            b, h, n, d = shape
            causal = (i + rnd) % 2 == 0
            q, k, v, o = (s[: b * h * n * d].view(shape) for s in store)
            src = _inputs(shape, 100 + i)
            for dst, x in zip((q, k, v), src):
                dst.copy_(x)
            lse = lse_store[: b * h * n].view(b, h, n)
            binding.fa_fwd(q, k, v, o, lse, d ** -0.5, causal)
            torch.cuda.synchronize()
            assert binding.fa_check_status() == binding.FA_OK
            ro, rl = _reference(shape, 100 + i, causal)
            assert torch.equal(o, ro), (rnd, shape)
            assert torch.equal(lse, rl), (rnd, shape)


def test_backward_workspace_reused_across_shapes():
    import torch
    ws = torch.empty(max(binding.fa_bwd_workspace_size(b, h, n, d) for b, h, n, d in SHAPES), dtype=torch.uint8,
                     device="cuda")
    for i, shape in enumerate(SHAPES):
        q, k, v = _inputs(shape, 200 + i)
        do = _inputs(shape, 300 + i)[0]
        scale = shape[3] ** -0.5
        o, lse = binding.attention_forward(q, k, v, scale, True)
        got = binding.attention_backward(q, k, v, o, lse, do, scale, True, workspace=ws, deterministic=True)
        ref = binding.attention_backward(q, k, v, o, lse, do, scale, True, deterministic=True)
        torch.cuda.synchronize()
        assert binding.fa_check_status() == binding.FA_OK
        for a, b in zip(got, ref):
            assert torch.equal(a, b), shape


def test_concurrent_host_threads():
    import torch
    jobs = [(shape, 400 + i, i % 2 == 1) for i, shape in enumerate(SHAPES * 2)]
    refs = [_reference(shape, seed, causal) for shape, seed, causal in jobs]
    torch.cuda.synchronize()
    work = []
    for shape, seed, causal in jobs:
        q, k, v = _inputs(shape, seed)
        o = torch.empty_like(q)
        lse = torch.empty(shape[:3], dtype=torch.float32, device="cuda")
        work.append((q, k, v, o, lse, shape[3] ** -0.5, causal, torch.cuda.Stream()))
    torch.cuda.synchronize()
    errors = []

    def run(job):
        q, k, v, o, lse, scale, causal, stream = job
        try:
            for _ in range(20):
                binding.fa_fwd(q, k, v, o, lse, scale, causal, None, stream)
        except Exception as e:  # surfaced below
            errors.append(e)

    threads = [threading.Thread(target=run, args=(job,)) for job in work]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    assert binding.fa_check_status() == binding.FA_OK
    for (q, k, v, o, lse, *_), (ro, rl) in zip(work, refs):
        assert torch.equal(o, ro)
        assert torch.equal(lse, rl)
