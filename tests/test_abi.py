"""The C-ABI library: it loads, exports every declared symbol, and rejects bad
arguments on the host (no kernel launch needed for those)."""
import ctypes
import os
import re

import pytest

from exact_io_aware_29_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa_gb300.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load_library()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for n in ("fa_fwd", "fa_bwd", "fa_bwd_workspace_size", "fa_status_string", "fa_check_status"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name
        assert name in binding.SIGNATURES, name


def test_status_strings(lib):
    for st in (0, -1, -2, -3, -4, -5):
        assert lib.fa_status_string(st)
    assert b"unknown" in lib.fa_status_string(99)


def test_workspace_size(lib):
    B, H, N, d = 4, 16, 4096, 128
    rows = B * H * N
    assert lib.fa_bwd_workspace_size(B, H, N, d) >= rows * 4 * 2 + rows * d * 4
    assert lib.fa_bwd_workspace_size(0, 1, 1, 64) == 0
    assert lib.fa_bwd_workspace_size(1, 1, 1, 96) == 0


FAKE = 0x10000  # a 16-byte aligned non-null address; never dereferenced (rejected first)


@pytest.mark.parametrize("args,expect", [
    (dict(q=None), binding.FA_ERR_INVALID),
    (dict(B=0), binding.FA_ERR_INVALID),
    (dict(N=0), binding.FA_ERR_INVALID),
    (dict(scale=float("nan")), binding.FA_ERR_INVALID),
    (dict(scale=0.0), binding.FA_ERR_INVALID),
    (dict(scale=-1.0), binding.FA_ERR_INVALID),
    (dict(d=96), binding.FA_ERR_UNSUPPORTED),
    (dict(d=256), binding.FA_ERR_UNSUPPORTED),
    (dict(q=FAKE + 2), binding.FA_ERR_UNSUPPORTED),
])
def test_fwd_argument_errors(lib, args, expect):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, H=1, N=16, d=64, scale=0.125, causal=0,
             kv=None, stream=None)
    a.update(args)
    st = lib.fa_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["N"], a["d"], a["scale"],
                    a["causal"], a["kv"], a["stream"])
    assert st == expect


def test_bwd_workspace_error(lib):
    st = lib.fa_bwd(*([FAKE] * 9), 1, 1, 16, 64, 0.125, 0, None, None, 0, None)
    assert st == binding.FA_ERR_WORKSPACE
    st = lib.fa_bwd(*([FAKE] * 9), 1, 1, 16, 64, 0.125, 0, None, FAKE, 16, None)
    assert st == binding.FA_ERR_WORKSPACE


@pytest.mark.parametrize("fn", ["fa_bwd", "fa_bwd_deterministic"])
def test_bwd_argument_errors(lib, fn):
    f = getattr(lib, fn)
    ws = lib.fa_bwd_workspace_size(1, 1, 16, 64)
    assert f(None, *([FAKE] * 8), 1, 1, 16, 64, 0.125, 0, None, FAKE, ws, None) == binding.FA_ERR_INVALID
    assert f(*([FAKE] * 9), 1, 1, 16, 96, 0.125, 0, None, FAKE, ws, None) == binding.FA_ERR_UNSUPPORTED
    assert f(*([FAKE] * 9), 1, 1, 16, 64, 0.125, 0, None, FAKE, ws - 1, None) == binding.FA_ERR_WORKSPACE


def test_workspace_holds_the_deterministic_counters(lib):
    # padded rows x (2 vectors + d accumulator columns) fp32, then one counter
    # per 128-row block and the ticket
    B, H, N, d = 2, 3, 300, 64
    rows = B * H * 384
    assert lib.fa_bwd_workspace_size(B, H, N, d) >= rows * 4 * 2 + rows * d * 4 + rows // 128 * 4 + 4
