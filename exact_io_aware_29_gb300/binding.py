"""Python binding of the C ABI in ``include/fa_gb300.h`` (ctypes).

Argument marshalling only: tensors become device pointers, the stream becomes
a ``cudaStream_t``; every step of the computation runs in the CUDA library.
There is no fallback: if the library is missing or cannot be loaded, every
call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

from . import build as _build

_LIB: Optional[ctypes.CDLL] = None

FA_OK = 0
FA_ERR_INVALID = -1
FA_ERR_UNSUPPORTED = -2
FA_ERR_LAUNCH = -3
FA_ERR_TIMEOUT = -4
FA_ERR_WORKSPACE = -5
FA_ERR_SCRATCH_LIMIT = -6
NOALLOC_SCRATCH_BYTES = 64 << 20

# Every symbol the header declares, with its ctypes signature.
_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
SIGNATURES = {
    "fa_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _P, _P]),
    "fa_fwd_varlen": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P]),
    "fa_bwd_workspace_size": (ctypes.c_size_t, [_I, _I, _I, _I]),
    "fa_decode_workspace_size": (ctypes.c_size_t, [_I, _I, _I, _I]),
    "fa_quantize_fp8": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "fa_fwd_fp8": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _P, _P]),
    "fa_decode_paged": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, ctypes.c_size_t, _P]),
    "fa_bwd_varlen": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P,
                           ctypes.c_size_t, _P]),
    "fa_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _P, _P, ctypes.c_size_t, _P]),
    "fa_bwd_deterministic": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _P, _P,
                                  ctypes.c_size_t, _P]),
    "fa_bwd_varlen_deterministic": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I,
                                         _F, _I, _P, ctypes.c_size_t, _P]),
    "fa_check_status": (_I, [_P]),
    "fa_status_string": (ctypes.c_char_p, [_I]),
    "fa_last_cuda_error": (ctypes.c_char_p, []),
    "fa_bwd_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _P, _P]),
    "fa_timing_begin": (_I, [_I]),
    "fa_timing_read": (_I, [_I, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int)]),
    "fa_timing_end": (_I, []),
}

(KERNEL_FWD, KERNEL_BWD_PRE, KERNEL_BWD_MAIN, KERNEL_BWD_DQ, KERNEL_DECODE, KERNEL_DECODE_MERGE,
 KERNEL_FWD_FP8) = range(7)


class FaError(RuntimeError):
    def __init__(self, status: int, where: str):
        lib = load_library()
        msg = lib.fa_status_string(status).decode()
        if status == FA_ERR_LAUNCH:
            msg += " (" + lib.fa_last_cuda_error().decode() + ")"
        super().__init__(f"{where}: {msg}")
        self.status = status


def library_path() -> str:
    return _build.LIB


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load the CUDA library (raises if it has not been built)."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    p = path or _build.LIB
    if not os.path.exists(p):
        raise RuntimeError(f"CUDA attention library not built ({p}); run exact_io_aware_29_gb300.build.build()")
    lib = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _LIB = lib
    return lib


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _check_bhnd(name, t, shape=None):
    import torch
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if t.dtype != torch.bfloat16:
        raise ValueError(f"{name} must be bfloat16")
    if t.dim() != 4 or (shape is not None and tuple(t.shape) != tuple(shape)):
        raise ValueError(f"{name} must have shape [B, H, N, d] = {shape}")


def fa_fwd(q, k, v, o, lse, scale: float, causal: bool, kv_lens=None, stream=None) -> None:
    """O, LSE <- attention(Q, K, V); same semantics as the C entry point."""
    import torch
    _check_bhnd("q", q)
    B, H, N, d = q.shape
    for name, t in (("k", k), ("v", v), ("o", o)):
        _check_bhnd(name, t, q.shape)
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 [B, H, N] CUDA tensor")
    if kv_lens is not None and (kv_lens.dtype != torch.int32 or not kv_lens.is_cuda or kv_lens.numel() != B):
        raise ValueError("kv_lens must be an int32 [B] CUDA tensor")
    st = load_library().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d, float(scale),
                               int(bool(causal)), _ptr(kv_lens), _stream(stream))
    if st != FA_OK:
        raise FaError(st, "fa_fwd")


def _check_thd(name, t, H=None, d=None):
    import torch
    if not t.is_cuda or not t.is_contiguous() or t.dtype != torch.bfloat16 or t.dim() != 3:
        raise ValueError(f"{name} must be a contiguous bfloat16 CUDA tensor [total, H, d]")
    if (H is not None and t.shape[1] != H) or (d is not None and t.shape[2] != d):
        raise ValueError(f"{name} has the wrong H or d")


def _check_cu(name, cu, batch=None):
    import torch
    if cu.dtype != torch.int32 or not cu.is_cuda or cu.dim() != 1 or (batch is not None and cu.numel() != batch + 1):
        raise ValueError(f"{name} must be an int32 CUDA tensor [batch + 1]")


def fa_fwd_varlen(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, max_seqlen_k: int,
                  scale: float, causal: bool, stream=None) -> None:
    """Packed variable-length forward; same semantics as the C entry point."""
    import torch
    _check_thd("q", q)
    total_q, H, d = q.shape
    _check_thd("k", k, H, d)
    _check_thd("v", v, H, d)
    _check_thd("o", o, H, d)
    if tuple(o.shape) != tuple(q.shape) or tuple(v.shape) != tuple(k.shape):
        raise ValueError("o must match q and v must match k")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (H, total_q) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 [H, total_q] CUDA tensor")
    _check_cu("cu_seqlens_q", cu_seqlens_q)
    batch = cu_seqlens_q.numel() - 1
    _check_cu("cu_seqlens_k", cu_seqlens_k, batch)
    st = load_library().fa_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(cu_seqlens_q),
                                      _ptr(cu_seqlens_k), batch, H, d, total_q, k.shape[0], int(max_seqlen_q),
                                      int(max_seqlen_k), float(scale), int(bool(causal)), _stream(stream))
    if st != FA_OK:
        raise FaError(st, "fa_fwd_varlen")


def attention_forward_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, scale, causal,
                             stream=None):
    """Allocates O [total_q, H, d] and LSE [H, total_q], then calls fa_fwd_varlen."""
    import torch
    o = torch.empty_like(q)
    lse = torch.empty((q.shape[1], q.shape[0]), dtype=torch.float32, device=q.device)
    fa_fwd_varlen(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, scale, causal, stream)
    return o, lse


def fa_bwd_varlen(q, k, v, o, lse, dO, dq, dk, dv, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int,
                  max_seqlen_k: int, scale: float, causal: bool, workspace=None, stream=None) -> None:
    """Packed variable-length backward; same semantics as the C entry point."""
    _bwd_varlen("fa_bwd_varlen", q, k, v, o, lse, dO, dq, dk, dv, cu_seqlens_q, cu_seqlens_k, max_seqlen_q,
                max_seqlen_k, scale, causal, workspace, stream)


def fa_bwd_varlen_deterministic(q, k, v, o, lse, dO, dq, dk, dv, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int,
                                max_seqlen_k: int, scale: float, causal: bool, workspace=None,
                                stream=None) -> None:
    """fa_bwd_varlen with dQ summed in a fixed order: bitwise reproducible results."""
    _bwd_varlen("fa_bwd_varlen_deterministic", q, k, v, o, lse, dO, dq, dk, dv, cu_seqlens_q, cu_seqlens_k,
                max_seqlen_q, max_seqlen_k, scale, causal, workspace, stream)


def _bwd_varlen(fn, q, k, v, o, lse, dO, dq, dk, dv, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k,
                scale, causal, workspace, stream) -> None:
    import torch
    _check_thd("q", q)
    total_q, H, d = q.shape
    for name, t in (("k", k), ("v", v), ("o", o), ("dO", dO), ("dq", dq), ("dk", dk), ("dv", dv)):
        _check_thd(name, t, H, d)
    if lse.dtype != torch.float32 or tuple(lse.shape) != (H, total_q):
        raise ValueError("lse must be float32 [H, total_q]")
    _check_cu("cu_seqlens_q", cu_seqlens_q)
    batch = cu_seqlens_q.numel() - 1
    _check_cu("cu_seqlens_k", cu_seqlens_k, batch)
    need = fa_bwd_workspace_size(batch, H, int(max_seqlen_q), d)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    st = getattr(load_library(), fn)(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq),
                                     _ptr(dk), _ptr(dv), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), batch, H, d,
                                     total_q, k.shape[0], int(max_seqlen_q), int(max_seqlen_k), float(scale),
                                     int(bool(causal)), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(), _stream(stream))
    if st != FA_OK:
        raise FaError(st, fn)


def attention_backward_varlen(q, k, v, o, lse, dO, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k,
                              scale, causal, workspace=None, stream=None, deterministic: bool = False):
    """Allocates dQ, dK, dV, then calls fa_bwd_varlen (or its deterministic
    form). Returns (dQ, dK, dV)."""
    import torch
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    fn = fa_bwd_varlen_deterministic if deterministic else fa_bwd_varlen
    fn(q, k, v, o, lse, dO, dq, dk, dv, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, scale, causal,
       workspace, stream)
    return dq, dk, dv


def fa_bwd_workspace_size(B: int, H: int, N: int, d: int) -> int:
    return int(load_library().fa_bwd_workspace_size(B, H, N, d))


def fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, scale: float, causal: bool, kv_lens=None, workspace=None,
           stream=None) -> None:
    """dQ, dK, dV <- gradients of sum(O * dO); same semantics as the C entry point."""
    _bwd_fixed("fa_bwd", q, k, v, o, lse, dO, dq, dk, dv, scale, causal, kv_lens, workspace, stream)


def fa_bwd_deterministic(q, k, v, o, lse, dO, dq, dk, dv, scale: float, causal: bool, kv_lens=None,
                         workspace=None, stream=None) -> None:
    """fa_bwd with dQ summed in a fixed order: bitwise reproducible results."""
    _bwd_fixed("fa_bwd_deterministic", q, k, v, o, lse, dO, dq, dk, dv, scale, causal, kv_lens, workspace, stream)


def _bwd_fixed(fn, q, k, v, o, lse, dO, dq, dk, dv, scale, causal, kv_lens, workspace, stream) -> None:
    import torch
    _check_bhnd("q", q)
    B, H, N, d = q.shape
    for name, t in (("k", k), ("v", v), ("o", o), ("dO", dO), ("dq", dq), ("dk", dk), ("dv", dv)):
        _check_bhnd(name, t, q.shape)
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N):
        raise ValueError("lse must be float32 [B, H, N]")
    need = fa_bwd_workspace_size(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    st = getattr(load_library(), fn)(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq),
                                     _ptr(dk), _ptr(dv), B, H, N, d, float(scale), int(bool(causal)),
                                     _ptr(kv_lens), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                     _stream(stream))
    if st != FA_OK:
        raise FaError(st, fn)


def fa_bwd_noalloc(q, k, v, o, lse, dO, dq, dk, dv, scale: float, causal: bool, kv_lens=None,
                   stream=None) -> None:
    """fa_bwd with the library's fixed static scratch instead of a workspace:
    for callers that cannot allocate device memory at this point."""
    import torch
    _check_bhnd("q", q)
    B, H, N, d = q.shape
    for name, t in (("k", k), ("v", v), ("o", o), ("dO", dO), ("dq", dq), ("dk", dk), ("dv", dv)):
        _check_bhnd(name, t, q.shape)
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N):
        raise ValueError("lse must be float32 [B, H, N]")
    st = load_library().fa_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq),
                                       _ptr(dk), _ptr(dv), B, H, N, d, float(scale), int(bool(causal)),
                                       _ptr(kv_lens), _stream(stream))
    if st != FA_OK:
        raise FaError(st, "fa_bwd_noalloc")


def fa_check_status(stream=None) -> int:
    return int(load_library().fa_check_status(_stream(stream)))


def fa_status_string(status: int) -> str:
    return load_library().fa_status_string(status).decode()


def attention_forward(q, k, v, scale: float, causal: bool, kv_lens=None, stream=None):
    """Allocates O and LSE with torch, then calls fa_fwd. Returns (O, LSE)."""
    import torch
    B, H, N, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    fa_fwd(q, k, v, o, lse, scale, causal, kv_lens, stream)
    return o, lse


def attention_backward(q, k, v, o, lse, dO, scale: float, causal: bool, kv_lens=None, workspace=None,
                       stream=None, deterministic: bool = False):
    """Allocates dQ, dK, dV with torch, then calls fa_bwd (fa_bwd_deterministic
    if ``deterministic``). Returns (dQ, dK, dV)."""
    import torch
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    fn = fa_bwd_deterministic if deterministic else fa_bwd
    fn(q, k, v, o, lse, dO, dq, dk, dv, scale, causal, kv_lens, workspace, stream)
    return dq, dk, dv


def fa_decode_workspace_size(B: int, H: int, d: int, max_seq_len: int) -> int:
    return int(load_library().fa_decode_workspace_size(B, H, d, max_seq_len))


def fa_decode_paged(q, k_cache, v_cache, o, lse, block_table, seq_lens, max_seq_len: int, scale: float,
                    workspace=None, stream=None) -> None:
    """One decoding step over a paged KV cache; same semantics as the C entry point."""
    import torch
    if q.dtype != torch.bfloat16 or q.dim() != 3 or not q.is_contiguous():
        raise ValueError("q must be contiguous bf16 [B, H, d]")
    B, H, d = q.shape
    for name, t in (("k_cache", k_cache), ("v_cache", v_cache)):
        if t.dtype != torch.bfloat16 or t.dim() != 4 or tuple(t.shape[2:]) != (H, d) or not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous bf16 [num_blocks, block_size, H, d]")
    if tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("k_cache and v_cache must have the same shape")
    if o.dtype != torch.bfloat16 or tuple(o.shape) != (B, H, d) or not o.is_contiguous():
        raise ValueError("o must be contiguous bf16 [B, H, d]")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H):
        raise ValueError("lse must be float32 [B, H]")
    if block_table.dtype != torch.int32 or block_table.dim() != 2 or block_table.shape[0] != B \
            or not block_table.is_contiguous():
        raise ValueError("block_table must be contiguous int32 [B, max_blocks_per_seq]")
    if seq_lens.dtype != torch.int32 or tuple(seq_lens.shape) != (B,):
        raise ValueError("seq_lens must be int32 [B]")
    num_blocks, block_size = k_cache.shape[:2]
    if workspace is None:
        workspace = torch.empty(max(fa_decode_workspace_size(B, H, d, int(max_seq_len)), 1), dtype=torch.uint8,
                                device=q.device)
    st = load_library().fa_decode_paged(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o), _ptr(lse),
                                        _ptr(block_table), _ptr(seq_lens), B, H, d, num_blocks, block_size,
                                        block_table.shape[1], int(max_seq_len), float(scale), _ptr(workspace),
                                        workspace.numel() * workspace.element_size(), _stream(stream))
    if st != FA_OK:
        raise FaError(st, "fa_decode_paged")


def attention_decode_paged(q, k_cache, v_cache, block_table, seq_lens, max_seq_len, scale, workspace=None,
                           stream=None):
    """Allocates O and LSE, then calls fa_decode_paged. Returns (O, LSE)."""
    import torch
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
    fa_decode_paged(q, k_cache, v_cache, o, lse, block_table, seq_lens, max_seq_len, scale, workspace, stream)
    return o, lse


def fa_quantize_fp8(x, out, block_scale, transpose: bool, stream=None) -> None:
    """bf16 [B, H, N, d] -> E4M3 codes (uint8 [B, H, N, d], or [B, H, d, Np]
    with Np = N rounded up to 128 when ``transpose``) and fp32 block scales
    [B, H, ceil(N / 128)]; same semantics as the C entry point."""
    import torch
    _check_bhnd("x", x)
    B, H, N, d = x.shape
    nb = (N + 127) // 128
    shape = (B, H, d, nb * 128) if transpose else (B, H, N, d)
    if out.dtype != torch.uint8 or tuple(out.shape) != shape or not out.is_contiguous():
        raise ValueError(f"out must be contiguous uint8 {shape}")
    if block_scale.dtype != torch.float32 or tuple(block_scale.shape) != (B, H, nb):
        raise ValueError("block_scale must be float32 [B, H, ceil(N / 128)]")
    st = load_library().fa_quantize_fp8(_ptr(x), _ptr(out), _ptr(block_scale), B, H, N, d, int(bool(transpose)),
                                        _stream(stream))
    if st != FA_OK:
        raise FaError(st, "fa_quantize_fp8")


def quantize_fp8(x, transpose: bool = False, stream=None):
    """Allocates the codes and scales, then calls fa_quantize_fp8."""
    import torch
    B, H, N, d = x.shape
    nb = (N + 127) // 128
    shape = (B, H, d, nb * 128) if transpose else (B, H, N, d)
    out = torch.empty(shape, dtype=torch.uint8, device=x.device)
    sc = torch.empty((B, H, nb), dtype=torch.float32, device=x.device)
    fa_quantize_fp8(x, out, sc, transpose, stream)
    return out, sc


def fa_fwd_fp8(q8, k8, v8t, q_scale, k_scale, v_scale, o, lse, scale: float, causal: bool, kv_lens=None,
               stream=None) -> None:
    """FP8 forward from E4M3 codes and block scales; same semantics as the C entry point."""
    import torch
    B, H, N, d = q8.shape
    nb = (N + 127) // 128
    for name, t, shape in (("q8", q8, (B, H, N, d)), ("k8", k8, (B, H, N, d)), ("v8t", v8t, (B, H, d, nb * 128))):
        if t.dtype != torch.uint8 or tuple(t.shape) != shape or not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous uint8 {shape}")
    for name, t in (("q_scale", q_scale), ("k_scale", k_scale), ("v_scale", v_scale)):
        if t.dtype != torch.float32 or tuple(t.shape) != (B, H, nb):
            raise ValueError(f"{name} must be float32 [B, H, ceil(N / 128)]")
    _check_bhnd("o", o, (B, H, N, d))
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N):
        raise ValueError("lse must be float32 [B, H, N]")
    st = load_library().fa_fwd_fp8(_ptr(q8), _ptr(k8), _ptr(v8t), _ptr(q_scale), _ptr(k_scale), _ptr(v_scale),
                                   _ptr(o), _ptr(lse), B, H, N, d, float(scale), int(bool(causal)), _ptr(kv_lens),
                                   _stream(stream))
    if st != FA_OK:
        raise FaError(st, "fa_fwd_fp8")


def attention_forward_fp8(q, k, v, scale: float, causal: bool, kv_lens=None, stream=None):
    """Quantises bf16 Q, K, V (V transposed) and runs the FP8 forward.
    Returns (O, LSE, (q8, q_scale, k8, k_scale, v8t, v_scale))."""
    import torch
    q8, sq = quantize_fp8(q, False, stream)
    k8, sk = quantize_fp8(k, False, stream)
    v8t, sv = quantize_fp8(v, True, stream)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    fa_fwd_fp8(q8, k8, v8t, sq, sk, sv, o, lse, scale, causal, kv_lens, stream)
    return o, lse, (q8, sq, k8, sk, v8t, sv)


def fa_timing_begin(max_calls: int) -> None:
    st = load_library().fa_timing_begin(int(max_calls))
    if st != FA_OK:
        raise FaError(st, "fa_timing_begin")


def fa_timing_read(kind: int) -> tuple[float, int]:
    """(summed milliseconds, number of timed launches) of one kernel kind."""
    ms = ctypes.c_double(0.0)
    n = ctypes.c_int(0)
    st = load_library().fa_timing_read(int(kind), ctypes.byref(ms), ctypes.byref(n))
    if st != FA_OK:
        raise FaError(st, "fa_timing_read")
    return ms.value, n.value


def fa_timing_end() -> None:
    load_library().fa_timing_end()
