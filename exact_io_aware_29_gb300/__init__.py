"""Exact IO-aware attention (forward and backward) for GB300, sm_103a.

The computation lives in a CUDA library with a C ABI (``include/fa_gb300.h``);
this package holds its sources (``csrc/``), the in-tree build step
(``build.py``), the ctypes binding (``binding.py``) and the seeded synthetic
workloads (``synth.py``). Importing the package loads nothing; the first call
into the binding loads the library and raises if it is missing.
"""
from .binding import (  # noqa: F401
    FA_ERR_INVALID,
    FA_ERR_LAUNCH,
    FA_ERR_TIMEOUT,
    FA_ERR_UNSUPPORTED,
    FA_ERR_WORKSPACE,
    FA_OK,
    FaError,
    attention_backward,
    attention_backward_varlen,
    attention_decode_paged,
    attention_forward,
    attention_forward_fp8,
    attention_forward_varlen,
    fa_bwd,
    fa_bwd_deterministic,
    fa_bwd_varlen,
    fa_bwd_varlen_deterministic,
    fa_bwd_workspace_size,
    fa_check_status,
    fa_decode_paged,
    fa_decode_workspace_size,
    fa_fwd,
    fa_fwd_fp8,
    fa_fwd_varlen,
    fa_quantize_fp8,
    fa_status_string,
    library_path,
    load_library,
    quantize_fp8,
)
