"""GB300-native fused multi-head attention forward (sm_103a).

The compute path lives in the C-ABI library ``libattn.so`` (hand-written CUDA,
see ``csrc/`` and ``include/attn.h``).  This package is its thin ctypes
binding: argument marshalling only.  The library is loaded on first use and a
missing or unbuilt library is an error, never a fallback.
"""
from . import binding
from .binding import (ATTN_BF16, ATTN_F16, ATTN_OK, AttnError, attn_bwd, attn_fwd, attn_fwd_f32,
                      attn_fwd_host, attn_fwd_strided, bwd_workspace_size, declared_symbols,
                      fwd_masked_raw, fwd_raw, fwd_strided_raw, fwd_workspace_size, host_plan,
                      lib_path, load, pool_stats, query, shutdown, status, strerror)

__all__ = ["ATTN_BF16", "ATTN_F16", "ATTN_OK", "AttnError", "attn_bwd", "attn_fwd", "attn_fwd_f32",
           "attn_fwd_host", "attn_fwd_strided", "binding", "bwd_workspace_size",
           "declared_symbols", "fwd_masked_raw", "fwd_raw", "fwd_strided_raw",
           "fwd_workspace_size", "host_plan", "lib_path", "load", "pool_stats", "query",
           "shutdown", "status", "strerror"]
