"""Block-causal video attention for B300 (sm_103a).

Masked space attention and sliding-window causal time attention (with
grouped-query heads) of the block-causal transformer backbone shared by the
Open Dreamer tokenizer and dynamics model, forward and backward, as
hand-written CUDA behind a C ABI (include/od_attn.h).  This package is the thin
Python binding: it marshals torch tensors into that ABI and nothing else.

The CUDA library is loaded on first use of an op; if it has not been built,
the op raises instead of falling back to any other implementation.
"""
from __future__ import annotations

_API = (
    "space_attn_fwd", "space_attn_bwd", "time_attn_fwd", "time_attn_bwd", "time_attn_decode",
    "space_attn_fwd_packed", "time_attn_fwd_packed", "space_attn_bwd_packed", "time_attn_bwd_packed",
    "space_attn_fwd_varlen", "space_attn_bwd_varlen", "selftest_expired_wait",
    "bwd_workspace_bytes", "get_device_status", "get_device_status_detail", "library", "library_path",
    "debug_build", "debug_library",
    "ODError", "EXPORTED_SYMBOLS",
)


def __getattr__(name):
    if name in _API:
        from . import api
        return getattr(api, name)
    raise AttributeError(name)


__all__ = list(_API)
