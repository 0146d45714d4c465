"""B300-native RoPE repositioning and SegPagedAttention (per-head paged KV, no mask).

The compute lives in librk.so (C ABI, include/rk_api.h); `_binding` marshals torch
tensors into it.  The library is loaded on first use of any binding name, and that
fails with ImportError if librk.so has not been built (`python -m
head_aware_paged_rope_b300.build`).  The `build` and `roofline` submodules import
without it.
"""
_EXPORTS = (
    "AppendArgs", "RingArgs", "rope_coefficients", "SparseFfnArgs", "sparse_ffn_args", "sparse_ffn", "append_args", "append_kv", "ring_args", "ring_advance", "AttnArgs", "RkError", "RopeArgs", "RopeRun", "LIB", "attn_args", "rope_reposition", "rope_workspace_size",
    "segpaged_decode", "segpaged_decode_workspace_size", "segpaged_prefill", "segpaged_prefill_workspace_size",
    "status_string", "version", "RK_CLASS_DENSE", "RK_CLASS_GLOBAL", "RK_CLASS_LOCAL", "RK_CLASS_RETRIEVAL",
    "RK_ROPE_HALF_SPLIT", "RK_ROPE_INTERLEAVED", "RK_ATTN_METADATA_STABLE", "RK_ATTN_POOLS_STABLE", "RK_ATTN_DIAG_EXPIRE_WAIT",
)


def __getattr__(name):
    if name in _EXPORTS:
        from . import _binding
        return getattr(_binding, name)
    raise AttributeError(name)


__all__ = list(_EXPORTS)
