"""B300-native RoPE repositioning and SegPagedAttention (per-head paged KV, no mask).

The compute lives in librk.so (C ABI, include/rk_api.h); `_binding` marshals torch
tensors into it.  Importing the package loads the library and fails if it is missing.
"""
from ._binding import (  # noqa: F401
    AttnArgs, RkError, RopeArgs, RopeRun, LIB, attn_args, rope_reposition, rope_workspace_size,
    segpaged_decode, segpaged_decode_workspace_size, segpaged_prefill, segpaged_prefill_workspace_size,
    status_string, version, RK_CLASS_DENSE, RK_CLASS_GLOBAL, RK_CLASS_LOCAL, RK_CLASS_RETRIEVAL,
    RK_ROPE_HALF_SPLIT, RK_ROPE_INTERLEAVED,
)
