"""Kimi Delta Attention (KDA) on GB300 (sm_103a).

The compute lives in ``libkda.so`` (hand-written CUDA kernels behind the C ABI
declared in ``include/kda.h``); this package is its thin Python binding.  The
library is built in-tree by ``kimi_delta_attention_18_gb300.build`` and loaded
on first use; if it cannot be built or loaded, every call raises.
"""
from ._native import (  # noqa: F401
    KDAError,
    PrefillDesc,
    decode_step,
    lib,
    prefill_combine,
    library_path,
    prefill_backward,
    prefill_backward_num_segments,
    prefill_backward_workspace_size,
    prefill_chunked,
    prefill_chunked_ckpt,
    prefill_chunked_gated,
    prefill_ckpt_workspace_size,
    num_checkpoints,
    prefill_desc,
    prefill_num_segments,
    prefill_segments,
    prefill_workspace_size,
    state_compose,
    state_transfer,
)

__all__ = ["KDAError", "PrefillDesc", "decode_step", "lib", "library_path", "num_checkpoints",
           "prefill_backward",
           "prefill_backward_num_segments", "prefill_backward_workspace_size", "prefill_chunked", "prefill_chunked_ckpt", "prefill_chunked_gated",
           "prefill_ckpt_workspace_size", "prefill_combine", "prefill_desc",
           "prefill_num_segments", "prefill_segments", "prefill_workspace_size", "state_compose",
           "state_transfer"]
