"""tg: training products of linear layers on GB300 (sm_103a).

The compute lives in ``libtg.so`` (hand-written CUDA behind a C ABI, declared
in ``include/tg.h``).  This package is a thin ctypes binding with the same
names as the C entry points; it only marshals torch tensors' device pointers,
shapes and the current CUDA stream.  Importing the package does not load the
library; the first call does, and fails loudly if it has not been built.
"""
from __future__ import annotations

__all__ = [
    "tg_gemm_fwd", "tg_gemm_dgrad", "tg_gemm_wgrad", "tg_gemm_fwd_lora", "tg_gemm_dgrad_lora",
    "tg_gemm_wgrad_noalloc", "tg_gemm_wgrad_accumulate",
    "tg_lora_down", "tg_lora_up", "tg_lora_grad", "tg_lora_up_add", "tg_lora_grad_add",
    "tg_lora_down_f32w", "tg_lora_up_f32w", "tg_lora_grad_f32w", "tg_bmm_attn", "tg_attn_fwd", "tg_attn_bwd",
    "tg_workspace_size", "tg_plan_describe", "tg_stream_status",
    "tg_status_string", "tg_load_table", "tg_version", "tg_last_call", "tg_wait_probe", "lib",
    "TGError",
]


def __getattr__(name):
    if name in __all__:
        from . import _binding
        return getattr(_binding, name)
    raise AttributeError(name)
