"""QLoRA NF4 + LoRA linear layer on B300 (sm_103a): thin Python binding of the C ABI.

The entry points have the names of the C ABI in ``include/qlora_nf4.h``:
``nf4_quantize``, ``nf4_dequantize``, ``qlora_linear_fwd``, ``qlora_linear_bwd``, their fp16
compute-type twins (``*_f16``), plus the merge, error-statistics, per-token-adapter and
size/utility calls.  This module only marshals torch tensors (device memory and the
current stream) into raw pointers; every step of the computation runs in the CUDA library
``libqlora_nf4.so``.  There is no CPU fallback: without the library or a compute-capability
10.3 GPU the calls raise.
"""
from __future__ import annotations

from ._binding import (  # noqa: F401
    NF4Tensor,
    QLoRAError,
    device_status,
    level_table,
    lib,
    nf4_dequantize,
    nf4_dequantize_f16,
    nf4_int4_error_stats,
    nf4_merge_lora,
    nf4_quantize,
    nf4_quantize_noalloc,
    nf4_quantize_workspace_bytes,
    nf4_storage_bytes,
    profile_start,
    profile_stop,
    qlora_linear_bwd,
    qlora_linear_bwd_f16,
    qlora_linear_fwd,
    qlora_linear_fwd_f16,
    qlora_linear_fwd_multi,
    qlora_workspace_bytes,
    status_str,
    wait_timeout_selftest,
)

__all__ = [
    "NF4Tensor", "QLoRAError", "device_status", "level_table", "lib", "nf4_dequantize",
    "nf4_dequantize_f16", "nf4_int4_error_stats", "nf4_merge_lora", "nf4_quantize",
    "nf4_quantize_noalloc", "nf4_quantize_workspace_bytes", "nf4_storage_bytes",
    "profile_start", "profile_stop", "qlora_linear_bwd", "qlora_linear_bwd_f16",
    "qlora_linear_fwd", "qlora_linear_fwd_f16", "qlora_linear_fwd_multi",
    "qlora_workspace_bytes", "status_str", "wait_timeout_selftest",
]
