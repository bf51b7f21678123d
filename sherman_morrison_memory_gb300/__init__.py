"""GB300 (sm_103a) Variational Linear Attention forward recurrence.

A thin ctypes binding over the C ABI declared in ``include/vla.h``
(``_build/libvla_gb300.so``). Every step of the recurrence runs in the CUDA
kernels of that library; this module only checks and marshals arguments and
uses torch for device memory and streams. There is no CPU fallback: if the
library is missing, calls raise.

    o, (S, A, zk) = vla_forward(q, k, v, u, lambda0=0.1, eps=1e-4, state=None)

q, k, v, u: [B, H, T, d] float32 or bfloat16 tensors (d in 32, 64, 96, 128).
CUDA tensors run on their device's current stream; CPU tensors are copied to
the current CUDA device, run, and the results copied back (the end-to-end
path of a caller holding host buffers).
"""
from __future__ import annotations

from ._binding import (  # noqa: F401
    VLA_OK,
    VLA_ERR_INVALID_ARG,
    VLA_ERR_UNSUPPORTED,
    VLA_ERR_CUDA,
    VLA_ERR_TIMEOUT,
    VLA_ERR_NONFINITE,
    VLA_ALGO_AUTO,
    VLA_ALGO_PER_TOKEN,
    VLA_ALGO_CHUNKED,
    VLA_ALGO_DECODE,
    VLA_ALGO_CHUNKED_PAIR,
    VLA_ALGO_CHUNKED_ROWS,
    VLA_ALGO_SEGMENTED,
    VLAError,
    library_path,
    load_library,
    vla_backward,
    vla_forward,
    vla_get_last_device_status,
    vla_linear_attention_state,
    vla_status_string,
    vla_workspace_bytes,
)

__all__ = [
    "vla_forward",
    "vla_backward",
    "vla_get_last_device_status",
    "vla_linear_attention_state",
    "vla_status_string",
    "vla_workspace_bytes",
    "VLAError",
]
