"""Exact IO-aware attention for GB300 (sm_103a).

A thin Python binding over the C ABI of ``libfa.so`` (declared in
``include/fa.h``): every step of the attention path runs in the library's CUDA
kernels; this package only marshals PyTorch tensors into pointers, sizes and a
stream.  There is no fallback: if the library is missing or the device is not
sm_103, the calls raise.
"""
from ._binding import (  # noqa: F401
    FaError,
    HostPlan,
    fa_backward,
    fa_backward_blocksparse,
    fa_backward_dkdv,
    fa_backward_dq,
    fa_backward_dropout,
    fa_backward_noalloc,
    fa_backward_preprocess,
    fa_backward_workspace_size,
    fa_decode,
    fa_decode_workspace_size,
    fa_forward,
    fa_forward_blocksparse,
    fa_forward_dropout,
    fa_forward_fp8,
    fa_forward_tile_count,
    fa_get_device_error,
    fa_selftest_wait_timeout,
    fa_status_string,
    library,
    library_path,
)

__all__ = [
    "FaError", "HostPlan", "fa_forward", "fa_backward", "fa_decode", "fa_decode_workspace_size", "fa_forward_blocksparse", "fa_backward_blocksparse",
    "fa_forward_dropout", "fa_backward_dropout", "fa_forward_fp8", "fa_backward_preprocess", "fa_backward_dkdv",
    "fa_backward_dq", "fa_backward_noalloc",
    "fa_backward_workspace_size", "fa_forward_tile_count", "fa_get_device_error",
    "fa_selftest_wait_timeout", "fa_status_string", "library", "library_path",
]
