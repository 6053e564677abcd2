"""Fused multi-head attention forward (and its backward) for NVIDIA GB300 (sm_103a).

The compute runs in hand-written CUDA (``csrc/``) behind the C ABI of
``include/mha_fwd.h``; this package only builds that library and binds its
entry points with ctypes.
"""
from ._binding import (MHA_ERR_CUDA, MHA_ERR_INVALID_ARG, MHA_ERR_MISALIGNED, MHA_ERR_NO_DEVICE,
                       MHA_ERR_SCRATCH_LIMIT, mha_fwd_kv_noalloc, mha_fwd_paged,
                       MHA_ERR_TIMEOUT, MHA_ERR_UNSUPPORTED_DIM, MHA_OK, MhaError, forward,
                       forward_kv, lib, mha_device_status, mha_fwd, mha_fwd_kv,
                       mha_fwd_kv_workspace_size, mha_set_wait_limit, mha_strerror,
                       mha_wait_selftest, mha_bwd, mha_bwd_workspace_size, backward,
                       mha_fwd_tile_order)
from .build import LIB, build

__all__ = [
    "MHA_OK", "MHA_ERR_INVALID_ARG", "MHA_ERR_UNSUPPORTED_DIM", "MHA_ERR_MISALIGNED",
    "MHA_ERR_CUDA", "MHA_ERR_TIMEOUT", "MHA_ERR_NO_DEVICE", "MhaError", "forward", "forward_kv",
    "mha_fwd_kv", "mha_fwd_kv_workspace_size", "mha_fwd_kv_noalloc", "MHA_ERR_SCRATCH_LIMIT", "mha_fwd_paged", "lib",
    "mha_device_status", "mha_fwd", "mha_set_wait_limit", "mha_strerror", "mha_wait_selftest",
    "LIB", "build", "mha_bwd", "mha_bwd_workspace_size", "backward", "mha_fwd_tile_order",
]
