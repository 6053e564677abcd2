"""ctypes binding over libmha_fwd.so: argument marshalling only.

Every function here forwards to the C entry point of the same name declared
in include/mha_fwd.h.  Nothing is computed in Python; if the compiled
library is missing the first call raises instead of falling back.
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB

MHA_OK = 0
MHA_ERR_INVALID_ARG = 1
MHA_ERR_UNSUPPORTED_DIM = 2
MHA_ERR_MISALIGNED = 3
MHA_ERR_CUDA = 4
MHA_ERR_TIMEOUT = 5
MHA_ERR_NO_DEVICE = 6
MHA_ERR_SCRATCH_LIMIT = 7

_lib = None


class MhaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {mha_strerror(status)} (status {status})")


def lib() -> ctypes.CDLL:
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError(
                f"CUDA library not built: {LIB} is missing (run __graft_entry__.build())")
        L = ctypes.CDLL(LIB)
        vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        L.mha_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
        L.mha_fwd.restype = i
        L.mha_strerror.argtypes = [i]
        L.mha_strerror.restype = ctypes.c_char_p
        L.mha_device_status.argtypes = [vp, i, ctypes.POINTER(ctypes.c_uint)]
        L.mha_device_status.restype = i
        L.mha_set_wait_limit.argtypes = [ctypes.c_longlong]
        L.mha_set_wait_limit.restype = i
        L.mha_wait_selftest.argtypes = [ctypes.c_longlong, vp]
        L.mha_wait_selftest.restype = i
        L.mha_fwd_kv.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp, ctypes.c_size_t, vp]
        L.mha_fwd_kv.restype = i
        L.mha_fwd_kv_workspace_size.argtypes = [i, i, i, i, i, i]
        L.mha_fwd_kv_workspace_size.restype = ctypes.c_size_t
        L.mha_fwd_paged.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, i, vp,
                                    ctypes.c_size_t, vp]
        L.mha_fwd_paged.restype = i
        L.mha_fwd_kv_noalloc.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp]
        L.mha_fwd_kv_noalloc.restype = i
        L.mha_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp,
                              ctypes.c_size_t, vp]
        L.mha_bwd.restype = i
        L.mha_bwd_workspace_size.argtypes = [i, i, i, i]
        L.mha_bwd_workspace_size.restype = ctypes.c_size_t
        L.mha_fwd_tile_order.argtypes = [i, i, i, i, i, i, ctypes.POINTER(i)]
        L.mha_fwd_tile_order.restype = i
        _lib = L
    return _lib


def _ptr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream(stream) -> int:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def mha_strerror(status: int) -> str:
    return lib().mha_strerror(int(status)).decode()


def mha_fwd(q, k, v, o, lse, B: int, H: int, N: int, d: int, scale: float, causal: bool,
            stream=None) -> None:
    """C ``mha_fwd``: tensors (or raw device addresses) in, status checked."""
    rc = lib().mha_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(H), int(N),
                       int(d), ctypes.c_float(scale), int(bool(causal)), _stream(stream))
    if rc != MHA_OK:
        raise MhaError(rc, "mha_fwd")


def mha_device_status(stream=None, reset: bool = True):
    """(status, raw word) of the current device after synchronising ``stream``."""
    word = ctypes.c_uint(0)
    rc = lib().mha_device_status(_stream(stream), int(bool(reset)), ctypes.byref(word))
    return rc, word.value


def mha_set_wait_limit(cycles: int) -> None:
    rc = lib().mha_set_wait_limit(int(cycles))
    if rc != MHA_OK:
        raise MhaError(rc, "mha_set_wait_limit")


def mha_wait_selftest(cycles: int, stream=None) -> int:
    return int(lib().mha_wait_selftest(int(cycles), _stream(stream)))


def forward(q, k, v, causal: bool = False, scale: float | None = None, stream=None):
    """Allocate O and LSE with torch and run ``mha_fwd`` on [B, H, N, d] bf16 tensors."""
    import torch
    if q.dtype != torch.bfloat16 or k.dtype != torch.bfloat16 or v.dtype != torch.bfloat16:
        raise TypeError("q, k, v must be bfloat16")
    if not (q.shape == k.shape == v.shape) or q.dim() != 4:
        raise ValueError("q, k, v must share one [B, H, N, d] shape")
    if not (q.is_contiguous() and k.is_contiguous() and v.is_contiguous()):
        raise ValueError("q, k, v must be contiguous")
    B, H, N, d = q.shape
    if scale is None:
        scale = float(torch.tensor(d, dtype=torch.float32).rsqrt())
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    mha_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, stream)
    return o, lse


def mha_fwd_kv_workspace_size(B: int, H: int, Nq: int, Nk: int, d: int, num_splits: int = 0) -> int:
    return int(lib().mha_fwd_kv_workspace_size(int(B), int(H), int(Nq), int(Nk), int(d), int(num_splits)))


def mha_fwd_kv(q, k, v, o, lse, B: int, H: int, Nq: int, Nk: int, d: int, scale: float,
               causal: bool, num_splits: int, workspace, workspace_bytes: int, stream=None) -> None:
    """C ``mha_fwd_kv``: tensors (or raw device addresses) in, status checked."""
    rc = lib().mha_fwd_kv(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(H), int(Nq),
                          int(Nk), int(d), ctypes.c_float(scale), int(bool(causal)), int(num_splits),
                          _ptr(workspace), int(workspace_bytes), _stream(stream))
    if rc != MHA_OK:
        raise MhaError(rc, "mha_fwd_kv")


def forward_kv(q, k, v, causal: bool = False, scale: float | None = None, num_splits: int = 0,
               stream=None):
    """Allocate O, LSE and the workspace with torch and run ``mha_fwd_kv``."""
    import torch
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if scale is None:
        scale = float(torch.tensor(d, dtype=torch.float32).rsqrt())
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    ws_bytes = mha_fwd_kv_workspace_size(B, H, Nq, Nk, d, num_splits)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=q.device)
    mha_fwd_kv(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, num_splits, ws, ws_bytes, stream)
    return o, lse


def mha_fwd_kv_noalloc(q, k, v, o, lse, B: int, H: int, Nq: int, Nk: int, d: int, scale: float,
                       causal: bool, num_splits: int = 0, stream=None) -> None:
    """C ``mha_fwd_kv_noalloc``: the split-KV forward on the library's built-in
    scratch buffer, for callers that cannot allocate device memory."""
    rc = lib().mha_fwd_kv_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(H),
                                  int(Nq), int(Nk), int(d), ctypes.c_float(scale), int(bool(causal)),
                                  int(num_splits), _stream(stream))
    if rc != MHA_OK:
        raise MhaError(rc, "mha_fwd_kv_noalloc")


def mha_fwd_paged(q, k_cache, v_cache, block_table, seq_lens, o, lse, B: int, H: int, Nq: int,
                  d: int, page_size: int, num_blocks: int, max_blocks: int, scale: float,
                  causal: bool, num_splits: int, workspace, workspace_bytes: int, stream=None) -> None:
    """C ``mha_fwd_paged``: tensors (or raw device addresses) in, status checked."""
    rc = lib().mha_fwd_paged(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seq_lens),
                             _ptr(o), _ptr(lse), int(B), int(H), int(Nq), int(d), int(page_size),
                             int(num_blocks), int(max_blocks), ctypes.c_float(scale),
                             int(bool(causal)), int(num_splits), _ptr(workspace), int(workspace_bytes),
                             _stream(stream))
    if rc != MHA_OK:
        raise MhaError(rc, "mha_fwd_paged")


def mha_bwd_workspace_size(B: int, H: int, N: int, d: int) -> int:
    return int(lib().mha_bwd_workspace_size(int(B), int(H), int(N), int(d)))


def mha_fwd_tile_order(B: int, H: int, N: int, d: int, causal: bool, sms: int) -> int:
    """C ``mha_fwd_tile_order``: 0 for the default work order, 1 for the
    head-major one, as mha_fwd would launch on a device with ``sms``
    multiprocessors (host only, no CUDA call)."""
    order = ctypes.c_int(-1)
    rc = lib().mha_fwd_tile_order(int(B), int(H), int(N), int(d), int(bool(causal)), int(sms),
                                  ctypes.byref(order))
    if rc != MHA_OK:
        raise MhaError(rc, "mha_fwd_tile_order")
    return int(order.value)


def mha_bwd(q, k, v, o, lse, dout, dq, dk, dv, B: int, H: int, N: int, d: int, scale: float,
            causal: bool, workspace, workspace_bytes: int, stream=None) -> None:
    """C ``mha_bwd``: tensors (or raw device addresses) in, status checked."""
    rc = lib().mha_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
                       _ptr(dv), int(B), int(H), int(N), int(d), ctypes.c_float(scale),
                       int(bool(causal)), _ptr(workspace), int(workspace_bytes), _stream(stream))
    if rc != MHA_OK:
        raise MhaError(rc, "mha_bwd")


def backward(q, k, v, o, lse, dout, causal: bool = False, scale: float | None = None, stream=None):
    """Allocate dQ, dK, dV and the workspace with torch and run ``mha_bwd``."""
    import torch
    B, H, N, d = q.shape
    if scale is None:
        scale = float(torch.tensor(d, dtype=torch.float32).rsqrt())
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws_bytes = mha_bwd_workspace_size(B, H, N, d)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=q.device)
    mha_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, scale, causal, ws, ws_bytes, stream)
    return dq, dk, dv
