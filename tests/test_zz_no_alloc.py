"""mha_fwd_kv_noalloc: the split-KV forward for callers that cannot allocate
device memory (they hold pointers to their own inputs and outputs but have
no way to obtain a workspace), running on the library's built-in scratch
buffer.  Its output must equal that of mha_fwd_kv with a caller-provided
workspace, on two calls in a row (the second one reuses the buffer the first
left behind): bit for bit with the same split plan.  This file is collected
last on purpose."""
import ctypes

import numpy as np
import pytest

import synth
from helpers import TOL_MAX_LSE, TOL_MAX_O, TOL_MEAN_O, bf16_to_f64, scale_for, to_device

pytestmark = pytest.mark.gpu


def _inputs(seed, B, H, Nq, Nk, d):
    q = synth.normal_bf16(seed, synth.STREAM_Q, B * H * Nq * d).reshape(B, H, Nq, d)
    k = synth.normal_bf16(seed, synth.STREAM_K, B * H * Nk * d).reshape(B, H, Nk, d)
    v = synth.normal_bf16(seed, synth.STREAM_V, B * H * Nk * d).reshape(B, H, Nk, d)
    return to_device(q), to_device(k), to_device(v), (q, k, v)


def test_no_alloc_matches_workspace_path_twice():
    """Both entry points run the same kernels on the same split plan, so the
    outputs must agree bit for bit; the first case is also held to the
    oracle.  A scratch-reuse fault that shifted results slightly would fail
    the bitwise check even where a tolerance would hide it."""
    import torch

    import head_attention_forward_gb300 as mha
    import oracle
    mha.build()
    L = mha.lib()
    stream = int(torch.cuda.current_stream().cuda_stream)
    # two calls in a row with different shapes: the second finds the first
    # call's partial results still in the shared buffer
    cases = [(2, 4, 1, 5000, 128, False, 0), (1, 3, 3, 777, 64, True, 0), (2, 4, 1, 5000, 128, False, 7)]
    for seed, (B, H, Nq, Nk, d, causal, splits) in enumerate(cases):
        q, k, v, bits = _inputs(90 + seed, B, H, Nq, Nk, d)
        scale = scale_for(d)
        # existing entry point with a workspace from torch
        o_ref = torch.full_like(q, float("nan"))
        l_ref = torch.full((B, H, Nq), float("nan"), dtype=torch.float32, device="cuda")
        ws_bytes = mha.mha_fwd_kv_workspace_size(B, H, Nq, Nk, d, splits)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        mha.mha_fwd_kv(q, k, v, o_ref, l_ref, B, H, Nq, Nk, d, scale, causal, splits, ws, ws_bytes)
        # the no-allocation entry point, called through the C ABI
        o = torch.full_like(q, float("nan"))
        lse = torch.full((B, H, Nq), float("nan"), dtype=torch.float32, device="cuda")
        rc = L.mha_fwd_kv_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                  lse.data_ptr(), B, H, Nq, Nk, d, ctypes.c_float(scale),
                                  int(causal), splits, stream)
        assert rc == mha.MHA_OK, mha.mha_strerror(rc)
        rc, word = mha.mha_device_status()
        assert rc == mha.MHA_OK, f"device status {word:#x}"
        a, b = bf16_to_f64(o), bf16_to_f64(o_ref)
        la, lb = lse.cpu().numpy(), l_ref.cpu().numpy()
        assert np.isfinite(a).all() and np.isfinite(la).all()
        assert np.array_equal(o.view(torch.int16).cpu().numpy(), o_ref.view(torch.int16).cpu().numpy())
        assert np.array_equal(la.view(np.uint32), lb.view(np.uint32))
        if seed == 0:
            o_or, l_or = oracle.attention_kv(*bits, scale, causal)
            do = np.abs(a - o_or)
            dl = np.abs(la.astype(np.float64) - l_or)
            assert do.max() <= TOL_MAX_O and do.mean() <= TOL_MEAN_O and dl.max() <= TOL_MAX_LSE


def test_no_alloc_rejects_problems_beyond_the_buffer():
    import head_attention_forward_gb300 as mha
    L = mha.lib()
    big = 1 << 40  # never dereferenced: the size check comes first
    B, H, Nq, Nk, d = 64, 64, 16, 4096, 128
    assert mha.mha_fwd_kv_workspace_size(B, H, Nq, Nk, d, 16) > (16 << 20)
    rc = L.mha_fwd_kv_noalloc(big, 2 * big, 3 * big, 4 * big, 5 * big, B, H, Nq, Nk, d,
                              ctypes.c_float(0.125), 0, 16, None)
    assert rc == mha.MHA_ERR_SCRATCH_LIMIT
