"""Calls on different streams at the same time: the forward and split-KV
entry points keep no state between launches (tensor maps go by value, the
split pass's counter lives in the caller's workspace), so concurrent calls
give the bits of serial ones."""
import numpy as np
import pytest

import synth
from helpers import scale_for, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import head_attention_forward_gb300 as mha
    mha.build()
    mha.lib()


def test_concurrent_streams_match_serial_calls():
    import torch

    import head_attention_forward_gb300 as mha
    jobs = []
    # (B, H, N, d, causal, tile order): both head dimensions, both masks,
    # both tile orders
    for i, (B, H, N, d, causal, order) in enumerate([(2, 8, 1500, 64, True, 0), (1, 16, 3000, 128, False, 0),
                                                     (4, 4, 700, 128, True, 0), (1, 32, 16384, 128, True, 1)]):
        assert mha.mha_fwd_tile_order(B, H, N, d, causal, 152) == order
        q, k, v = (to_device(a) for a in synth.qkv(70 + i, B, H, N, d))
        jobs.append(("fwd", (B, H, N, d, causal), q, k, v))
    for i, (B, H, Nq, Nk, d, causal) in enumerate([(2, 8, 4, 5000, 128, True), (4, 4, 1, 9000, 64, False)]):
        q = to_device(synth.normal_bf16(80 + i, 0, B * H * Nq * d).reshape(B, H, Nq, d))
        k = to_device(synth.normal_bf16(80 + i, 1, B * H * Nk * d).reshape(B, H, Nk, d))
        v = to_device(synth.normal_bf16(80 + i, 2, B * H * Nk * d).reshape(B, H, Nk, d))
        jobs.append(("kv", (B, H, Nq, Nk, d, causal), q, k, v))

    def outputs(job):
        kind, shape, q, k, v = job
        o = torch.full_like(q, float("nan"))
        lse = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device="cuda")
        ws = None
        if kind == "kv":
            B, H, Nq, Nk, d, causal = shape
            nbytes = mha.mha_fwd_kv_workspace_size(B, H, Nq, Nk, d, 0)
            ws = (torch.full((nbytes,), 0xFF, dtype=torch.uint8, device="cuda"), nbytes)
        return o, lse, ws

    def launch(job, o, lse, ws, stream):
        kind, shape, q, k, v = job
        sptr = int(stream.cuda_stream)
        if kind == "fwd":
            B, H, N, d, causal = shape
            mha.mha_fwd(q, k, v, o, lse, B, H, N, d, scale_for(d), causal, sptr)
        else:
            B, H, Nq, Nk, d, causal = shape
            mha.mha_fwd_kv(q, k, v, o, lse, B, H, Nq, Nk, d, scale_for(d), causal, 0, ws[0], ws[1], sptr)

    main = torch.cuda.current_stream()
    serial = []
    for job in jobs:
        o, lse, ws = outputs(job)
        launch(job, o, lse, ws, main)
        serial.append((o, lse))
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in jobs]
    for rep in range(3):
        outs = [outputs(job) for job in jobs]
        torch.cuda.synchronize()
        for job, (o, lse, ws), st in zip(jobs, outs, streams):
            launch(job, o, lse, ws, st)
        torch.cuda.synchronize()
        rc, word = mha.mha_device_status()
        assert rc == mha.MHA_OK, f"device status {rc} word {word:#x}"
        for (o, lse, _), (o_ref, l_ref), job in zip(outs, serial, jobs):
            assert torch.equal(o, o_ref) and torch.equal(lse, l_ref), (rep, job[0], job[1])
