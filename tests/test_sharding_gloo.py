"""The multi-rank split of the attention path, run as two gloo ranks on the
CPU: each rank computes its own contiguous slice of the B*H axis (with the
fp64 oracle standing in for the kernel, which needs a GPU); gathering the
slices afterwards - for checking only - must reproduce the single-process
result exactly."""
import os
import socket

import numpy as np
import pytest

from head_attention_forward_gb300.sharding import head_slice, replica_seed


def test_head_slice_covers_once():
    for heads in (0, 1, 5, 64, 131):
        for world in (1, 2, 3, 8):
            spans = [head_slice(heads, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == heads
            for (a, b), (c, d) in zip(spans, spans[1:]):
                assert b == c
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        head_slice(4, 2, 2)


def test_replica_seeds_distinct():
    assert len({replica_seed(4, r) for r in range(8)}) == 8


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist

    import oracle
    import synth
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    B, H, N, d = 1, 5, 40, 16
    q, k, v = synth.qkv(21, B, H, N, d, compiled=False)
    lo, hi = head_slice(B * H, world, rank)
    qs = q.reshape(B * H, 1, N, d)[lo:hi].reshape(1, hi - lo, N, d)
    ks = k.reshape(B * H, 1, N, d)[lo:hi].reshape(1, hi - lo, N, d)
    vs = v.reshape(B * H, 1, N, d)[lo:hi].reshape(1, hi - lo, N, d)
    o, lse = oracle.attention_fwd(qs, ks, vs, 0.25, True, nthreads=1)
    got = [None] * world
    dist.all_gather_object(got, (lo, hi, o, lse))  # checking only
    if rank == 0:
        np.save(os.path.join(out_dir, "o.npy"), np.concatenate([g[2] for g in got], axis=1))
        np.save(os.path.join(out_dir, "lse.npy"), np.concatenate([g[3] for g in got], axis=1))
        np.save(os.path.join(out_dir, "spans.npy"), np.array([(g[0], g[1]) for g in got]))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_reassemble(tmp_path):
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp

    import oracle
    import synth
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    B, H, N, d = 1, 5, 40, 16
    q, k, v = synth.qkv(21, B, H, N, d, compiled=False)
    o_ref, lse_ref = oracle.attention_fwd(q, k, v, 0.25, True, nthreads=1)
    assert np.array_equal(np.load(tmp_path / "o.npy"), o_ref)
    assert np.array_equal(np.load(tmp_path / "lse.npy"), lse_ref)
    spans = np.load(tmp_path / "spans.npy")
    assert spans.tolist() == [[0, 3], [3, 5]]
