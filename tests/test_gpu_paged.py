"""GPU parity of the paged-KV path: random block tables and per-sequence
lengths, checked against the fp64 oracle on each sequence's gathered keys."""
import numpy as np
import pytest

import oracle
import synth
from helpers import TOL_MAX_LSE, TOL_MAX_O, TOL_MEAN_O, bf16_to_f64, scale_for, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import head_attention_forward_gb300 as mha
    mha.build()
    mha.lib()


def make_paged(seed, B, H, Nq, d, page, max_blocks, seq_lens, extra_blocks=3):
    """A paged cache holding each sequence's pages at shuffled block ids."""
    rng = np.random.default_rng(seed)
    pages_needed = [(int(n) + page - 1) // page for n in seq_lens]
    num_blocks = sum(pages_needed) + extra_blocks
    perm = rng.permutation(num_blocks)
    table = np.full((B, max_blocks), -1, dtype=np.int32)  # unused entries: out of range
    nxt = 0
    for b in range(B):
        for i in range(pages_needed[b]):
            table[b, i] = perm[nxt]
            nxt += 1
    kc = synth.normal_bf16(seed, synth.STREAM_K, num_blocks * H * page * d).reshape(num_blocks, H, page, d)
    vc = synth.normal_bf16(seed, synth.STREAM_V, num_blocks * H * page * d).reshape(num_blocks, H, page, d)
    q = synth.normal_bf16(seed, synth.STREAM_Q, B * H * Nq * d).reshape(B, H, Nq, d)
    return q, kc, vc, table, num_blocks


def gather(kc, table, b, n, page):
    """Keys 0..n-1 of batch entry b as a contiguous [H, n, d] array."""
    rows = [kc[table[b, t // page], :, t % page] for t in range(n)]
    return np.ascontiguousarray(np.stack(rows, axis=1))


@pytest.mark.parametrize("page", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d,Nq", [(128, 1), (128, 16), (64, 4), (64, 2)])
def test_paged_against_oracle(page, causal, d, Nq):
    import torch

    import head_attention_forward_gb300 as mha
    B, H = 3, 2
    max_blocks = (700 + page - 1) // page + 1
    seq_lens = np.array([1, 333, 700], dtype=np.int32)[:B]
    q, kc, vc, table, nb = make_paged(40 + page + d, B, H, Nq, d, page, max_blocks, seq_lens)
    scale = scale_for(d)
    qd, kd, vd = to_device(q), to_device(kc), to_device(vc)
    td = torch.from_numpy(table).cuda()
    sd = torch.from_numpy(seq_lens).cuda()
    o = torch.full_like(qd, float("nan"))
    lse = torch.full((B, H, Nq), float("nan"), dtype=torch.float32, device="cuda")
    ws_bytes = mha.mha_fwd_kv_workspace_size(B, H, Nq, max_blocks * page, d, 0)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    mha.mha_fwd_paged(qd, kd, vd, td, sd, o, lse, B, H, Nq, d, page, nb, max_blocks, scale, causal, 0,
                      ws, ws_bytes)
    rc, word = mha.mha_device_status()
    assert rc == mha.MHA_OK, f"status {word:#x}"
    og, lg = bf16_to_f64(o), lse.cpu().numpy().astype(np.float64)
    for b in range(B):
        n = int(seq_lens[b])
        kb, vb = gather(kc, table, b, n, page), gather(vc, table, b, n, page)
        o_ref, l_ref = oracle.attention_kv(q[b:b + 1], kb[None], vb[None], scale, causal)
        empty = np.isneginf(l_ref[0])
        assert np.array_equal(np.isneginf(lg[b]), empty)
        assert np.all(og[b][empty] == 0)
        do = np.abs(og[b] - o_ref[0])
        dl = np.abs(lg[b][~empty] - l_ref[0][~empty]) if (~empty).any() else np.zeros(1)
        assert do.max() <= TOL_MAX_O and do.mean() <= TOL_MEAN_O and dl.max() <= TOL_MAX_LSE, \
            (b, do.max(), do.mean(), dl.max())


@pytest.mark.parametrize("d,Nq,page", [(64, 2, 64), (128, 1, 64), (128, 4, 128), (64, 8, 16)])
def test_paged_equals_contiguous_when_identity(d, Nq, page):
    """An identity block table over a cache laid out like [B*H...] gives the
    same result, bit for bit, as the contiguous split-KV entry point: both
    run the same partial pass with the same splits, and the 600-key
    sequences end inside a page, where the paged pass clears the rows past
    the end that the contiguous one reads as zeros."""
    import torch

    import head_attention_forward_gb300 as mha
    B, H, n = 2, 2, 600
    mb = (n + page - 1) // page
    q = synth.normal_bf16(3, 0, B * H * Nq * d).reshape(B, H, Nq, d)
    k = synth.normal_bf16(3, 1, B * H * n * d).reshape(B, H, n, d)
    v = synth.normal_bf16(3, 2, B * H * n * d).reshape(B, H, n, d)
    pad = np.zeros((B, H, mb * page - n, d), dtype=k.dtype)
    kp, vp = np.concatenate([k, pad], axis=2), np.concatenate([v, pad], axis=2)
    # cache block (b * mb + i) holds keys i*page.. of entry b, all heads
    kc = np.ascontiguousarray(kp.reshape(B, H, mb, page, d).transpose(0, 2, 1, 3, 4).reshape(B * mb, H, page, d))
    vc = np.ascontiguousarray(vp.reshape(B, H, mb, page, d).transpose(0, 2, 1, 3, 4).reshape(B * mb, H, page, d))
    table = np.arange(B * mb, dtype=np.int32).reshape(B, mb)
    seq = np.full(B, n, dtype=np.int32)
    scale = scale_for(d)
    ws_bytes = max(mha.mha_fwd_kv_workspace_size(B, H, Nq, n, d, 3),
                   mha.mha_fwd_kv_workspace_size(B, H, Nq, mb * page, d, 3))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    o1 = torch.empty((B, H, Nq, d), dtype=torch.bfloat16, device="cuda")
    l1 = torch.empty((B, H, Nq), dtype=torch.float32, device="cuda")
    mha.mha_fwd_paged(to_device(q), to_device(kc), to_device(vc), torch.from_numpy(table).cuda(),
                      torch.from_numpy(seq).cuda(), o1, l1, B, H, Nq, d, page, B * mb, mb, scale, True,
                      3, ws, ws_bytes)
    o2 = torch.empty_like(o1)
    l2 = torch.empty_like(l1)
    mha.mha_fwd_kv(to_device(q), to_device(k), to_device(v), o2, l2, B, H, Nq, n, d, scale, True, 3,
                   ws, ws_bytes)
    rc, word = mha.mha_device_status()
    assert rc == mha.MHA_OK, f"status {word:#x}"
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("page", [16, 64, 256])
@pytest.mark.parametrize("d,Nq,causal", [(128, 1, False), (128, 2, True), (64, 1, False), (64, 2, True)])
def test_paged_nan_outside_sequences(page, d, Nq, causal):
    """Every cache row outside the sequences' keys holds NaN: the rest of
    each sequence's last page, the unused pages, and the rows the table
    entries past each length point at.  None of it may reach O or LSE.  A
    zero-length sequence gives O = 0 and LSE = -inf."""
    import torch

    import head_attention_forward_gb300 as mha
    B, H = 4, 2
    max_blocks = (700 + page - 1) // page + 1
    seq = np.array([0, 1, 333, 700], dtype=np.int32)
    q, kc, vc, table, nb = make_paged(90 + page + d, B, H, Nq, d, page, max_blocks, seq)
    nan = np.uint16(0x7FC0)  # bf16 quiet NaN
    live = np.zeros((nb, page), dtype=bool)
    for b in range(B):
        for t in range(int(seq[b])):
            live[table[b, t // page], t % page] = True
    kn, vn = kc.copy(), vc.copy()
    kn[~live[:, None, :].repeat(H, axis=1)] = nan
    vn[~live[:, None, :].repeat(H, axis=1)] = nan
    # table entries past each length point at real (NaN-filled) blocks
    spare = [blk for blk in range(nb) if not live[blk].any()]
    for b in range(B):
        used = (int(seq[b]) + page - 1) // page
        for i in range(used, max_blocks):
            table[b, i] = spare[(b + i) % len(spare)]
    scale = scale_for(d)
    o = torch.full((B, H, Nq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, H, Nq), float("nan"), dtype=torch.float32, device="cuda")
    ws_bytes = mha.mha_fwd_kv_workspace_size(B, H, Nq, max_blocks * page, d, 0)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    mha.mha_fwd_paged(to_device(q), to_device(kn), to_device(vn), torch.from_numpy(table).cuda(),
                      torch.from_numpy(seq).cuda(), o, lse, B, H, Nq, d, page, nb, max_blocks, scale,
                      causal, 0, ws, ws_bytes)
    rc, word = mha.mha_device_status()
    assert rc == mha.MHA_OK, f"status {word:#x}"
    og, lg = bf16_to_f64(o), lse.cpu().numpy().astype(np.float64)
    assert np.all(og[0] == 0) and np.all(np.isneginf(lg[0]))
    assert np.isfinite(og).all()
    for b in range(1, B):
        n = int(seq[b])
        kb, vb = gather(kc, table, b, n, page), gather(vc, table, b, n, page)
        o_ref, l_ref = oracle.attention_kv(q[b:b + 1], kb[None], vb[None], scale, causal)
        empty = np.isneginf(l_ref[0])
        assert np.array_equal(np.isneginf(lg[b]), empty)
        do = np.abs(og[b] - o_ref[0])
        dl = np.abs(lg[b][~empty] - l_ref[0][~empty]) if (~empty).any() else np.zeros(1)
        assert do.max() <= TOL_MAX_O and do.mean() <= TOL_MEAN_O and dl.max() <= TOL_MAX_LSE, \
            (b, do.max(), do.mean(), dl.max())


def gather_or_zero(kc, table, b, n, page, num_blocks):
    """Like gather(), but a block id outside [0, num_blocks) reads as zeros."""
    H, d = kc.shape[1], kc.shape[3]
    out = np.zeros((H, n, d), dtype=kc.dtype)
    for t in range(n):
        blk = table[b, t // page]
        if 0 <= blk < num_blocks:
            out[:, t] = kc[blk, :, t % page]
    return out


@pytest.mark.parametrize("page", [32, 256])
def test_paged_odd_tables(page):
    """Repeated block ids, ids outside the cache (read as zeros) and a length
    beyond the table (clamped to max_blocks * page)."""
    import torch

    import head_attention_forward_gb300 as mha
    B, H, Nq, d = 3, 2, 2, 128
    max_blocks = 6
    num_blocks = 8
    rng = np.random.default_rng(page)
    table = rng.integers(0, num_blocks, size=(B, max_blocks)).astype(np.int32)
    table[0, 1] = table[0, 3]            # one physical block used twice
    table[1, 2] = num_blocks + 5         # past the cache
    table[1, 4] = -3                     # negative
    table[2, 5] = 1 << 30                # far past the cache
    seq = np.array([max_blocks * page - 5, 5 * page + 7, max_blocks * page + 100], dtype=np.int32)
    kc = synth.normal_bf16(70 + page, synth.STREAM_K, num_blocks * H * page * d).reshape(num_blocks, H, page, d)
    vc = synth.normal_bf16(70 + page, synth.STREAM_V, num_blocks * H * page * d).reshape(num_blocks, H, page, d)
    q = synth.normal_bf16(70 + page, synth.STREAM_Q, B * H * Nq * d).reshape(B, H, Nq, d)
    scale = scale_for(d)
    o = torch.full((B, H, Nq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, H, Nq), float("nan"), dtype=torch.float32, device="cuda")
    ws_bytes = mha.mha_fwd_kv_workspace_size(B, H, Nq, max_blocks * page, d, 0)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    mha.mha_fwd_paged(to_device(q), to_device(kc), to_device(vc), torch.from_numpy(table).cuda(),
                      torch.from_numpy(seq).cuda(), o, lse, B, H, Nq, d, page, num_blocks, max_blocks,
                      scale, False, 0, ws, ws_bytes)
    rc, word = mha.mha_device_status()
    assert rc == mha.MHA_OK, f"status {word:#x}"
    og, lg = bf16_to_f64(o), lse.cpu().numpy().astype(np.float64)
    for b in range(B):
        n = min(int(seq[b]), max_blocks * page)
        kb = gather_or_zero(kc, table, b, n, page, num_blocks)
        vb = gather_or_zero(vc, table, b, n, page, num_blocks)
        o_ref, l_ref = oracle.attention_kv(q[b:b + 1], kb[None], vb[None], scale, False)
        do = np.abs(og[b] - o_ref[0])
        dl = np.abs(lg[b] - l_ref[0])
        assert do.max() <= TOL_MAX_O and do.mean() <= TOL_MEAN_O and dl.max() <= TOL_MAX_LSE, \
            (b, do.max(), do.mean(), dl.max())


def test_paged_full_workload_sampled():
    """The whole 32-sequence, 64-key-page decode workload in one call; a few
    (sequence, head) rows checked against the oracle."""
    import torch

    import head_attention_forward_gb300 as mha
    qb, kcb, vcb, table, seq = synth.paged_inputs("pag2")
    c = synth.PAGED_CONFIGS["pag2"]
    B, H, Nq, d, page = c["B"], c["H"], c["Nq"], c["d"], c["page"]
    num_blocks, max_blocks = kcb.shape[0], table.shape[1]
    scale = scale_for(d)
    o = torch.full((B, H, Nq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, H, Nq), float("nan"), dtype=torch.float32, device="cuda")
    ws_bytes = mha.mha_fwd_kv_workspace_size(B, H, Nq, max_blocks * page, d, 0)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    mha.mha_fwd_paged(to_device(qb), to_device(kcb), to_device(vcb), torch.from_numpy(table).cuda(),
                      torch.from_numpy(seq).cuda(), o, lse, B, H, Nq, d, page, num_blocks, max_blocks,
                      scale, False, 0, ws, ws_bytes)
    rc, word = mha.mha_device_status()
    assert rc == mha.MHA_OK, f"status {word:#x}"
    og, lg = bf16_to_f64(o), lse.cpu().numpy().astype(np.float64)
    assert np.isfinite(og).all() and np.isfinite(lg).all()
    for b in (0, 7, 31):
        n = int(seq[b])
        kb, vb = gather(kcb, table, b, n, page), gather(vcb, table, b, n, page)
        for h in (0, 17, 31):
            o_ref, l_ref = oracle.attention_kv(qb[b:b + 1, h:h + 1], kb[None, h:h + 1], vb[None, h:h + 1],
                                               scale, False)
            do = np.abs(og[b, h] - o_ref[0, 0])
            dl = np.abs(lg[b, h] - l_ref[0, 0])
            assert do.max() <= TOL_MAX_O and dl.max() <= TOL_MAX_LSE, (b, h, do.max(), dl.max())
