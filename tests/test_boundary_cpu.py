"""The C ABI on a machine without a GPU: the library loads, exports every
entry point include/mha_fwd.h declares, and rejects bad arguments before
any CUDA call."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mha_fwd.h")


@pytest.fixture(scope="module")
def L():
    import head_attention_forward_gb300 as mha
    mha.build()
    return mha.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(mha_\w+)\s*\(", text, flags=re.M)


def test_header_declares_entry_points():
    names = declared_functions()
    assert {"mha_fwd", "mha_strerror", "mha_device_status", "mha_set_wait_limit",
            "mha_wait_selftest"} <= set(names)


def test_every_declared_symbol_is_exported(L):
    import head_attention_forward_gb300 as mha
    out = subprocess.run(["nm", "-D", "--defined-only", mha.LIB], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in declared_functions():
        assert name in exported, name
        getattr(L, name)


def test_no_driver_dependency():
    import head_attention_forward_gb300 as mha
    out = subprocess.run(["ldd", mha.LIB], capture_output=True, text=True).stdout
    assert "libcuda.so" not in out


def _fwd(L, q=16, k=32, v=48, o=64, lse=80, B=1, H=1, N=4, d=64, scale=0.125, causal=0):
    return L.mha_fwd(q, k, v, o, lse, B, H, N, d, ctypes.c_float(scale), causal, None)


def test_argument_checks(L):
    import head_attention_forward_gb300 as mha
    big = 1 << 40  # far-apart fake addresses; never dereferenced
    ok = dict(q=big, k=2 * big, v=3 * big, o=4 * big, lse=5 * big)
    assert _fwd(L, **ok, d=96) == mha.MHA_ERR_UNSUPPORTED_DIM
    assert _fwd(L, **ok, d=0) == mha.MHA_ERR_UNSUPPORTED_DIM
    assert _fwd(L, **ok, B=-1) == mha.MHA_ERR_INVALID_ARG
    assert _fwd(L, **ok, N=-5) == mha.MHA_ERR_INVALID_ARG
    assert _fwd(L, **ok, scale=0.0) == mha.MHA_ERR_INVALID_ARG
    assert _fwd(L, **ok, scale=float("inf")) == mha.MHA_ERR_INVALID_ARG
    assert _fwd(L, **ok, scale=float("nan")) == mha.MHA_ERR_INVALID_ARG
    assert _fwd(L, **dict(ok, q=0)) == mha.MHA_ERR_INVALID_ARG
    assert _fwd(L, **dict(ok, lse=0)) == mha.MHA_ERR_INVALID_ARG
    assert _fwd(L, **dict(ok, k=2 * big + 8)) == mha.MHA_ERR_MISALIGNED
    assert _fwd(L, **dict(ok, o=big)) == mha.MHA_ERR_INVALID_ARG  # o aliases q
    assert _fwd(L, **dict(ok, lse=2 * big + 64)) == mha.MHA_ERR_INVALID_ARG  # lse inside k
    # sizes past the int counters (far beyond any device memory)
    assert _fwd(L, **ok, B=1 << 16, H=1 << 16) == mha.MHA_ERR_INVALID_ARG  # B*H > INT_MAX
    assert _fwd(L, **ok, B=1 << 15, H=1 << 15, N=257) == mha.MHA_ERR_INVALID_ARG  # 2^31 work tiles
    # empty problems return before any CUDA call
    assert _fwd(L, **ok, N=0) == mha.MHA_OK
    assert _fwd(L, **ok, B=0) == mha.MHA_OK
    assert _fwd(L, q=0, k=0, v=0, o=0, lse=0, H=0) == mha.MHA_OK


def test_other_entry_points_validate(L):
    import head_attention_forward_gb300 as mha
    assert L.mha_set_wait_limit(0) == mha.MHA_ERR_INVALID_ARG
    assert L.mha_set_wait_limit(-3) == mha.MHA_ERR_INVALID_ARG
    assert L.mha_wait_selftest(0, None) == mha.MHA_ERR_INVALID_ARG
    for s in range(0, 8):
        assert isinstance(mha.mha_strerror(s), str) and mha.mha_strerror(s)


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    import head_attention_forward_gb300._binding as b
    monkeypatch.setattr(b, "LIB", str(tmp_path / "missing.so"))
    monkeypatch.setattr(b, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        b.lib()


def test_kv_workspace_size_is_pure():
    import head_attention_forward_gb300 as mha
    a = mha.mha_fwd_kv_workspace_size(2, 8, 1, 32768, 128, 0)
    assert a > 0 and a == mha.mha_fwd_kv_workspace_size(2, 8, 1, 32768, 128, 0)
    # explicit split count: two fp32 partials per split (o_part, then the
    # 16-byte aligned lse_part) + the 16-byte slot of the work-tile counter
    assert mha.mha_fwd_kv_workspace_size(1, 1, 4, 1000, 64, 2) == 2 * 2 * 4 * 64 * 4 + 2 * 2 * 4 * 4 + 16
    assert mha.mha_fwd_kv_workspace_size(1, 1, 17, 100, 64, 0) == 0   # Nq > 16
    assert mha.mha_fwd_kv_workspace_size(1, 1, 1, 100, 96, 0) == 0    # bad d
    assert mha.mha_fwd_kv_workspace_size(0, 1, 1, 100, 64, 0) == 0    # empty


def _kv_workspace(B, H, Nq, Nk, d, splits):
    """Workspace bytes for a given split count: o_part fp32 [B*H, 2*splits,
    Nq, d], lse_part fp32 [B*H, 2*splits, Nq] (16-byte aligned), then the
    16-byte counter slot."""
    o = B * H * 2 * splits * Nq * d * 4
    lse = B * H * 2 * splits * Nq * 4
    return (o + 15) // 16 * 16 + (lse + 15) // 16 * 16 + 16


@pytest.mark.parametrize("shape,splits", [
    # one wave: fewer heads than the 152 SMs, at most 64 K/V tiles per SM and
    # splits filling >= 4/5 of the SMs; floor(152 / (B*H)) splits, rounded so
    # that each split has an even number of 128-key tiles
    ((1, 32, 1, 4096, 128), 4),     # 32 tiles: 4 splits of 8
    ((1, 8, 1, 16384, 128), 16),    # 19 splits would be 7 tiles each: 8 -> 16 splits
    ((4, 8, 4, 8192, 64), 4),
    ((1, 16, 1, 32768, 128), 9),    # 256 tiles: 9 splits of 30 (29 rounded up)
    ((1, 151, 1, 8192, 128), 1),
    ((1, 1, 1, 300, 128), 3),       # 3 tiles: one per split
    # six work tiles per SM: ceil(912 / (B*H)) splits
    ((4, 32, 1, 16384, 128), 8),    # ~108 tiles per SM
    ((1, 100, 1, 4096, 128), 8),    # 100 heads leave a third of the SMs idle in one wave
    ((8, 32, 1, 32768, 128), 4),    # 256 heads: more heads than SMs
    ((1, 32, 4, 131072, 128), 29),  # 1024 tiles per head, ~216 per SM
])
def test_kv_split_plan(shape, splits):
    """The automatic split count, seen through the workspace size."""
    import head_attention_forward_gb300 as mha
    assert mha.mha_fwd_kv_workspace_size(*shape, 0) == _kv_workspace(*shape, splits)
    assert mha.mha_fwd_kv_workspace_size(*shape, splits) == _kv_workspace(*shape, splits)


def test_kv_argument_checks(L):
    import head_attention_forward_gb300 as mha
    big = 1 << 40
    args = dict(q=big, k=2 * big, v=3 * big, o=4 * big, lse=5 * big, B=1, H=1, Nq=1, Nk=100,
                d=64, scale=0.125, causal=0, splits=0, ws=6 * big, wsb=1 << 20)

    def call(**kw):
        a = dict(args, **kw)
        return L.mha_fwd_kv(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["Nq"],
                            a["Nk"], a["d"], ctypes.c_float(a["scale"]), a["causal"], a["splits"],
                            a["ws"], a["wsb"], None)
    assert call(d=96) == mha.MHA_ERR_UNSUPPORTED_DIM
    assert call(Nq=17) == mha.MHA_ERR_INVALID_ARG
    assert call(Nk=0) == mha.MHA_ERR_INVALID_ARG
    assert call(splits=-1) == mha.MHA_ERR_INVALID_ARG
    assert call(ws=0) == mha.MHA_ERR_INVALID_ARG
    assert call(wsb=16) == mha.MHA_ERR_INVALID_ARG            # workspace too small
    assert call(ws=6 * big + 4) == mha.MHA_ERR_MISALIGNED
    assert call(ws=2 * big) == mha.MHA_ERR_INVALID_ARG        # workspace over k
    assert call(scale=-1.0) == mha.MHA_ERR_INVALID_ARG
    assert call(Nq=0) == mha.MHA_OK and call(B=0) == mha.MHA_OK


def test_paged_argument_checks(L):
    import head_attention_forward_gb300 as mha
    big = 1 << 40
    a = dict(q=big, kc=2 * big, vc=3 * big, bt=4 * big, sl=5 * big, o=6 * big, lse=7 * big, B=1,
             H=1, Nq=1, d=64, page=64, nb=10, mb=4, scale=0.125, causal=0, splits=0, ws=8 * big,
             wsb=1 << 20)

    def call(**kw):
        x = dict(a, **kw)
        return L.mha_fwd_paged(x["q"], x["kc"], x["vc"], x["bt"], x["sl"], x["o"], x["lse"], x["B"],
                               x["H"], x["Nq"], x["d"], x["page"], x["nb"], x["mb"],
                               ctypes.c_float(x["scale"]), x["causal"], x["splits"], x["ws"], x["wsb"],
                               None)
    assert call(page=48) == mha.MHA_ERR_INVALID_ARG
    assert call(page=8) == mha.MHA_ERR_INVALID_ARG
    assert call(page=512) == mha.MHA_ERR_INVALID_ARG
    assert call(mb=0) == mha.MHA_ERR_INVALID_ARG
    assert call(nb=0) == mha.MHA_ERR_INVALID_ARG
    assert call(nb=1 << 30, H=2) == mha.MHA_ERR_INVALID_ARG   # block * H + head overflows int
    assert call(bt=0) == mha.MHA_ERR_INVALID_ARG
    assert call(bt=4 * big + 2) == mha.MHA_ERR_MISALIGNED
    assert call(d=80) == mha.MHA_ERR_UNSUPPORTED_DIM
    assert call(wsb=8) == mha.MHA_ERR_INVALID_ARG
    assert call(Nq=0) == mha.MHA_OK


def test_bwd_workspace_size_is_pure():
    import head_attention_forward_gb300 as mha
    assert mha.mha_bwd_workspace_size(2, 3, 100, 128) == (2 * 3 * 100 * 4 + 15) // 16 * 16
    assert mha.mha_bwd_workspace_size(1, 1, 7, 64) == 32
    assert mha.mha_bwd_workspace_size(1, 1, 7, 96) == 0
    assert mha.mha_bwd_workspace_size(-1, 1, 7, 64) == 0
    assert mha.mha_bwd_workspace_size(0, 1, 7, 64) == 0


def test_bwd_argument_checks(L):
    import head_attention_forward_gb300 as mha
    big = 1 << 40
    a = dict(q=big, k=2 * big, v=3 * big, o=4 * big, lse=5 * big, do=6 * big, dq=7 * big,
             dk=8 * big, dv=9 * big, B=1, H=2, N=100, d=64, scale=0.125, causal=1, ws=10 * big,
             wsb=1 << 20)

    def call(**kw):
        x = dict(a, **kw)
        return L.mha_bwd(x["q"], x["k"], x["v"], x["o"], x["lse"], x["do"], x["dq"], x["dk"],
                         x["dv"], x["B"], x["H"], x["N"], x["d"], ctypes.c_float(x["scale"]),
                         x["causal"], x["ws"], x["wsb"], None)
    assert call(d=96) == mha.MHA_ERR_UNSUPPORTED_DIM
    assert call(N=-1) == mha.MHA_ERR_INVALID_ARG
    assert call(scale=0.0) == mha.MHA_ERR_INVALID_ARG
    assert call(do=0) == mha.MHA_ERR_INVALID_ARG
    assert call(ws=0) == mha.MHA_ERR_INVALID_ARG
    assert call(dk=8 * big + 8) == mha.MHA_ERR_MISALIGNED
    assert call(wsb=16) == mha.MHA_ERR_INVALID_ARG             # workspace too small
    assert call(dq=big) == mha.MHA_ERR_INVALID_ARG             # dq over q
    assert call(dv=7 * big) == mha.MHA_ERR_INVALID_ARG         # dv over dq
    assert call(ws=9 * big) == mha.MHA_ERR_INVALID_ARG         # workspace over dv
    assert call(N=0) == mha.MHA_OK and call(B=0) == mha.MHA_OK


@pytest.mark.parametrize("shape,order", [
    ((1, 2, 128, 64, False), 0), ((16, 16, 512, 64, False), 0), ((4, 16, 2048, 64, True), 0),
    ((2, 32, 4096, 128, False), 1),   # 128 MiB of K/V, 1024 equal tiles fill 96% of 7 rounds
    ((2, 32, 4096, 128, True), 0),    # 512 equal pairs would fill only 84% of 4 rounds
    ((1, 32, 16384, 128, True), 1),   # 256 MiB, 1024 pairs: 96%
    ((1, 32, 16603, 128, True), 1),   # odd m-block count: 1056 items, 7 rounds, 99%
    ((2, 32, 4000, 128, False), 1),
    ((1, 32, 16384, 64, True), 0),    # d = 64 always takes the default order
    ((1, 8, 4096, 128, True), 0),     # 32 MiB of K/V fits in L2
])
def test_fwd_tile_order(L, shape, order):
    """The work order mha_fwd chooses, from the host-only query."""
    import head_attention_forward_gb300 as mha
    B, H, N, d, causal = shape
    assert mha.mha_fwd_tile_order(B, H, N, d, causal, 152) == order


def test_fwd_tile_order_argument_checks(L):
    import head_attention_forward_gb300 as mha
    out = ctypes.c_int(7)
    assert L.mha_fwd_tile_order(1, 1, 8, 96, 0, 152, ctypes.byref(out)) == mha.MHA_ERR_UNSUPPORTED_DIM
    assert L.mha_fwd_tile_order(-1, 1, 8, 64, 0, 152, ctypes.byref(out)) == mha.MHA_ERR_INVALID_ARG
    assert L.mha_fwd_tile_order(1, 1, 8, 64, 0, 0, ctypes.byref(out)) == mha.MHA_ERR_INVALID_ARG
    assert L.mha_fwd_tile_order(1, 1, 8, 64, 0, 152, None) == mha.MHA_ERR_INVALID_ARG
    assert L.mha_fwd_tile_order(0, 1, 8, 128, 1, 152, ctypes.byref(out)) == mha.MHA_OK and out.value == 0
    # the sizes mha_fwd rejects (2^31 work tiles)
    assert L.mha_fwd_tile_order(1 << 15, 1 << 15, 257, 128, 1, 152, ctypes.byref(out)) == mha.MHA_ERR_INVALID_ARG
