"""The benchmark's host-side bookkeeping, without a GPU: FLOP counting, the
roofline denominator rule, the clock record, the traffic records' validity
and the config object both arms print."""
import json
import os

import pytest

import bench
import synth


def test_counted_flops_follow_the_metric():
    # 4 B H N^2 d, halved under the causal mask
    assert bench.counted_flops(synth.CONFIGS["cfg5"]) == 4.0 * 1 * 32 * 16384 * 16384 * 128 / 2
    assert bench.counted_flops(synth.CONFIGS["cfg4a"]) == 4.0 * 2 * 32 * 4096 * 4096 * 128
    assert bench.counted_flops(synth.CONFIGS["cfg4b"]) == bench.counted_flops(synth.CONFIGS["cfg4a"]) / 2


def test_peak_follows_the_timed_region(monkeypatch):
    monkeypatch.setattr(bench, "load_peaks", lambda: (1700.0, 1900.0, "test"))
    assert bench.pick_peak(0.7)[0] == 1900.0  # under a second: the burst figure
    assert bench.pick_peak(bench.BURST_REGION_S)[0] == 1700.0
    assert bench.pick_peak(5.0)[0] == 1700.0


def test_clock_record_merges_reasons():
    nv = {"sm_mhz": 1950.0, "reasons": ["sw_power_cap"], "samples": 40}
    smi = {"sm_mhz": 1940.0, "reasons": ["hw_slowdown"], "samples": 2}
    out = bench.merge_clocks(nv, smi)
    assert out["sm_mhz"] == 1950.0 and out["samples"] == 40
    assert out["reasons"] == ["hw_slowdown", "sw_power_cap"]
    assert out["nvidia_smi"] == smi
    assert bench.merge_clocks(None, smi) == smi


def test_recorded_traffic_is_dropped_when_the_kernel_changes(tmp_path, monkeypatch):
    rec = {"cfg5": {"kernel_family": "mha_fwd_kernel", "dram_bytes_per_launch": 123,
                    "kernel_source_hash": bench.kernel_source_hash("mha_fwd_kernel")},
           "cfg4a": {"kernel_family": "mha_fwd_kernel", "dram_bytes_per_launch": 456,
                     "kernel_source_hash": "0" * 16}}
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "ncu_traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda k: rec["cfg5"]["kernel_source_hash"])
    assert bench.recorded_traffic("cfg5") == 123
    assert bench.recorded_traffic("cfg4a") is None  # taken on another source
    assert bench.recorded_traffic("cfg2") is None   # no record


def test_source_hash_ignores_comments(tmp_path, monkeypatch):
    csrc = tmp_path / "head_attention_forward_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for fn in bench.KERNEL_SOURCES["mha_fwd_kernel"]:
        (csrc / fn).write_text("int a = 1;  // one\n\nint b = 2;\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h1 = bench.kernel_source_hash("mha_fwd_kernel")
    for fn in bench.KERNEL_SOURCES["mha_fwd_kernel"]:
        (csrc / fn).write_text("int a = 1;  // another comment\nint b = 2;   \n")
    assert bench.kernel_source_hash("mha_fwd_kernel") == h1
    (csrc / bench.KERNEL_SOURCES["mha_fwd_kernel"][0]).write_text("int a = 3;\nint b = 2;\n")
    assert bench.kernel_source_hash("mha_fwd_kernel") != h1


@pytest.mark.parametrize("name", sorted(synth.CONFIGS))
def test_config_object_names_the_workload(name):
    c = synth.CONFIGS[name]
    cfg = bench.config_dict(name, c)
    for key in ("B", "H", "N", "d", "causal", "seed"):
        assert cfg[key] == c[key]
    assert cfg["flops_per_step"] == bench.counted_flops(c)
    assert cfg["workload"].startswith(name)
    assert cfg["parallelism"] == "single GPU"
    assert bench.config_dict(name, c, world=4)["parallelism"] == "replicas x4"
