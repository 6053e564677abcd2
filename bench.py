"""Benchmark of the fused attention forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
                    [--impl ours|reference] [--no-cpu-baseline] [--backward]
                    [--e2e-steps E]

One step is one attention forward pass (the whole hot path: Q/K/V tile
loads, S = Q K^T, masked online softmax, O += P V, O/LSE epilogue) over one
synthetic batch.  The default workload is the long-sequence causal case
B=1, H=32, N=16384, d=128 ("cfg5"); other names are listed in synth.CONFIGS.
The decode names (synth.DECODE_CONFIGS, synth.PAGED_CONFIGS) time the
split-KV and paged paths against the HBM roofline instead, and --backward
times mha_bwd on a forward workload.

Metric: attention forward TFLOP/s, counting 4*B*H*N^2*d FLOPs per pass
(half of that with the causal mask), aggregated over all ranks.  Rank 0
prints one JSON line.  Under torchrun each rank runs its own independent
batch (a replica with its own seed; weak scaling, no data-path collective).

`--impl reference` times the fp64 CPU oracle (the reference arm) on a
bounded sample of rows of the same workload, on this machine's host cores.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

# NVIDIA's dense bf16 figure for one GB300, reported beside the measured
# denominators: the HGX B300 datasheet gives 36 PFLOP/s FP16/BF16 for eight
# GPUs with 2:4 sparsity, i.e. 4.5 per GPU sparse and 2.25 dense.
NOMINAL_BF16_TFLOPS = 2250.0
# A timed region shorter than this runs before the board's power cap settles
# the clock, the situation of the burst cuBLAS measurement; longer regions
# are compared with the sustained one.
BURST_REGION_S = 1.0
L2_BYTES = 129e6
METRIC = "attention fwd TFLOP/s and % of GB300 bf16 tensor peak, per (B,H,N,d,causal)"
UNIT = "TFLOP/s"
FALLBACK_PEAK_TFLOPS = 1900.0  # used only when MEASURED_PEAKS.json is absent
FALLBACK_PEAK_SUSTAINED = 1700.0


def counted_flops(c) -> float:
    f = 4.0 * c["B"] * c["H"] * c["N"] * c["N"] * c["d"]
    return f / 2 if c["causal"] else f


def fwd_kernel_name(B, H, N, d, causal, sms) -> str:
    """The forward instantiation mha_fwd launches for a shape on a device
    with `sms` multiprocessors, as the library reports its tile order, for
    labelling the measurements."""
    import head_attention_forward_gb300 as mha
    hmajor = mha.mha_fwd_tile_order(B, H, N, d, causal, sms) == 1
    return f"mha_fwd_kernel<{d},{'true' if causal else 'false'}{',head-major' if hmajor else ''}>"


def workload_name(name, c) -> str:
    return (f"{name}: B={c['B']},H={c['H']},N={c['N']},d={c['d']},"
            f"{'causal' if c['causal'] else 'non-causal'}")


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def load_peaks():
    """(sustained, burst, source) dense bf16 peaks in TFLOP/s."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        burst = float(pk["bf16_tflops"])
        sustained = float(pk.get("bf16_tflops_sustained", burst))
        return sustained, burst, "measured (MEASURED_PEAKS.json)"
    return FALLBACK_PEAK_SUSTAINED, FALLBACK_PEAK_TFLOPS, "fallback (no MEASURED_PEAKS.json)"


def pick_peak(region_s: float):
    """The roofline denominator for a timed region of `region_s` seconds:
    the burst cuBLAS figure below BURST_REGION_S (the clock has not yet
    settled under the power cap), the sustained one above it."""
    sustained, burst, src = load_peaks()
    if region_s < BURST_REGION_S:
        return burst, f"{src} bf16_tflops (burst: timed region {region_s:.3f} s < {BURST_REGION_S:.0f} s)"
    return sustained, f"{src} bf16_tflops_sustained (timed region {region_s:.3f} s >= {BURST_REGION_S:.0f} s)"


# Source files each kernel is compiled from (and the host file that picks
# its launch shape and tile order); a recorded ncu traffic figure is valid
# only while these are unchanged.
KERNEL_SOURCES = {
    "mha_fwd_kernel": ("mha_fwd_kernel.cuh", "sm103_ptx.cuh", "mha_wait.cuh", "mha_fwd.cu"),
}


def kernel_source_hash(kernel: str) -> str:
    """Hash of the kernel's code: its source files with // comments, trailing
    blanks and empty lines removed, so that editing a comment keeps the
    recorded traffic of an unchanged kernel."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "head_attention_forward_gb300", "csrc")
    for fn in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, fn), encoding="utf-8") as f:
            code = [ln.split("//", 1)[0].rstrip() for ln in f]
        h.update(fn.encode() + "\n".join(ln for ln in code if ln).encode())
    return h.hexdigest()[:16]


def recorded_traffic(name):
    """DRAM bytes per launch of the workload's dominant kernel from the
    committed ncu summary, if it was taken on that kernel's current source;
    otherwise None."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    ent = rec.get(name)
    if not ent or ent.get("kernel_family") not in KERNEL_SOURCES:
        return None
    if ent.get("kernel_source_hash") != kernel_source_hash(ent["kernel_family"]):
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self):
        if self.proc is None or not self.lines:
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


class NvmlSampler:
    """Reads the SM clock and the clock-event reasons in-process through
    NVML, every `period_s`, on a thread of its own.  Only read-only queries
    are made (clock info and event reasons); nothing is set.

    Samples carry host timestamps, so a caller can keep those that fall
    inside its timed region (`mark()` before and after it)."""

    # nvmlClocksEventReason* bits of the reasons named in the timing rules
    REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                   0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index: int, period_s: float = 0.0005):
        self.device_index = device_index
        self.period_s = period_s
        self.samples = []  # (host time, sm MHz, reasons bitmask)
        self.marks = []
        self.max_mhz = None
        self._stop = threading.Event()
        self._thread = None
        self._lib = None
        self._h = None

    def _open(self):
        import ctypes
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError:
            return False
        if lib.nvmlInit_v2() != 0:
            return False
        h = ctypes.c_void_p()
        bus = None
        try:
            import torch
            pr = torch.cuda.get_device_properties(self.device_index)
            bus = "%08x:%02x:%02x.0" % (pr.pci_domain_id, pr.pci_bus_id, pr.pci_device_id)
        except Exception:
            bus = None
        ok = bus is not None and lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) == 0
        if not ok and lib.nvmlDeviceGetHandleByIndex_v2(self.device_index, ctypes.byref(h)) != 0:
            return False
        self._lib, self._h = lib, h
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:  # NVML_CLOCK_SM
            self.max_mhz = float(mx.value)
        try:
            self._reasons = lib.nvmlDeviceGetCurrentClocksEventReasons
        except AttributeError:
            self._reasons = lib.nvmlDeviceGetCurrentClocksThrottleReasons
        return True

    def _run(self):
        import ctypes
        mhz, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            t = time.perf_counter()
            if self._lib.nvmlDeviceGetClockInfo(self._h, 1, ctypes.byref(mhz)) == 0:
                r = rs.value if self._reasons(self._h, ctypes.byref(rs)) == 0 else 0
                self.samples.append((t, float(mhz.value), int(r)))
            self._stop.wait(self.period_s)

    def __enter__(self):
        if self._open():
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()
        return self

    def __exit__(self, *exc):
        self._stop.set()
        if self._thread is not None:
            self._thread.join(timeout=5)
        if self._lib is not None:
            self._lib.nvmlShutdown()

    def mark(self):
        self.marks.append(time.perf_counter())

    def summary(self, t0=None, t1=None):
        """Median SM clock and the union of reasons over the samples taken
        between t0 and t1 (default: the first two marks)."""
        if t0 is None and len(self.marks) >= 2:
            t0, t1 = self.marks[0], self.marks[1]
        inside = [s for s in self.samples if (t0 is None or t0 <= s[0] <= t1)]
        if not inside:
            return None
        reasons = sorted({nm for _, _, r in inside for bit, nm in self.REASON_BITS.items() if r & bit})
        mhz = [m for _, m, _ in inside]
        return {"sm_mhz": statistics.median(mhz), "sm_mhz_min": min(mhz), "sm_mhz_max": max(mhz),
                "sm_max_mhz": self.max_mhz, "reasons": reasons, "samples": len(inside),
                "source": f"NVML in-process, every {self.period_s * 1e3:.1f} ms"}


def merge_clocks(nvml_summary, smi_summary):
    """The clock record of a timed region: the in-process NVML samples inside
    it, with the reasons nvidia-smi saw added (its 100 ms samples are too
    coarse for the clock of a short region, but catch every reason)."""
    if nvml_summary is None:
        return smi_summary
    out = dict(nvml_summary)
    if smi_summary:
        out["reasons"] = sorted(set(out["reasons"]) | set(smi_summary.get("reasons", [])))
        out["nvidia_smi"] = smi_summary
    return out


def oracle_sample(c, q, k, v, rows_per_head: int, heads, nthreads: int = 0):
    """Times the oracle on `rows_per_head` evenly spread rows of each head in
    `heads`; returns (seconds, counted FLOPs of those rows, rows)."""
    import oracle
    N, d = c["N"], c["d"]
    scale = float(np.float32(1.0 / math.sqrt(d)))
    rows = np.unique(np.linspace(0, N - 1, rows_per_head).astype(np.int64))
    per_row = 4.0 * N * d * (0.5 if c["causal"] else 1.0)
    t0 = time.perf_counter()
    for bh in heads:
        oracle.attention_rows(q, k, v, scale, c["causal"], int(bh), rows, nthreads)
    dt = time.perf_counter() - t0
    return dt, per_row * rows.size * len(heads), rows.size * len(heads)


def size_oracle_sample(c, q, k, v, target_s: float, nthreads: int = 0):
    """(rows per head, number of heads) so that the oracle runs about target_s."""
    import oracle
    oracle.build()
    dt, _, n = oracle_sample(c, q, k, v, 64, [0], nthreads)
    per_row = max(dt / max(n, 1), 1e-6)
    rows = int(min(c["N"], max(16, target_s / per_row)))
    heads = int(max(1, min(c["B"] * c["H"], round(target_s / (per_row * rows)))))
    return rows, heads


def config_dict(name, c, world: int = 1):
    """The `config` object of a forward workload's JSON line (the same for
    both arms, so that their lines name one workload)."""
    set_bytes = 4 * c["B"] * c["H"] * c["N"] * c["d"] * 2
    return {"workload": workload_name(name, c), "B": c["B"], "H": c["H"], "N": c["N"], "d": c["d"],
            "causal": c["causal"], "seed": c["seed"], "sigma_qk": c["sigma_qk"], "sigma_v": c["sigma_v"],
            "flops_per_step": counted_flops(c),
            "l2": ("inputs larger than L2 (Q+K+V+O = %.0f MB > 129 MB)" % (set_bytes / 1e6)
                   if set_bytes > L2_BYTES else "inputs fit L2; rotated over copies or L2 flushed"),
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def run_reference(args, c, name):
    """Reference arm: the fp64 oracle on the host cores, per step a bounded
    sample of rows of the same workload."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    q, k, v = synth.qkv(c["seed"], c["B"], c["H"], c["N"], c["d"], c["sigma_qk"], c["sigma_v"])
    budget = 150.0 / max(1, args.steps + args.warmup)
    cores = host_cores()
    rows, _ = size_oracle_sample(c, q, k, v, budget, cores)
    for i in range(args.warmup):
        oracle_sample(c, q, k, v, rows, [i % (c["B"] * c["H"])], cores)
    tot_t, tot_f, tot_rows = 0.0, 0.0, 0
    for i in range(args.steps):
        dt, fl, nr = oracle_sample(c, q, k, v, rows, [(i + args.warmup) % (c["B"] * c["H"])], cores)
        tot_t += dt
        tot_f += fl
        tot_rows += nr
    value = tot_f / tot_t / 1e12
    sample = f"{rows} evenly spaced query rows of one head per step ({tot_rows} rows total)"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 0,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_dict(name, c, 1),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_decode(args, name):
    """Split-KV path on a decode-shaped workload (single GPU): TFLOP/s with
    the same counting rule, plus the HBM roofline, which bounds this path."""
    import torch

    import head_attention_forward_gb300 as mha
    c = synth.DECODE_CONFIGS[name]
    B, H, Nq, Nk, d, causal = c["B"], c["H"], c["Nq"], c["Nk"], c["d"], c["causal"]
    qb, kb, vb = synth.decode_inputs(name)
    if args.impl == "reference":
        import oracle
        heads = 1
        t0 = time.perf_counter()
        oracle.attention_kv(qb[:1, :heads], kb[:1, :heads], vb[:1, :heads],
                            float(np.float32(1 / math.sqrt(d))), causal)
        dt = time.perf_counter() - t0
        fl = 4.0 * heads * Nq * Nk * d
        print(json.dumps({"impl": "reference", "metric": METRIC, "value": fl / dt / 1e12, "unit": UNIT,
                          "n_gpus": 0, "steps": 1, "warmup": 0, "ms_per_step": dt * 1e3,
                          "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                          "dtype": "f64", "data": "synthetic",
                          "config": {"workload": f"{name}: B={B},H={H},Nq={Nq},Nk={Nk},d={d}"},
                          "cpu_baseline": {"value": fl / dt / 1e12, "unit": UNIT,
                                           "cores": oracle.num_threads(), "kind": "oracle",
                                           "sample": f"{heads} head(s) of the workload"},
                          "e2e": {"value": fl / dt / 1e12, "unit": UNIT, "h2d_bytes_per_step": 0,
                                  "d2h_bytes_per_step": 0}}), flush=True)
        return 0
    torch.cuda.set_device(0)
    mha.build()
    mha.lib()

    def dev(bits):
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()

    q, k, v = dev(qb), dev(kb), dev(vb)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device="cuda")
    ws_bytes = mha.mha_fwd_kv_workspace_size(B, H, Nq, Nk, d, 0)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    scale = float(np.float32(1.0 / math.sqrt(d)))
    stream = torch.cuda.current_stream()
    sptr = int(stream.cuda_stream)

    def step():
        mha.mha_fwd_kv(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, 0, ws, ws_bytes, sptr)

    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    with ClockSampler(0) as clk:
        torch.cuda.synchronize()
        evs[0].record(stream)
        for i in range(args.steps):
            step()
            evs[i + 1].record(stream)
        torch.cuda.synchronize()
    rc, word = mha.mha_device_status(sptr)
    if rc != mha.MHA_OK:
        raise RuntimeError(f"device status {rc} ({word:#x})")
    total_ms = evs[0].elapsed_time(evs[-1])
    ms = total_ms / args.steps
    # FLOPs: 4 Nq Nk d per head (every key visible to the newest query)
    flops = 4.0 * B * H * Nq * Nk * d
    algo_bytes = 2 * (q.numel() + k.numel() + v.numel() + o.numel()) + 4 * lse.numel()
    gbs = algo_bytes / (ms / 1e3) / 1e9
    hbm_peak = 6773.5
    pk_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(pk_path):
        with open(pk_path) as f:
            hbm_peak = float(json.load(f).get("hbm_gbs", hbm_peak))
    line = {
        "metric": METRIC, "value": flops / (ms / 1e3) / 1e12, "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{name}: B={B},H={H},Nq={Nq},Nk={Nk},d={d},"
                               f"{'causal' if causal else 'non-causal'} (split-KV path)",
                   "l2": "inputs larger than L2 (K+V = %.0f MB)" % (2 * k.numel() * 2 / 1e6),
                   "workspace_bytes": ws_bytes},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s",
                     "frac": gbs / hbm_peak, "traffic": recorded_traffic(name),
                     "algorithmic_bytes_per_step": algo_bytes,
                     "kernel": f"mha_fwd_kernel<{d},{int(bool(causal))},split> + splitkv_merge_kernel<{d}>"},
        "gpu_launches": 3 * args.steps,
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)
    return 0


def hbm_peak_gbs():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return float(json.load(f).get("hbm_gbs", 6773.5)), "measured (MEASURED_PEAKS.json hbm_gbs)"
    return 6800.0, "fallback (no MEASURED_PEAKS.json)"


def run_paged(args, name):
    """Paged-KV path on a decode workload with mixed sequence lengths."""
    import torch

    import head_attention_forward_gb300 as mha
    c = synth.PAGED_CONFIGS[name]
    B, H, Nq, d, page, causal = c["B"], c["H"], c["Nq"], c["d"], c["page"], c["causal"]
    qb, kcb, vcb, table, seq = synth.paged_inputs(name)
    num_blocks, max_blocks = kcb.shape[0], table.shape[1]
    torch.cuda.set_device(0)
    mha.build()
    mha.lib()

    def dev(bits):
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()

    q, kc, vc = dev(qb), dev(kcb), dev(vcb)
    td, sd = torch.from_numpy(table).cuda(), torch.from_numpy(seq).cuda()
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device="cuda")
    ws_bytes = mha.mha_fwd_kv_workspace_size(B, H, Nq, max_blocks * page, d, 0)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    scale = float(np.float32(1.0 / math.sqrt(d)))
    stream = torch.cuda.current_stream()
    sptr = int(stream.cuda_stream)

    def step():
        mha.mha_fwd_paged(q, kc, vc, td, sd, o, lse, B, H, Nq, d, page, num_blocks, max_blocks, scale,
                          causal, 0, ws, ws_bytes, sptr)

    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(0) as clk:
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
    rc, word = mha.mha_device_status(sptr)
    if rc != mha.MHA_OK:
        raise RuntimeError(f"device status {rc} ({word:#x})")
    ms = e0.elapsed_time(e1) / args.steps
    keys = int(seq.astype(np.int64).sum())
    flops = 4.0 * H * Nq * keys * d
    algo_bytes = 2 * 2 * keys * H * d + 2 * (q.numel() + o.numel()) + 4 * lse.numel() + table.nbytes + seq.nbytes
    gbs = algo_bytes / (ms / 1e3) / 1e9
    peak, src = hbm_peak_gbs()
    print(json.dumps({
        "metric": METRIC, "value": flops / (ms / 1e3) / 1e12, "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{name}: B={B},H={H},Nq={Nq},d={d},page={page},"
                               f"seq {int(seq.min())}..{int(seq.max())} (paged-KV path)",
                   "cached_keys": keys, "l2": "K/V caches larger than L2 (%.0f MB)" % (2 * kc.numel() * 2 / 1e6)},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                     "peak_source": src, "traffic": recorded_traffic(name),
                     "algorithmic_bytes_per_step": algo_bytes,
                     "kernel": f"mha_fwd_kernel<{d},{int(bool(causal))},split,paged> + splitkv_merge_kernel<{d}>"},
        "gpu_launches": 3 * args.steps, "clocks": clk.summary(),
    }), flush=True)
    return 0

def time_decode_block(mha, dev, stream, steps: int):
    """The split-KV and paged decode workloads for the default bench line,
    each timed over `steps` back-to-back calls (counter reset, partial pass,
    merge) after 3 warm-ups, against the measured HBM copy rate.  Their
    shapes, masks and (paged) block tables and lengths are the parity
    workloads'; the K/V values are seeded torch normals drawn on the device,
    which times the same work without generating gigabytes on the host."""
    import torch
    peak, src = hbm_peak_gbs()
    gen = torch.Generator(device=dev)
    gen.manual_seed(21)
    sptr = int(stream.cuda_stream)

    def randn(shape):
        return torch.randn(shape, generator=gen, device=dev).to(torch.bfloat16)

    def timed(step):
        for _ in range(3):
            step()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with NvmlSampler(dev.index) as nv:
            nv.mark()
            e0.record(stream)
            for _ in range(steps):
                step()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            nv.mark()
        rc, word = mha.mha_device_status(sptr)
        if rc != mha.MHA_OK:
            raise RuntimeError(f"device status {rc} ({word:#x})")
        return e0.elapsed_time(e1) / steps, nv.summary()

    out = {}
    for name, c in synth.DECODE_CONFIGS.items():
        B, H, Nq, Nk, d, causal = c["B"], c["H"], c["Nq"], c["Nk"], c["d"], c["causal"]
        q, k, v = randn((B, H, Nq, d)), randn((B, H, Nk, d)), randn((B, H, Nk, d))
        o = torch.empty_like(q)
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=dev)
        ws_bytes = mha.mha_fwd_kv_workspace_size(B, H, Nq, Nk, d, 0)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        scale = float(np.float32(1.0 / math.sqrt(d)))
        ms, clocks = timed(lambda: mha.mha_fwd_kv(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, 0,
                                                 ws, ws_bytes, sptr))
        algo = 2 * (q.numel() + k.numel() + v.numel() + o.numel()) + 4 * lse.numel()
        gbs = algo / (ms / 1e3) / 1e9
        out[name] = {"workload": f"B={B},H={H},Nq={Nq},Nk={Nk},d={d},{'causal' if causal else 'non-causal'} "
                                 "(split-KV path)",
                     "ms_per_call": ms, "gbs": gbs, "frac": gbs / peak, "peak_gbs": peak, "peak_source": src,
                     "algorithmic_bytes": algo, "steps": steps, "clocks": clocks,
                     "kernel": f"mha_fwd_kernel<{d},{int(bool(causal))},split> + splitkv_merge_kernel<{d}>"}
        del q, k, v, o, lse, ws
    for name, c in synth.PAGED_CONFIGS.items():
        B, H, Nq, d, page, causal = c["B"], c["H"], c["Nq"], c["d"], c["page"], c["causal"]
        seq, table, num_blocks = synth.paged_layout(name)
        max_blocks = table.shape[1]
        q = randn((B, H, Nq, d))
        kc, vc = randn((num_blocks, H, page, d)), randn((num_blocks, H, page, d))
        td, sd = torch.from_numpy(table).to(dev), torch.from_numpy(seq).to(dev)
        o = torch.empty_like(q)
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=dev)
        ws_bytes = mha.mha_fwd_kv_workspace_size(B, H, Nq, max_blocks * page, d, 0)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        scale = float(np.float32(1.0 / math.sqrt(d)))
        ms, clocks = timed(lambda: mha.mha_fwd_paged(q, kc, vc, td, sd, o, lse, B, H, Nq, d, page, num_blocks,
                                                    max_blocks, scale, causal, 0, ws, ws_bytes, sptr))
        keys = int(seq.astype(np.int64).sum())
        algo = 2 * 2 * keys * H * d + 2 * (q.numel() + o.numel()) + 4 * lse.numel() + table.nbytes + seq.nbytes
        gbs = algo / (ms / 1e3) / 1e9
        out[name] = {"workload": f"B={B},H={H},Nq={Nq},d={d},page={page},seq {int(seq.min())}..{int(seq.max())} "
                                 "(paged-KV path)",
                     "ms_per_call": ms, "gbs": gbs, "frac": gbs / peak, "peak_gbs": peak, "peak_source": src,
                     "algorithmic_bytes": algo, "steps": steps, "clocks": clocks,
                     "kernel": f"mha_fwd_kernel<{d},{int(bool(causal))},split,paged> + splitkv_merge_kernel<{d}>"}
        del q, kc, vc, td, sd, o, lse, ws
    return out


def run_page_sweep(args):
    """The paged-KV path against page size: one query per sequence, 32
    sequences of 8192 keys each, 32 heads, d = 128 (a 1.07 GB cache), with the
    pages in sequence order (identity table) and shuffled over the cache.
    Prints one JSON line: per page size and table, the call time and the
    achieved fraction of the measured HBM copy rate."""
    import torch

    import head_attention_forward_gb300 as mha
    torch.cuda.set_device(0)
    mha.build()
    mha.lib()
    B, H, Nq, d, keys = 32, 32, 1, 128, 8192
    scale = float(np.float32(1.0 / math.sqrt(d)))
    stream = torch.cuda.current_stream()
    sptr = int(stream.cuda_stream)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(12)
    q = torch.randn((B, H, Nq, d), generator=gen, device="cuda").to(torch.bfloat16)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device="cuda")
    seq = torch.full((B,), keys, dtype=torch.int32, device="cuda")
    peak, src = hbm_peak_gbs()
    rows = []
    for page in (16, 32, 64, 128, 256):
        pages = keys // page
        num_blocks = B * pages
        kc = torch.randn((num_blocks, H, page, d), generator=gen, device="cuda").to(torch.bfloat16)
        vc = torch.randn((num_blocks, H, page, d), generator=gen, device="cuda").to(torch.bfloat16)
        ws_bytes = mha.mha_fwd_kv_workspace_size(B, H, Nq, keys, d, 0)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        for order in ("identity", "shuffled"):
            ids = torch.arange(num_blocks, dtype=torch.int32, device="cuda")
            if order == "shuffled":
                ids = ids[torch.randperm(num_blocks, generator=gen, device="cuda")]
            table = ids.reshape(B, pages).contiguous()

            def step():
                mha.mha_fwd_paged(q, kc, vc, table, seq, o, lse, B, H, Nq, d, page, num_blocks, pages,
                                  scale, False, 0, ws, ws_bytes, sptr)

            for _ in range(max(args.warmup, 3)):
                step()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with NvmlSampler(0) as nv:
                nv.mark()
                e0.record(stream)
                for _ in range(args.steps):
                    step()
                e1.record(stream)
                torch.cuda.synchronize()
                nv.mark()
            rc, word = mha.mha_device_status(sptr)
            if rc != mha.MHA_OK:
                raise RuntimeError(f"page {page}: device status {rc} ({word:#x})")
            ms = e0.elapsed_time(e1) / args.steps
            algo = 2 * 2 * B * H * keys * d + 2 * (q.numel() + o.numel()) + 4 * lse.numel() + 4 * table.numel() + 4 * B
            gbs = algo / (ms / 1e3) / 1e9
            rows.append({"page": page, "table": order, "ms": ms, "gbs": gbs, "frac": gbs / peak,
                         "clocks": nv.summary()})
        del kc, vc, ws
    print(json.dumps({"mode": "page_sweep", "workload": f"B={B},H={H},Nq={Nq},d={d},{keys} keys per sequence",
                      "steps": args.steps, "peak_gbs": peak, "peak_source": src, "rows": rows}), flush=True)
    return 0


_INPUT_CACHE = {}


def time_forward_config(mha, name, dev, stream, min_steps: int, min_region_s: float = 0.2):
    """One forward workload timed on its own, for the per_config block.

    Inputs larger than L2 run back to back.  Smaller ones rotate over enough
    copies of Q, K, V, O and LSE that each launch finds its inputs evicted
    (more than twice L2 in all); where that would take more than 16 copies
    (the tiny workload), L2 is flushed before every launch instead and each
    launch is timed alone.  At least `min_steps` launches, and enough for
    about `min_region_s` seconds, so that the in-process clock samples cover
    the region."""
    import torch
    c = synth.CONFIGS[name]
    B, H, N, d, causal = c["B"], c["H"], c["N"], c["d"], c["causal"]
    key = (c["seed"], B, H, N, d, c["sigma_qk"], c["sigma_v"])
    if key not in _INPUT_CACHE:
        _INPUT_CACHE.clear()
        _INPUT_CACHE[key] = synth.config_inputs(name)
    qb, kb, vb = _INPUT_CACHE[key]
    set_bytes = 4 * qb.nbytes + 4 * B * H * N
    copies = 1 if set_bytes > L2_BYTES else int(math.ceil(2 * L2_BYTES / set_bytes))
    flush = None
    if copies > 16:
        copies = 1
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    def dev_tensor(bits):
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev)
    q0, k0, v0 = dev_tensor(qb), dev_tensor(kb), dev_tensor(vb)
    sets = []
    for i in range(copies):
        q, k, v = (q0, k0, v0) if i == 0 else (q0.clone(), k0.clone(), v0.clone())
        sets.append((q, k, v, torch.empty_like(q), torch.empty((B, H, N), dtype=torch.float32, device=dev)))
    scale = float(np.float32(1.0 / math.sqrt(d)))
    sptr = int(stream.cuda_stream)

    def launch(i):
        q, k, v, o, lse = sets[i % copies]
        mha.mha_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, sptr)

    for i in range(3):
        launch(i)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for i in range(4):
        launch(i)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    est_ms = max(e0.elapsed_time(e1) / 4, 1e-3)
    steps = max(min_steps, int(math.ceil(min_region_s * 1e3 / est_ms)))
    if flush is not None:
        steps = min(steps, 400)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(2 * steps)]
    with NvmlSampler(dev.index) as nv:
        torch.cuda.synchronize(dev)
        nv.mark()
        for i in range(steps):
            if flush is not None:
                flush.fill_(i & 255)
            evs[2 * i].record(stream)
            launch(i)
            evs[2 * i + 1].record(stream)
        torch.cuda.synchronize(dev)
        nv.mark()
    rc, word = mha.mha_device_status(sptr)
    if rc != mha.MHA_OK:
        raise RuntimeError(f"{name}: device status {rc} ({word:#x})")
    per = [evs[2 * i].elapsed_time(evs[2 * i + 1]) for i in range(steps)]
    if flush is None:
        ms = evs[0].elapsed_time(evs[-1]) / steps  # back to back: launch gaps count
        timing = ("back to back, inputs larger than L2" if copies == 1 else
                  f"back to back, rotating over {copies} copies of the inputs ({copies * set_bytes / 1e6:.0f} MB)")
    else:
        ms = statistics.mean(per)
        timing = "one launch at a time, each after a 256 MB write that flushes L2"
    region_s = (nv.marks[1] - nv.marks[0]) if len(nv.marks) >= 2 else ms * steps / 1e3
    peak, peak_src = pick_peak(region_s)
    _, peak_burst, _ = load_peaks()
    tf = counted_flops(c) / (ms / 1e3) / 1e12
    clocks = nv.summary()
    del sets, q0, k0, v0, flush
    return {"workload": workload_name(name, c), "tflops": tf, "pct_of_peak": 100.0 * tf / peak,
            "peak": peak, "peak_source": peak_src, "pct_of_burst_peak": 100.0 * tf / peak_burst,
            "ms_per_launch": ms, "median_launch_ms": statistics.median(per), "steps": steps,
            "timing": timing, "clocks": clocks,
            "kernel": fwd_kernel_name(B, H, N, d, causal, torch.cuda.get_device_properties(dev).multi_processor_count)}


BWD_METRIC = ("attention bwd TFLOP/s (counted 10*B*H*N^2*d, halved when causal) and % of GB300 "
              "bf16 tensor peak, per (B,H,N,d,causal)")


def run_backward(args, name):
    """mha_bwd on a forward workload: O and LSE come from one mha_fwd call,
    dO is a synthetic N(0,1) tensor; each step is one mha_bwd call (three
    kernels).  Single GPU."""
    import torch

    import head_attention_forward_gb300 as mha
    c = synth.CONFIGS[name]
    B, H, N, d, causal = c["B"], c["H"], c["N"], c["d"], c["causal"]
    torch.cuda.set_device(0)
    mha.build()
    mha.lib()
    qb, kb, vb = synth.qkv(c["seed"], B, H, N, d, c["sigma_qk"], c["sigma_v"])
    dob = synth.normal_bf16_c(c["seed"], 3, B * H * N * d).reshape(B, H, N, d)

    def dev(bits):
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()

    q, k, v, do = dev(qb), dev(kb), dev(vb), dev(dob)
    scale = float(np.float32(1.0 / math.sqrt(d)))
    stream = torch.cuda.current_stream()
    sptr = int(stream.cuda_stream)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    mha.mha_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, sptr)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws_bytes = mha.mha_bwd_workspace_size(B, H, N, d)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")

    def step():
        mha.mha_bwd(q, k, v, o, lse, do, dq, dk, dv, B, H, N, d, scale, causal, ws, ws_bytes, sptr)

    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    with ClockSampler(0) as clk:
        torch.cuda.synchronize()
        evs[0].record(stream)
        for i in range(args.steps):
            step()
            evs[i + 1].record(stream)
        torch.cuda.synchronize()
    rc, word = mha.mha_device_status(sptr)
    if rc != mha.MHA_OK:
        raise RuntimeError(f"device status {rc} ({word:#x})")
    ms = evs[0].elapsed_time(evs[-1]) / args.steps
    flops = 10.0 * B * H * N * N * d / (2 if causal else 1)
    tf = flops / (ms * 1e-3) / 1e12
    peak, peak_burst = 1703.5, 1891.4
    pk_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(pk_path):
        with open(pk_path) as f:
            pk = json.load(f)
        peak = float(pk.get("bf16_tflops_sustained", peak))
        peak_burst = float(pk.get("bf16_tflops", peak_burst))
    print(json.dumps({
        "metric": BWD_METRIC, "value": tf, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{name} backward: B={B},H={H},N={N},d={d},"
                               f"{'causal' if causal else 'non-causal'}",
                   "flops_per_step": flops,
                   "l2": "inputs larger than L2" if 6 * B * H * N * d * 2 > 129e6 else
                         "inputs smaller than L2 (not flushed)"},
        "roofline": {"bound": "tensor", "achieved": tf, "peak": peak, "unit": "TFLOP/s",
                     "frac": tf / peak, "peak_source": "measured (MEASURED_PEAKS.json: "
                     "bf16_tflops_sustained; burst beside it)", "peak_burst": peak_burst,
                     "frac_burst": tf / peak_burst, "traffic": None,
                     "kernel": f"mha_bwd call: bwd_rowdot_kernel<{d}> + bwd_tile_kernel<{d}> x2 "
                               "(counted FLOPs over the call's time)"},
        "gpu_launches": 3 * args.steps, "clocks": clk.summary(),
    }), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="cfg5",
                    choices=sorted(synth.CONFIGS) + sorted(synth.DECODE_CONFIGS)
                    + sorted(synth.PAGED_CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="time only the chosen workload (no per_config or per_decode block)")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--backward", action="store_true",
                    help="time mha_bwd on the chosen forward workload instead of mha_fwd")
    ap.add_argument("--page-sweep", action="store_true",
                    help="time the paged-KV path at page sizes 16..256, pages in order and shuffled")
    args = ap.parse_args()
    if args.page_sweep:
        return run_page_sweep(args)
    name = args.config
    if args.backward:
        if name not in synth.CONFIGS:
            ap.error("--backward takes one of the forward workloads")
        return run_backward(args, name)
    if name in synth.DECODE_CONFIGS:
        return run_decode(args, name)
    if name in synth.PAGED_CONFIGS:
        return run_paged(args, name)
    c = synth.CONFIGS[name]
    if args.impl == "reference":
        return run_reference(args, c, name)
    if args.warmup < 3:
        print("note: fewer than 3 warm-up steps; the number is not a bench value", file=sys.stderr)

    import torch

    import head_attention_forward_gb300 as mha
    from head_attention_forward_gb300.sharding import replica_seed

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", local if world > 1 else 0)
    mha.build()
    mha.lib()

    B, H, N, d, causal = c["B"], c["H"], c["N"], c["d"], c["causal"]
    seed = replica_seed(c["seed"], rank)
    qb, kb, vb = synth.qkv(seed, B, H, N, d, c["sigma_qk"], c["sigma_v"])

    def dev_tensor(bits):
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev)

    q, k, v = dev_tensor(qb), dev_tensor(kb), dev_tensor(vb)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    scale = float(np.float32(1.0 / math.sqrt(d)))
    stream = torch.cuda.current_stream(dev)
    sptr = int(stream.cuda_stream)

    def step():
        mha.mha_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, sptr)

    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize(dev)
    rc, word = mha.mha_device_status(sptr)
    if rc != mha.MHA_OK:
        raise RuntimeError(f"device status after warm-up: {rc} ({word:#x})")

    # timed region: K launches, one event pair around each on the launch stream
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    with ClockSampler(dev.index) as clk, NvmlSampler(dev.index) as nv:
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)
        nv.mark()
        evs[0].record(stream)
        for i in range(args.steps):
            step()
            evs[i + 1].record(stream)
        torch.cuda.synchronize(dev)
        nv.mark()
        if dist is not None:
            dist.barrier()
    per_launch_ms = [evs[i].elapsed_time(evs[i + 1]) for i in range(args.steps)]
    total_ms = evs[0].elapsed_time(evs[-1])
    if dist is not None:
        t = torch.tensor([total_ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    rc, word = mha.mha_device_status(sptr)
    if rc != mha.MHA_OK:
        raise RuntimeError(f"device status after timing: {rc} ({word:#x})")

    # one launch right after L2 has been flushed (a 256 MB write), timed alone
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    cold_ms = []
    for _ in range(3):
        flush.fill_(1)
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        step()
        c1.record(stream)
        torch.cuda.synchronize(dev)
        cold_ms.append(c0.elapsed_time(c1))
    del flush

    flops = counted_flops(c)
    value = flops * args.steps * world / (total_ms / 1e3) / 1e12
    mean_launch_ms = statistics.mean(per_launch_ms)
    achieved = flops / (mean_launch_ms / 1e3) / 1e12
    peak_sustained, peak_burst, _ = load_peaks()
    peak, peak_src = pick_peak(total_ms / 1e3)
    clocks = merge_clocks(nv.summary(), clk.summary())
    if clocks and clocks.get("sm_mhz"):
        # launch duration in SM cycles at the median clock of the region,
        # comparable with the cycles a profiler reports for one launch
        clocks["cycles_per_launch"] = mean_launch_ms * 1e-3 * clocks["sm_mhz"] * 1e6

    per_config = None
    per_decode = None
    if world == 1 and not args.no_per_config:
        per_config = {}
        for other in synth.CONFIGS:
            if other != name:
                per_config[other] = time_forward_config(mha, other, dev, stream, args.steps)
        per_decode = time_decode_block(mha, dev, stream, 50)

    # End to end through the public C ABI: every step copies its Q, K, V from
    # pinned host memory to the device, runs mha_fwd, and copies O and LSE
    # back to pinned host memory.  Two device buffer sets and three streams
    # pipeline the steps: step k+1's inputs go up and step k-1's outputs come
    # down while step k's kernel runs; every step still moves all its bytes
    # inside the timed region.  The same loop with everything on one stream
    # is reported beside it ("serial").
    hq, hk, hv = (torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).pin_memory()
                  for b in (qb, kb, vb))
    ho = [torch.empty(o.shape, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    hl = [torch.empty(lse.shape, dtype=torch.float32).pin_memory() for _ in range(2)]
    sets = [(q, k, v, o, lse),
            (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), torch.empty_like(o),
             torch.empty_like(lse))]
    s_up, s_down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def e2e_run(steps, pipelined):
        up, down = (s_up, s_down) if pipelined else (stream, stream)
        ev_up = [torch.cuda.Event() for _ in range(steps)]
        ev_run = [torch.cuda.Event() for _ in range(steps)]
        ev_down = [torch.cuda.Event() for _ in range(steps)]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        up.wait_event(e0)
        down.wait_event(e0)
        for i in range(steps):
            dq, dk, dv, do_, dl = sets[i % 2]
            if i >= 2:
                up.wait_event(ev_run[i - 2])  # the kernel that read this set is done
            with torch.cuda.stream(up):
                dq.copy_(hq, non_blocking=True)
                dk.copy_(hk, non_blocking=True)
                dv.copy_(hv, non_blocking=True)
            ev_up[i].record(up)
            stream.wait_event(ev_up[i])
            if i >= 2:
                stream.wait_event(ev_down[i - 2])  # this set's outputs have been read back
            mha.mha_fwd(dq, dk, dv, do_, dl, B, H, N, d, scale, causal, sptr)
            ev_run[i].record(stream)
            down.wait_event(ev_run[i])
            with torch.cuda.stream(down):
                ho[i % 2].copy_(do_, non_blocking=True)
                hl[i % 2].copy_(dl, non_blocking=True)
            ev_down[i].record(down)
        stream.wait_event(ev_down[steps - 1])
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1)

    e2e_run(2, True)
    if dist is not None:
        dist.barrier()
    # the host link is shared with the machine's other GPUs: three timed
    # pipelined runs, the median reported and all three listed
    e2e_runs = [e2e_run(args.e2e_steps, True) for _ in range(3)]
    e2e_ms = statistics.median(e2e_runs)
    serial_ms = e2e_run(args.e2e_steps, False)
    if dist is not None:
        t = torch.tensor([e2e_ms, serial_ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_ms, serial_ms = float(t[0].item()), float(t[1].item())
    e2e_value = flops * args.e2e_steps * world / (e2e_ms / 1e3) / 1e12
    serial_value = flops * args.e2e_steps * world / (serial_ms / 1e3) / 1e12
    h2d = 3 * qb.nbytes
    d2h = o.numel() * 2 + lse.numel() * 4

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cores = host_cores()
        rows, heads = size_oracle_sample(c, qb, kb, vb, 15.0, cores)
        dt, fl, nr = oracle_sample(c, qb, kb, vb, rows, list(range(heads)), cores)
        cpu = {"value": fl / dt / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"{rows} evenly spaced query rows of each of heads 0..{heads - 1} "
                         f"({nr} rows, FLOPs counted as the metric counts them), fp64, {dt:.1f} s"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": config_dict(name, c, world),
            "pct_of_peak": 100.0 * value / world / peak,
            "pct_of_burst_peak": 100.0 * value / world / peak_burst,
            "pct_of_sustained_peak": 100.0 * value / world / peak_sustained,
            "pct_of_nominal_peak": 100.0 * value / world / NOMINAL_BF16_TFLOPS,
            "timed_region_s": total_ms / 1e3,
            "median_launch_ms": statistics.median(per_launch_ms),
            "cold_launch_ms": statistics.median(cold_ms),  # after an L2 flush
            # exponentials the softmax evaluates per second (one per visible
            # score, counted like the FLOPs: B*H*N^2, halved when causal)
            "exp2_per_s": flops / (4.0 * d) / (statistics.median(per_launch_ms) / 1e3),
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT,
                         "frac": achieved / peak, "peak_source": peak_src,
                         "peak_burst": peak_burst, "frac_burst": achieved / peak_burst,
                         "peak_sustained": peak_sustained, "frac_sustained": achieved / peak_sustained,
                         "traffic": recorded_traffic(name),
                         "algorithmic_flops_per_launch": flops,
                         "kernel": fwd_kernel_name(B, H, N, d, causal,
                                                   torch.cuda.get_device_properties(dev).multi_processor_count)},
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": args.e2e_steps,
                    "runs_tflops": [flops * args.e2e_steps * world / (ms / 1e3) / 1e12 for ms in e2e_runs],
                    "of_runs": "median of three timed pipelined runs",
                    "pipelined": "two device buffer sets; step k+1's upload and step k-1's "
                                 "download overlap step k's kernel",
                    "serial_value": serial_value},
            "gpu_launches": args.steps,
            "clocks": clocks,
            "cpu_baseline": cpu,
        }
        if per_config is not None:
            line["per_config"] = per_config
        if per_decode is not None:
            line["per_decode"] = per_decode
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
