#!/usr/bin/env python
"""Benchmark of the DCP LSE-weighted merge on GB300.

Metric: LSE-combine HBM GB/s (and % of the HBM roofline) and us/call at batch
rows 1-128, one GB300. Workload: Kimi-K2.5 geometry (cp = 4, 64 heads, 16 per
destination, D = 512, bf16 partials, base-2 fp32 LSEs U[-4, 24]) swept over
rows 1, 8, 16, 32, 64, 128.

One step = one pass of the whole merge over every row count of the sweep:
for each row count, one replay of a CUDA graph holding 60 calls (the pages'
per-layer microbenchmark method: "[DCP] Run fi_a2a on FlashInfer's fused
all-to-all + LSE reduce", "Speed Tests and Profiling"). Each of the 60 calls
reads and writes its own buffers, and L2 is flushed (a write larger than L2)
before every step, so every call starts cold and the GB/s are HBM GB/s.
Steps are timed with CUDA events on the launching stream; the flush sits
outside the events.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs the same workload on its own GPU
(independent replicas: the merge has no exchange step on one node here),
the time is the max over ranks and the value is the sum over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
NOMINAL_HBM_GBS = 8000.0  # GB300 HBM3e, nominal (the measured copy peak is the roofline's denominator)
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "LSE-combine HBM GB/s (% of peak) and µs/call at rows 1–128, 1×GB300"
CALLS_PER_GRAPH = 60
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
KERNEL_SOURCE = os.path.join(ROOT, "decode_context_mla_dcp_gb300", "csrc", "dcp_lse_reduce.cu")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.json")


# ---------------------------------------------------------------------------- utilities

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def aggregate_ranks(local_seconds: float, local_bytes: float, group=None):
    """Max of the timed-region seconds and sum of the bytes over all ranks
    (the whole-job figures). With one process this is the identity."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size(group) == 1:
        return local_seconds, local_bytes
    backend = dist.get_backend(group)
    dev = torch.device("cuda", torch.cuda.current_device()) if backend == "nccl" else torch.device("cpu")
    t = torch.tensor([local_seconds], dtype=torch.float64, device=dev)
    b = torch.tensor([local_bytes], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    dist.all_reduce(b, op=dist.ReduceOp.SUM, group=group)
    return float(t.item()), float(b.item())


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def measured_tensor_peak():
    """Dense bf16 TFLOP/s: the measured burst figure, else the fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"])
    except (OSError, KeyError, ValueError):
        return FALLBACK_BF16_TFLOPS


def kernel_source_sha():
    with open(KERNEL_SOURCE, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def recorded_traffic():
    """Per-launch DRAM bytes from the committed ncu summary, only if it was
    taken on the kernel source as it is now."""
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    if d.get("kernel_source_sha256") != kernel_source_sha():
        return None
    return d.get("per_launch_bytes_bench_step")


class NvmlClockSampler:
    """Read-only NVML samples (every few ms) of this GPU's SM clock, power and
    clock-event (throttle) reasons, through the driver's libnvidia-ml."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, uuid: str, period_s: float = 0.005):
        import ctypes
        self.ct = ctypes
        self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
        if self.nvml.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        if self.nvml.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.h)) != 0:
            raise OSError("no NVML handle for " + uuid)
        self.reason_fn = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        self.period = period_s
        self.samples = []
        self.stop_flag = threading.Event()
        self.thread = None

    def _one(self):
        ct = self.ct
        c, mx, mw, rs = ct.c_uint(), ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        if self.nvml.nvmlDeviceGetClockInfo(self.h, 1, ct.byref(c)) != 0:
            return None
        self.nvml.nvmlDeviceGetMaxClockInfo(self.h, 1, ct.byref(mx))
        self.nvml.nvmlDeviceGetPowerUsage(self.h, ct.byref(mw))
        self.reason_fn(self.h, ct.byref(rs))
        return c.value, mx.value, mw.value / 1000.0, rs.value

    def start(self):
        def run():
            while not self.stop_flag.is_set():
                v = self._one()
                if v is not None:
                    self.samples.append(v)
                self.stop_flag.wait(self.period)
        self.thread = threading.Thread(target=run, daemon=True)
        self.thread.start()

    def stop(self):
        self.stop_flag.set()
        if self.thread:
            self.thread.join(timeout=5)
        sm = [x[0] for x in self.samples]
        reasons = set()
        for x in self.samples:
            for bit, name in self.REASONS.items():
                if x[3] & bit:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(x[1] for x in self.samples) if sm else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(x[2] for x in self.samples) if sm else None, "source": "nvml"}


def clock_sampler(uuid):
    try:
        return NvmlClockSampler(uuid)
    except (OSError, AttributeError, TypeError):
        return ClockSampler(uuid)


class ClockSampler:
    """nvidia-smi samples of this GPU's clocks and throttle reasons."""
    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            if self.uuid and parts[0] != self.uuid:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None, "source": "nvidia-smi"}


# ---------------------------------------------------------------------------- the workload

def workload_config():
    from decode_context_mla_dcp_gb300.inputs import CONFIGS
    return CONFIGS["kimi"]


def sweep_bytes(cfg):
    from decode_context_mla_dcp_gb300 import algorithmic_bytes
    return {rows: algorithmic_bytes(cfg.cp, rows, cfg.H, cfg.D) for rows in cfg.rows}


class RowSet:
    """Device buffers for one row count: `slots` independent copies of the
    inputs and outputs, so consecutive calls never share cache lines."""

    def __init__(self, cfg, rows: int, slots: int, seed: int = 0):
        import torch
        from decode_context_mla_dcp_gb300.inputs import make_merge_inputs
        self.cfg, self.rows, self.slots = cfg, rows, slots
        self.inp = make_merge_inputs(cfg, rows, seed=seed)
        cp, H, D, Hl = cfg.cp, cfg.H, cfg.D, cfg.H // cfg.cp
        self.src = []
        self.lse = []
        for j in range(cp):
            s = torch.from_numpy(self.inp.srcs[j].view(np.int16)).view(torch.bfloat16).cuda()
            l = torch.from_numpy(np.ascontiguousarray(self.inp.lses[j]).reshape(rows, H)).cuda()  # [B,H,1] -> [B,H]
            self.src.append(s.unsqueeze(0).repeat(slots, 1, 1, 1).contiguous())
            self.lse.append(l.unsqueeze(0).repeat(slots, 1, 1).contiguous())
        self.dst = [torch.empty((slots, rows, Hl, D), dtype=torch.bfloat16, device="cuda") for _ in range(cp)]
        self.lse_out = [torch.empty((slots, rows, Hl), dtype=torch.float32, device="cuda") for _ in range(cp)]

    def ptrs(self, k: int):
        return ([s[k].data_ptr() for s in self.src], [l[k].data_ptr() for l in self.lse],
                [d[k].data_ptr() for d in self.dst], [l[k].data_ptr() for l in self.lse_out])

    def call(self, k: int, flags: int):
        import decode_context_mla_dcp_gb300 as dcp
        src, lse, dst, lout = self.ptrs(k)
        c = self.cfg
        dcp.dcp_lse_reduce_ex(src, lse, c.cp, self.rows, c.H, c.D, c.lse_base_e, dcp.DCP_DTYPE_BF16, dst, lout,
                              flags=flags)

    def capture(self, flags: int, same_slot: bool = False):
        import torch
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self.call(0, flags)  # warm-up outside the capture
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for k in range(CALLS_PER_GRAPH):
                self.call(0 if same_slot else k % self.slots, flags)
        return g


def time_graphs(graphs, reps: int, flush=None):
    """Median us per call of each graph over `reps` replays (events on the
    current stream; optional L2 flush before each replay, outside the events)."""
    import torch
    out = {}
    for key, g in graphs.items():
        times = []
        for _ in range(reps):
            if flush is not None:
                flush.add_(1)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            g.replay()
            b.record()
            b.synchronize()
            times.append(a.elapsed_time(b) * 1e3 / CALLS_PER_GRAPH)
        out[key] = statistics.median(times)
    return out


def configs_extra(peak, flush, flags):
    """The other merge workloads, timed like the sweep (cold L2, 60 calls per
    graph, each on its own buffers where they fit, the sweep's launch flags):
    the DeepSeek-V2 sweep (cp=8, 128 heads, base-e [B, H, 1] LSE) and the
    speculative-decode batch (1024 rows, 10% empty shards). The default
    schedule reads the empty shards' payloads too (it issues every payload
    load beside the LSE loads), so its fraction of peak counts every byte; the
    LSE_FIRST schedule, which never reads them, is timed beside it on the
    skip-aware bytes."""
    import torch
    import decode_context_mla_dcp_gb300 as dcp
    from decode_context_mla_dcp_gb300.inputs import CONFIGS
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    l2 = int(getattr(props, "L2_cache_size", 0) or 0) or (126 << 20)
    out = {}
    for name in ("deepseek", "spec"):
        cfg = CONFIGS[name]
        res = {}
        for rows in cfg.rows:
            nbytes = dcp.algorithmic_bytes(cfg.cp, rows, cfg.H, cfg.D)
            slots = max(2, min(CALLS_PER_GRAPH, -(-4 * l2 // nbytes)))
            rs = RowSet(cfg, rows, slots)
            g = rs.capture(flags)
            us = time_graphs({rows: g}, reps=10, flush=flush)[rows]
            gbs = nbytes / (us * 1e-6) / 1e9
            entry = {"us_per_call": round(us, 3), "bytes_per_call": nbytes, "gbs": round(gbs, 1),
                     "frac_of_measured_peak": round(gbs / peak, 4),
                     "frac_of_nominal_8tbs": round(gbs / NOMINAL_HBM_GBS, 4)}
            if rs.inp.empty is not None:
                skipped = int(rs.inp.empty.sum()) * cfg.H  # (row, head, source) payload rows of weight 0
                skip_bytes = dcp.algorithmic_bytes(cfg.cp, rows, cfg.H, cfg.D, skipped_payload_rows=skipped)
                g2 = rs.capture(flags | dcp.DCP_FLAG_LSE_FIRST)
                us2 = time_graphs({rows: g2}, reps=10, flush=flush)[rows]
                del g2
                entry["empty_row_shards"] = int(rs.inp.empty.sum())
                entry["schedule"] = "default (PRELOAD): reads every payload, zero-weight ones included"
                entry["lse_first"] = {
                    "us_per_call": round(us2, 3), "skip_aware_bytes_per_call": skip_bytes,
                    "gbs": round(skip_bytes / (us2 * 1e-6) / 1e9, 1),
                    "frac_of_measured_peak": round(skip_bytes / (us2 * 1e-6) / 1e9 / peak, 4),
                    "schedule": "LSE_FIRST: reads the LSEs first and no zero-weight payload"}
            res[str(rows)] = entry
            del g, rs
            torch.cuda.empty_cache()
        out[f"{cfg.name} (cp={cfg.cp}, H={cfg.H}, D={cfg.D})"] = res
    return out


def stress_extra(peak, flags, sample_rows: int = 32):
    """Bandwidth-stress config (cp=8, 128 heads, D=512, 4096 rows, base-e LSE
    U[0, 30]): 4.85 GB per call, cold by size. Inputs drawn on the device with
    a seeded torch generator (same laws as the host generator). The inputs and
    outputs of `sample_rows` seeded rows of the timed call are kept on the host,
    so the CPU-baseline leg can check those bytes against the oracle."""
    import torch
    import decode_context_mla_dcp_gb300 as dcp
    cp, H, D, B = 8, 128, 512, 4096
    Hl = H // cp
    gen = torch.Generator(device="cuda")
    gen.manual_seed(0)
    src = [torch.randn((B, H, D), generator=gen, device="cuda", dtype=torch.float32).to(torch.bfloat16)
           for _ in range(cp)]
    lse = [torch.rand((B, H), generator=gen, device="cuda") * 30.0 for _ in range(cp)]
    dst = [torch.empty((B, Hl, D), dtype=torch.bfloat16, device="cuda") for _ in range(cp)]
    lout = [torch.empty((B, Hl), dtype=torch.float32, device="cuda") for _ in range(cp)]

    def call():
        dcp.dcp_lse_reduce_ex(src, lse, cp, B, H, D, True, dcp.DCP_DTYPE_BF16, dst, lout, flags=flags)

    for _ in range(3):
        call()
    torch.cuda.synchronize()
    times = []
    for _ in range(15):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(4):
            call()
        b.record()
        b.synchronize()
        times.append(a.elapsed_time(b) * 1e3 / 4)
    us = statistics.median(times)
    nbytes = dcp.algorithmic_bytes(cp, B, H, D)
    gbs = nbytes / (us * 1e-6) / 1e9
    rows = np.sort(np.random.default_rng(2024).choice(B, size=sample_rows, replace=False))
    idx = torch.from_numpy(rows).cuda()
    sample = {"rows": rows.tolist(),
              "srcs": [s[idx].contiguous().view(torch.int16).cpu().numpy().view(np.uint16) for s in src],
              "lses": [l[idx].contiguous().cpu().numpy() for l in lse],
              "outs": [d[idx].float().cpu().numpy().astype(np.float64) for d in dst],
              "lse_outs": [l[idx].cpu().numpy().astype(np.float64) for l in lout]}
    del src, lse, dst, lout
    torch.cuda.empty_cache()
    return ({"workload": "bandwidth stress: cp=8, H=128, D=512, rows=4096, bf16, base-e LSE U[0,30]",
             "us_per_call": round(us, 2), "bytes_per_call": nbytes, "gbs": round(gbs, 1),
             "frac_of_measured_peak": round(gbs / peak, 4), "frac_of_nominal_8tbs": round(gbs / NOMINAL_HBM_GBS, 4),
             "parity_sample_rows": sample_rows}, sample)


def timed_outputs_sample(sets):
    """What the timed graphs left in their output buffers: per row count,
    whether all of its calls' outputs are bit-identical (every call reads its
    own copy of the same inputs), and host copies of the first and the last
    call's outputs for the oracle check in the CPU-baseline leg."""
    import torch
    identical = True
    sample = {}
    for rows, rs in sets.items():
        for d in rs.dst + rs.lse_out:
            v = d.view(torch.int16) if d.dtype == torch.bfloat16 else d.view(torch.int32)
            identical &= bool((v == v[0:1]).all())
        sample[rows] = {k: ([d[k].float().double().cpu().numpy() for d in rs.dst],
                            [l[k].double().cpu().numpy() for l in rs.lse_out]) for k in (0, rs.slots - 1)}
    return {"calls_bit_identical": identical, "sample": sample}


def timed_outputs_parity(cfg, timed):
    """The first and the last call of every timed graph against the oracle on
    the same seeded inputs, at the parity tests' tolerances."""
    import oracle
    from decode_context_mla_dcp_gb300.inputs import make_merge_inputs
    worst_out = worst_lse = 0.0
    ok = bool(timed["calls_bit_identical"])
    for rows, by_call in timed["sample"].items():
        inp = make_merge_inputs(cfg, rows, seed=0)
        ref, lref = oracle.merge(inp.srcs, inp.lses, inp.lse_base_e)
        for outs, louts in by_call.values():
            for go, gl, ro, rl in zip(outs, louts, ref, lref):
                err = np.abs(go - ro)
                ok &= bool((err <= 1e-2 + 8e-3 * np.abs(ro)).all()) and not bool(np.isnan(go).any())
                worst_out = max(worst_out, float(err.max()))
                fin = np.isfinite(rl)
                ok &= bool(np.array_equal(np.isfinite(gl), fin))
                lerr = np.abs(gl[fin] - rl[fin]) / np.maximum(np.abs(rl[fin]), 1.0)
                if lerr.size:
                    ok &= bool((lerr <= 1e-5).all())
                    worst_lse = max(worst_lse, float(lerr.max()))
    return {"ok": ok, "calls_checked": "the first and the last of each row count's 60-call graph, as left by the "
                                       "timed steps", "calls_bit_identical": bool(timed["calls_bit_identical"]),
            "max_abs_err_out": worst_out, "max_rel_err_lse": worst_lse}


def stress_sample_parity(sample):
    """The stress call's sampled rows (inputs and GPU outputs of the timed
    launch) against the oracle, at the parity tests' tolerances."""
    import oracle
    ref, lref = oracle.merge(sample["srcs"], sample["lses"], True)
    worst_out = worst_lse = 0.0
    ok = True
    for go, gl, ro, rl in zip(sample["outs"], sample["lse_outs"], ref, lref):
        err = np.abs(go - ro)
        ok &= bool((err <= 1e-2 + 8e-3 * np.abs(ro)).all()) and not bool(np.isnan(go).any())
        worst_out = max(worst_out, float(err.max()))
        lerr = np.abs(gl - rl) / np.maximum(np.abs(rl), 1.0)
        ok &= bool((lerr <= 1e-5).all())
        worst_lse = max(worst_lse, float(lerr.max()))
    return {"ok": ok, "rows": len(sample["rows"]), "max_abs_err_out": worst_out, "max_rel_err_lse": worst_lse}


def mla_extras(hbm_peak, tensor_peak):
    """The DCP producer (split-KV MLA decode attention over one shard) and the
    fused single-GPU decode (producer over cp shards + merge), timed on
    DeepSeek-V2-shaped (128 heads) and Kimi-K2.5-shaped (64 heads) shards:
    Dk = 576 (512 latent + 64 RoPE), Dv = 512, bf16, 4096 shard tokens per row,
    8 rows. Ten calls per CUDA graph, each on its own KV cache (cold: 377 MB
    of caches > L2). Inputs drawn on the device with a seeded generator
    (timing only)."""
    import torch
    import decode_context_mla_dcp_gb300 as dcp
    from decode_context_mla_dcp_gb300.inputs import MLA_SCALE
    gen = torch.Generator(device="cuda")
    gen.manual_seed(0)
    out = {}
    n_calls, B, T = 10, 8, 4096
    # split counts chosen so that one launch is about one wave of one-CTA-per-SM blocks
    for name, H, cp, n_split, ns in (("deepseek-v2 shard, 128 heads", 128, 8, 1, 9),
                                     ("kimi-k2.5 shard, 64 heads", 64, 4, 4, 16)):
        q = torch.randn((B, H, 576), generator=gen, device="cuda").to(torch.bfloat16)
        kvs = [torch.randn((B, T, 576), generator=gen, device="cuda").to(torch.bfloat16) for _ in range(n_calls)]
        lens = torch.full((B,), T, dtype=torch.int32, device="cuda")
        po = [torch.empty((B, H, 512), dtype=torch.bfloat16, device="cuda") for _ in range(ns)]
        pl = [torch.empty((B, H), dtype=torch.float32, device="cuda") for _ in range(ns)]

        def timed(fn):
            fn(0)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for k in range(n_calls):
                    fn(k)
            ts = []
            for _ in range(10):
                a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                g.replay()
                e.record()
                e.synchronize()
                ts.append(a.elapsed_time(e) * 1e3 / n_calls)
            return statistics.median(ts)

        pf = dcp.DCP_FLAG_PDL | dcp.DCP_FLAG_PREFETCH
        us = timed(lambda k: dcp.mla_decode_partial(q, kvs[k], lens, MLA_SCALE, n_split=ns, outs=po, lses=pl,
                                                    flags=pf))
        us_nopf = timed(lambda k: dcp.mla_decode_partial(q, kvs[k], lens, MLA_SCALE, n_split=ns, outs=po, lses=pl,
                                                         flags=dcp.DCP_FLAG_PDL))
        us_mma = timed(lambda k: dcp.mla_decode_partial(q, kvs[k], lens, MLA_SCALE, n_split=ns, outs=po, lses=pl,
                                                        flags=pf | dcp.DCP_MLA_FLAG_MMA_SYNC))
        kv_bytes = B * T * 576 * 2
        nbytes = kv_bytes + B * H * 576 * 2 + ns * B * H * (512 * 2 + 4)
        flops = 2 * B * H * T * (576 + 512)
        out[f"producer, {name}"] = {
            "shape": f"B={B}, H={H}, shard tokens={T}, n_split={ns}", "us_per_call": round(us, 2),
            "gbs": round(nbytes / us / 1e3, 1), "tflops": round(flops / us / 1e6, 1),
            "frac_of_measured_hbm": round(nbytes / us / 1e3 / hbm_peak, 4),
            "frac_of_measured_bf16_tensor": round(flops / us / 1e6 / tensor_peak, 4),
            "kernel": {dcp.DCP_MLA_KERNEL_TCGEN05: "tcgen05", dcp.DCP_MLA_KERNEL_MMA_SYNC: "mma.sync"}[
                dcp.dcp_mla_decode_kernel(H, T, ns, pf)],
            "launch": "PDL + L2 prefetch of Q and the first KV tile before the dependency wait",
            "us_per_call_without_prefetch": round(us_nopf, 2),
            "mma_sync_kernel_us_per_call": round(us_mma, 2)}
        # fused: the same cache split over cp shards of T/cp tokens each
        Ts = T // cp
        shard_kvs = [[kvs[k][:, j * Ts:(j + 1) * Ts].contiguous() for j in range(cp)] for k in range(n_calls)]
        shard_lens = [torch.full((B,), Ts, dtype=torch.int32, device="cuda") for _ in range(cp)]
        ws = torch.empty((dcp.dcp_mla_decode_workspace_bytes(cp, n_split, B, H),), dtype=torch.uint8, device="cuda")
        fo = [torch.empty((B, H // cp, 512), dtype=torch.bfloat16, device="cuda") for _ in range(cp)]
        fl = [torch.empty((B, H // cp), dtype=torch.float32, device="cuda") for _ in range(cp)]
        us_f = timed(lambda k: dcp.mla_decode_dcp(q, shard_kvs[k], shard_lens, MLA_SCALE, n_split=n_split,
                                                  workspace=ws, outs=fo, lse_outs=fl, flags=pf))
        us_f1 = timed(lambda k: dcp.mla_decode_dcp(q, shard_kvs[k], shard_lens, MLA_SCALE, n_split=n_split,
                                                   workspace=ws, outs=fo, lse_outs=fl,
                                                   flags=pf | dcp.DCP_MLA_FLAG_ONE_KERNEL))
        # Its two launches apart. The producer's grid (cp*n_split slots of
        # Ts/n_split tokens x head blocks x rows) is that of one producer call
        # over the whole cache with cp*n_split splits, since shard j holds the
        # cache's tokens [j*Ts, (j+1)*Ts). The merge alone reads the
        # workspace's partials with the fused call's layout.
        n_src = cp * n_split
        pp = [torch.empty((B, H, 512), dtype=torch.bfloat16, device="cuda") for _ in range(n_src)]
        ppl = [torch.empty((B, H), dtype=torch.float32, device="cuda") for _ in range(n_src)]
        us_p = timed(lambda k: dcp.mla_decode_partial(q, kvs[k], lens, MLA_SCALE, n_split=n_src, outs=pp, lses=ppl,
                                                      flags=pf))
        Hs = H // n_src
        m_dst = [fo[k // n_split].data_ptr() + (k % n_split) * Hs * 512 * 2 for k in range(n_src)]
        m_lout = [fl[k // n_split].data_ptr() + (k % n_split) * Hs * 4 for k in range(n_src)]
        lay = dcp.Layout(src_row=H * 512, src_head=512, lse_row=H, lse_head=1, dst_row=(H // cp) * 512,
                         dst_head=512, lse_out_row=H // cp)
        us_m = timed(lambda k: dcp.dcp_lse_reduce_ex(pp, ppl, n_src, B, H, 512, True, dcp.DCP_DTYPE_BF16, m_dst,
                                                     m_lout, layout=lay, flags=dcp.DCP_FLAG_PDL))
        out[f"fused producer+merge, {name}"] = {
            "shape": f"B={B}, H={H}, cp={cp} shards x {Ts} tokens, n_split={n_split}", "us_per_call": round(us_f, 2),
            "kv_gbs": round(kv_bytes / us_f / 1e3, 1), "tflops": round(flops / us_f / 1e6, 1),
            "launches": "two (producer, then the merge; PDL)",
            "one_kernel_us_per_call": round(us_f1, 2),
            "one_kernel": "DCP_MLA_FLAG_ONE_KERNEL: the merge inside the producer's cooperative launch after a "
                          "grid-wide sync",
            "producer_alone_us": round(us_p, 2), "merge_alone_us": round(us_m, 2),
            "fused_minus_parts_us": round(us_f - us_p - us_m, 2),
            "how_split": "producer alone = one producer call over the whole cache with cp*n_split splits (the fused "
                         "launch's grid); merge alone = the merge over those partials with the fused layout; each "
                         "timed like the fused call (ten calls per graph, PDL; the producer with its L2 prefetch)"}
        del q, kvs, shard_kvs, po, pl, ws, fo, fl, pp, ppl
        torch.cuda.empty_cache()
    return out


def e2e_measure(cfg, steps: int):
    """The same metric end to end through the public API: every step copies
    all row counts' inputs from pinned host memory, merges each row count,
    and reads the merged outputs and LSEs back into pinned host memory.
    A step's inputs sit in one pinned host arena and its results in another,
    so each direction is one large copy instead of dozens of small ones."""
    import torch
    import decode_context_mla_dcp_gb300 as dcp
    from decode_context_mla_dcp_gb300.inputs import make_merge_inputs
    Hl = cfg.H // cfg.cp
    plan = []  # (rows, [(in offset, nbytes) for srcs + lses], [(out offset, nbytes) for outs + lse outs])
    off_in = off_out = 0
    nbytes = 0
    arrays = []
    for rows in cfg.rows:
        inp = make_merge_inputs(cfg, rows, seed=0)
        ins = []
        for a in list(inp.srcs) + list(inp.lses):
            b = np.ascontiguousarray(a).view(np.uint8).reshape(-1)
            ins.append((off_in, b.size))
            arrays.append((off_in, b))
            off_in += b.size
        outs = []
        for shape, esize in [((rows, Hl, cfg.D), 2)] * cfg.cp + [((rows, Hl), 4)] * cfg.cp:
            n = int(np.prod(shape)) * esize
            outs.append((off_out, n))
            off_out += n
        plan.append((rows, ins, outs))
        nbytes += dcp.algorithmic_bytes(cfg.cp, rows, cfg.H, cfg.D)
    host_in = torch.empty(off_in, dtype=torch.uint8).pin_memory()
    hv = host_in.numpy()
    for o, b in arrays:
        hv[o:o + b.size] = b
    host_out = [torch.empty(off_out, dtype=torch.uint8).pin_memory() for _ in range(2)]
    # Two device arenas per direction, so that step k+1's inputs can arrive
    # and step k-1's results can leave while step k merges.
    dev_in = [torch.empty(off_in, dtype=torch.uint8, device="cuda") for _ in range(2)]
    dev_out = [torch.empty(off_out, dtype=torch.uint8, device="cuda") for _ in range(2)]
    calls = [[], []]
    for k in range(2):
        for rows, ins, outs in plan:
            srcs = [dev_in[k][o:o + n].view(torch.bfloat16).view(rows, cfg.H, cfg.D) for o, n in ins[:cfg.cp]]
            lses = [dev_in[k][o:o + n].view(torch.float32).view(rows, cfg.H) for o, n in ins[cfg.cp:]]
            dsts = [dev_out[k][o:o + n].view(torch.bfloat16).view(rows, Hl, cfg.D) for o, n in outs[:cfg.cp]]
            lse_outs = [dev_out[k][o:o + n].view(torch.float32).view(rows, Hl) for o, n in outs[cfg.cp:]]
            calls[k].append((rows, srcs, lses, dsts, lse_outs))
    s_h2d, s_cmp, s_d2h = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    done_merge = [torch.cuda.Event(), torch.cuda.Event()]   # the merges of the step in slot k are done
    done_d2h = [torch.cuda.Event(), torch.cuda.Event()]     # slot k's results have left
    landed = [torch.cuda.Event(), torch.cuda.Event()]       # slot k's inputs have arrived

    def run(steps):
        for k in range(steps):
            b = k & 1
            with torch.cuda.stream(s_h2d):
                if k >= 2:
                    s_h2d.wait_event(done_merge[b])  # slot b's inputs were read by step k-2
                dev_in[b].copy_(host_in, non_blocking=True)
                landed[b].record(s_h2d)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(landed[b])
                if k >= 2:
                    s_cmp.wait_event(done_d2h[b])  # slot b's outputs of step k-2 have left
                for rows, srcs, lses, dsts, lse_outs in calls[b]:
                    dcp.dcp_lse_reduce(srcs, lses, cfg.H, cfg.cp, rows, cfg.H, cfg.D, cfg.lse_base_e, dsts,
                                       lse_outs, stream=s_cmp)
                done_merge[b].record(s_cmp)
            with torch.cuda.stream(s_d2h):
                s_d2h.wait_event(done_merge[b])
                host_out[b].copy_(dev_out[b], non_blocking=True)
                done_d2h[b].record(s_d2h)

    run(3)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    main = torch.cuda.current_stream()
    a.record(main)
    for st in (s_h2d, s_cmp, s_d2h):
        st.wait_stream(main)
    run(steps)
    for st in (s_h2d, s_cmp, s_d2h):
        main.wait_stream(st)
    b.record(main)
    b.synchronize()
    sec = a.elapsed_time(b) * 1e-3
    tot_sec, tot_bytes = aggregate_ranks(sec, float(nbytes * steps))
    return {"value": round(tot_bytes / tot_sec / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": off_in,
            "d2h_bytes_per_step": off_out, "ms_per_step": round(tot_sec * 1e3 / steps, 4),
            "how": "per step: one pinned host -> device copy of the step's inputs, dcp_lse_reduce for each row "
                   "count, one device -> pinned host copy of the step's outputs; copies and merges on three "
                   "streams with two arenas each, so consecutive steps overlap; timed with CUDA events"}


def cpu_baseline(cfg, budget_s: float = 12.0):
    """The CPU oracle as it stands (single-threaded fp64 C), on the sweep's
    inputs, repeated until about `budget_s` seconds of CPU work."""
    import oracle
    from decode_context_mla_dcp_gb300 import algorithmic_bytes
    from decode_context_mla_dcp_gb300.inputs import make_merge_inputs
    oracle.build()
    inputs = [make_merge_inputs(cfg, rows, seed=0) for rows in cfg.rows]
    per_pass = sum(algorithmic_bytes(cfg.cp, i.B, cfg.H, cfg.D) for i in inputs)
    passes, t0 = 0, time.perf_counter()
    while True:
        for inp in inputs:
            oracle.merge(inp.srcs, inp.lses, inp.lse_base_e)
        passes += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    out = {"value": round(per_pass * passes / el / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
           "sample": f"{passes} passes over the rows {list(cfg.rows)} sweep ({per_pass} algorithmic bytes each), "
                     f"{el:.1f} s, single-threaded fp64 C"}
    out["all_cores"] = cpu_baseline_all_cores(cfg, budget_s / 2)
    out["parity_vs_oracle"] = sweep_parity(cfg, inputs)
    return out


def sweep_parity(cfg, inputs):
    """The timed path (dcp_lse_reduce_ex with the sweep's flags) on its inputs
    against the oracle: outputs within |gpu - ref| <= 1e-2 + 8e-3 |ref|,
    merged LSEs within 1e-5 * max(|ref|, 1)."""
    import torch
    import oracle
    import decode_context_mla_dcp_gb300 as dcp
    worst_out = worst_lse = 0.0
    ok = True
    for inp in inputs:
        srcs = [torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda() for x in inp.srcs]
        lses = [torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in inp.lses]
        got_o, got_l = dcp.merge(srcs, lses, inp.lse_base_e, flags=dcp.DCP_FLAG_PDL | dcp.DCP_FLAG_PREFETCH)
        torch.cuda.synchronize()
        ref_o, ref_l = oracle.merge(inp.srcs, inp.lses, inp.lse_base_e)
        for go, gl, ro, rl in zip(got_o, got_l, ref_o, ref_l):
            go = go.float().double().cpu().numpy()
            gl = gl.double().cpu().numpy()
            err = np.abs(go - ro)
            ok &= bool((err <= 1e-2 + 8e-3 * np.abs(ro)).all())
            worst_out = max(worst_out, float(err.max()))
            fin = np.isfinite(rl)
            ok &= bool(np.array_equal(np.isfinite(gl), fin))
            lerr = np.abs(gl[fin] - rl[fin]) / np.maximum(np.abs(rl[fin]), 1.0)
            if lerr.size:
                ok &= bool((lerr <= 1e-5).all())
                worst_lse = max(worst_lse, float(lerr.max()))
    return {"ok": ok, "rows": [int(i.B) for i in inputs], "max_abs_err_out": worst_out,
            "max_rel_err_lse": worst_lse}


def _oracle_worker(args):
    """One process of the all-cores oracle run: the same single-threaded
    loop over the sweep for about `budget_s` seconds."""
    cfg_name, budget_s = args
    sys.path.insert(0, ROOT)
    import oracle
    from decode_context_mla_dcp_gb300 import algorithmic_bytes
    from decode_context_mla_dcp_gb300.inputs import CONFIGS, make_merge_inputs
    cfg = CONFIGS[cfg_name]
    inputs = [make_merge_inputs(cfg, rows, seed=0) for rows in cfg.rows]
    per_pass = sum(algorithmic_bytes(cfg.cp, i.B, cfg.H, cfg.D) for i in inputs)
    passes, t0 = 0, time.perf_counter()
    while True:
        for inp in inputs:
            oracle.merge(inp.srcs, inp.lses, inp.lse_base_e)
        passes += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            return per_pass * passes, el


def cpu_baseline_all_cores(cfg, budget_s: float):
    """The oracle as it stands on every host core this process may use: one
    spawned process per core, each running the single-threaded loop
    concurrently; throughput = all bytes / the longest process time."""
    import multiprocessing as mp
    from decode_context_mla_dcp_gb300.inputs import CONFIGS
    name = next(k for k, v in CONFIGS.items() if v == cfg)
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    with mp.get_context("spawn").Pool(cores) as pool:
        res = pool.map(_oracle_worker, [(name, budget_s)] * cores)
    total = sum(r[0] for r in res)
    el = max(r[1] for r in res)
    return {"value": round(total / el / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{cores} concurrent processes (spawned; os.sched_getaffinity gives {cores} cores), "
                      f"each the single-threaded loop over the sweep for about {budget_s:.0f} s"}


# ---------------------------------------------------------------------------- arms

def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    from decode_context_mla_dcp_gb300 import algorithmic_bytes
    from decode_context_mla_dcp_gb300.inputs import make_merge_inputs
    cfg = workload_config()
    oracle.build()
    inputs = [make_merge_inputs(cfg, rows, seed=0) for rows in cfg.rows]
    per_step = sum(algorithmic_bytes(cfg.cp, i.B, cfg.H, cfg.D) for i in inputs)

    def step():
        for inp in inputs:
            oracle.merge(inp.srcs, inp.lses, inp.lse_base_e)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    sec = time.perf_counter() - t0
    value = per_step * args.steps / sec / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec * 1e3 / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_dict(cfg),
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": f"each step = one pass of the fp64 C oracle over rows {list(cfg.rows)}"},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def config_dict(cfg):
    return {"workload": f"{cfg.name} DCP LSE merge: cp={cfg.cp}, H={cfg.H} ({cfg.H // cfg.cp} per destination), "
                        f"D={cfg.D}, bf16 partials N(0,1), base-2 fp32 LSE U[-4,24], rows {list(cfg.rows)}",
            "cp": cfg.cp, "heads": cfg.H, "head_dim": cfg.D, "rows": list(cfg.rows),
            "calls_per_graph": CALLS_PER_GRAPH,
            "launch": "programmatic dependent launch; each warp brings its inputs into L2 before it waits for the "
                      "previous call (DCP_FLAG_PDL | DCP_FLAG_PREFETCH)",
            "l2": "flushed before every step (write of 4x L2); each of a graph's 60 calls has its own buffers",
            "parallelism": "replicas (one independent merge workload per GPU)"}


def run_ours(args):
    import torch
    import torch.distributed as dist

    import decode_context_mla_dcp_gb300 as dcp
    from decode_context_mla_dcp_gb300 import build as dcp_build

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dcp_build.build()
    dcp.load()
    cfg = workload_config()
    peak, peak_kind = measured_peaks()
    props = torch.cuda.get_device_properties(local)
    l2 = int(getattr(props, "L2_cache_size", 0) or 0) or (126 << 20)
    flush = torch.zeros((max(4 * l2, 512 << 20) // 4,), dtype=torch.float32, device="cuda")
    uuid = None
    try:
        uuid = "GPU-" + str(props.uuid)
    except Exception:
        pass

    flags = dcp.DCP_FLAG_PDL | dcp.DCP_FLAG_PREFETCH
    bytes_per_rows = sweep_bytes(cfg)
    step_bytes = sum(bytes_per_rows.values()) * CALLS_PER_GRAPH
    sets = {rows: RowSet(cfg, rows, CALLS_PER_GRAPH) for rows in cfg.rows}
    graphs = {rows: sets[rows].capture(flags) for rows in cfg.rows}
    torch.cuda.synchronize()

    def step(record=None):
        flush.add_(1.0)  # evict L2 (outside the step's events)
        if record is not None:
            record[0].record()
        for i, rows in enumerate(cfg.rows):
            graphs[rows].replay()
            if record is not None:
                record[i + 1].record()

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(cfg.rows) + 1)] for _ in range(args.steps)]
    sampler = clock_sampler(uuid)
    sampler.start()
    time.sleep(0.3 if isinstance(sampler, ClockSampler) else 0.02)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for k in range(args.steps):
        step(evs[k])
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - wall0
    clocks = sampler.stop()
    timed = timed_outputs_sample(sets) if rank == 0 and world == 1 and not args.no_cpu_baseline else None

    step_ms = [evs[k][0].elapsed_time(evs[k][-1]) for k in range(args.steps)]
    per_rows_us = {rows: statistics.median(evs[k][i].elapsed_time(evs[k][i + 1]) * 1e3 / CALLS_PER_GRAPH
                                           for k in range(args.steps))
                   for i, rows in enumerate(cfg.rows)}
    local_sec = sum(step_ms) * 1e-3
    tot_sec, tot_bytes = aggregate_ranks(local_sec, step_bytes * args.steps)
    value = tot_bytes / tot_sec / 1e9
    achieved = step_bytes * args.steps / local_sec / 1e9

    out = {"metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": round(tot_sec * 1e3 / args.steps, 4),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
           "data": "synthetic", "config": config_dict(cfg),
           "wall_ms_per_step": round(wall * 1e3 / args.steps, 4),
           "gpu_launches": args.steps * len(cfg.rows) * CALLS_PER_GRAPH,
           "sweep": {str(rows): {"us_per_call": round(per_rows_us[rows], 3), "bytes_per_call": bytes_per_rows[rows],
                                 "gbs": round(bytes_per_rows[rows] / (per_rows_us[rows] * 1e-6) / 1e9, 1),
                                 "frac_of_measured_peak": round(bytes_per_rows[rows] / (per_rows_us[rows] * 1e-6)
                                                                / 1e9 / peak, 4),
                                 "frac_of_nominal_8tbs": round(bytes_per_rows[rows] / (per_rows_us[rows] * 1e-6)
                                                               / 1e9 / NOMINAL_HBM_GBS, 4)}
                     for rows in cfg.rows},
           "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                        "frac": round(achieved / peak, 4), "traffic": recorded_traffic(),
                        "frac_of_nominal_8tbs": round(achieved / NOMINAL_HBM_GBS, 4),
                        "peak_kind": f"{peak_kind} (burst copy bandwidth)",
                        "per_unit": "algorithmic bytes per call = cp*B*H*D*2 + cp*B*H*4 + B*H*D*2 + B*H*4",
                        "bytes_per_launch_avg": step_bytes / (len(cfg.rows) * CALLS_PER_GRAPH)},
           "clocks": clocks}

    if rank == 0 and not args.no_extras:
        hot = {rows: sets[rows].capture(flags, same_slot=True) for rows in cfg.rows}
        nopdl = {rows: sets[rows].capture(0) for rows in cfg.rows}
        nopf = {rows: sets[rows].capture(dcp.DCP_FLAG_PDL) for rows in cfg.rows}
        hot_us = time_graphs(hot, 20)
        cold_nopdl_us = time_graphs(nopdl, 20, flush=flush)
        cold_nopf_us = time_graphs(nopf, 20, flush=flush)
        out["extras"] = {
            "l2_hot_us_per_call": {str(r): round(v, 3) for r, v in hot_us.items()},
            "cold_no_pdl_no_prefetch_us_per_call": {str(r): round(v, 3) for r, v in cold_nopdl_us.items()},
            "cold_pdl_no_prefetch_us_per_call": {str(r): round(v, 3) for r, v in cold_nopf_us.items()},
        }
        del hot, nopdl, nopf
    out["e2e"] = e2e_measure(cfg, max(10, min(args.steps, 100)))
    stress_sample = None
    if rank == 0 and not args.no_extras:
        del sets, graphs
        torch.cuda.empty_cache()
        out["extras"]["other_configs_cold"] = configs_extra(peak, flush, flags)
        out["extras"]["largest_config"], stress_sample = stress_extra(peak, flags)
        out["extras"]["dcp_producer_and_fused_decode"] = mla_extras(peak, measured_tensor_peak())
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(cfg)
        if stress_sample is not None:
            out["cpu_baseline"]["parity_vs_oracle"]["stress_sample"] = stress_sample_parity(stress_sample)
        if timed is not None:
            out["cpu_baseline"]["parity_vs_oracle"]["timed_calls"] = timed_outputs_parity(cfg, timed)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_case(args):
    """A few plain calls of one config, for ncu captures: `--case NAME
    --rows R1,R2,... --calls N` calls the merge N times per row count, each
    call on its own buffers, with no graph and no timing."""
    import torch
    import decode_context_mla_dcp_gb300 as dcp
    from decode_context_mla_dcp_gb300 import build as dcp_build
    from decode_context_mla_dcp_gb300.inputs import CONFIGS, make_merge_inputs
    torch.cuda.set_device(dist_env()[2])
    dcp_build.build()
    if args.case == "mla":
        # the producer on a DeepSeek-V2-shaped shard, as the bench times it: 8 rows x 128 heads x 4096
        # tokens, 9 splits (one wave), PDL and the L2 prefetch (--mla-kernel / --mla-splits change the
        # kernel and the split count)
        from decode_context_mla_dcp_gb300.inputs import MLA_SCALE
        gen = torch.Generator(device="cuda")
        gen.manual_seed(0)
        B, H, T = 8, 128, 4096
        q = torch.randn((B, H, 576), generator=gen, device="cuda").to(torch.bfloat16)
        kvs = [torch.randn((B, T, 576), generator=gen, device="cuda").to(torch.bfloat16) for _ in range(args.calls)]
        lens = torch.full((B,), T, dtype=torch.int32, device="cuda")
        kflags = {"auto": 0, "tcgen05": dcp.DCP_MLA_FLAG_TCGEN05, "mma_sync": dcp.DCP_MLA_FLAG_MMA_SYNC}[args.mla_kernel]
        for kv in kvs:
            dcp.mla_decode_partial(q, kv, lens, MLA_SCALE, n_split=args.mla_splits,
                                   flags=dcp.DCP_FLAG_PDL | dcp.DCP_FLAG_PREFETCH | kflags)
        torch.cuda.synchronize()
        print(f"case mla x {args.calls} calls done", flush=True)
        return 0
    if args.case == "fused":
        # the fused decode as the bench times it: 8 rows x 128 heads, cp = 8 shards of 512 tokens, one split
        # per shard, PDL and the producer's L2 prefetch; each call on its own caches
        from decode_context_mla_dcp_gb300.inputs import MLA_SCALE
        gen = torch.Generator(device="cuda")
        gen.manual_seed(0)
        B, H, cp, Ts = 8, 128, 8, 512
        q = torch.randn((B, H, 576), generator=gen, device="cuda").to(torch.bfloat16)
        lens = [torch.full((B,), Ts, dtype=torch.int32, device="cuda") for _ in range(cp)]
        caches = [[torch.randn((B, Ts, 576), generator=gen, device="cuda").to(torch.bfloat16) for _ in range(cp)]
                  for _ in range(args.calls)]
        torch.cuda.synchronize()
        for kvs in caches:
            dcp.mla_decode_dcp(q, kvs, lens, MLA_SCALE, n_split=1, flags=dcp.DCP_FLAG_PDL | dcp.DCP_FLAG_PREFETCH)
        torch.cuda.synchronize()
        print(f"case fused x {args.calls} calls done", flush=True)
        return 0
    cfg = CONFIGS[args.case]
    rows_list = [int(r) for r in args.rows.split(",")] if args.rows else list(cfg.rows)
    flags = dcp.DCP_FLAG_PDL | dcp.DCP_FLAG_PREFETCH
    if args.schedule == "lse_first":
        flags |= dcp.DCP_FLAG_LSE_FIRST
    for rows in rows_list:
        inp = make_merge_inputs(cfg, rows, seed=0)
        Hl = cfg.H // cfg.cp
        sets = []
        for _ in range(args.calls):
            src = [torch.from_numpy(s.view(np.int16)).view(torch.bfloat16).cuda() for s in inp.srcs]
            lse = [torch.from_numpy(l).cuda() for l in inp.lses]
            dst = [torch.empty((rows, Hl, cfg.D), dtype=torch.bfloat16, device="cuda") for _ in range(cfg.cp)]
            lout = [torch.empty((rows, Hl), dtype=torch.float32, device="cuda") for _ in range(cfg.cp)]
            sets.append((src, lse, dst, lout))
        torch.cuda.synchronize()
        for src, lse, dst, lout in sets:
            dcp.dcp_lse_reduce_ex(src, lse, cfg.cp, rows, cfg.H, cfg.D, cfg.lse_base_e, dcp.DCP_DTYPE_BF16,
                                  dst, lout, flags=flags)
        torch.cuda.synchronize()
        del sets
        torch.cuda.empty_cache()
    print(f"case {args.case} rows {rows_list} x {args.calls} calls done", flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extras", action="store_true", help="skip the L2-hot, no-PDL and stress extras")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--case", choices=["kimi", "deepseek", "spec", "stress", "mla", "fused"],
                    help="profiling mode: plain calls of one config, no timing")
    ap.add_argument("--rows", default="", help="with --case: comma-separated row counts")
    ap.add_argument("--calls", type=int, default=3, help="with --case: calls per row count")
    ap.add_argument("--mla-kernel", choices=["auto", "tcgen05", "mma_sync"], default="auto",
                    help="with --case mla: the producer kernel")
    ap.add_argument("--mla-splits", type=int, default=9, help="with --case mla: splits per row")
    ap.add_argument("--schedule", choices=["default", "lse_first"], default="default",
                    help="with --case (merge configs): the merge schedule")
    args = ap.parse_args(argv)
    if args.case:
        return run_case(args)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
