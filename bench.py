"""Benchmark of the Ulysses QKV front end on one GB300.

Headline step: one pass of the whole hot path over one batch of the largest
fused workload, "h8192_p8_b2_s16384" (P=8 virtual ranks x B=2 x S_local=2048 =
32768 tokens, hidden 8192, 64 heads, bshd, 13.19 TFLOP of projection):
  1. qnre_forward: fused QKV projection + RMSNorm + RoPE + band scatter of every
     token into the 8 ranks' [B, S_global, 8, 128] bands;
  2. the head-chunk pack of every band of the uneven schedule
     [(0,2),(2,4),(6,2)] over H_local = 8, on strided q/k/v views of a
     [P*B, S_local, 3, 64, 128] projection buffer (all virtual ranks, all bands
     in one ulysses_pack_head_chunk_schedule launch);
  3. the merge of each packed band's q slice back into a [P*B, S_local, 64, 128]
     output (one ulysses_merge_output_head_chunk_schedule launch; pack then
     merge reproduces q).
Steps 2-3 do not depend on step 1; by default they run on a second stream
beside it (--no-overlap serialises everything on one stream).  The inputs
(2.1 GB) and outputs are larger than the 129 MB L2, which is also flushed with
a 512 MB write between steps.  value = tokens of the step / step time.

The same JSON line reports rows timed alone (CUDA events around serialised
launches, L2 flushed between repetitions):
  * "pack" / "merge": the head-chunk pack and merge of [1, 37760, 56, 128] over
    two virtual ranks with the schedule [7, 14, 7] (the pages' shape), per
    chunk and as schedule calls;
  * "pack_output_sequence_chunk", "layout_rows" (scatter/gather heads and the
    composed head-chunk exchanges) and "sage2" over the same q/k/v;
  * "fused_h4096_p4_s4096": the fused op alone on the 4096-token workload;
  * "fused_alone" and "unfused_torch": the headline workload's fused op alone,
    and the same operator as separate PyTorch ops (cuBLAS GEMM, RMSNorm, RoPE,
    band scatter) with the fused kernel's speedup over it.

"e2e" runs the step through the same API with every step's inputs copied
from pinned host memory and its outputs copied back (three buffer sets, copy
streams overlapping compute), beside the same copies timed alone (the host
link's floor on the box).

This benchmark runs on one GPU: it refuses WORLD_SIZE > 1 and --gpus > 1 (the
fused kernel's two-pair clusters multicast W inside a cluster, and nothing on
this path exchanges data between GPUs).

`--impl reference` times the CPU oracle on the host cores instead: every step
is a bounded stratified sample of the same workload through the fp64
projection/norm/RoPE/placement, plus pack/merge of the matching rows.
"""
from __future__ import annotations

import argparse
import contextlib
import ctypes
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from ulysses_qkv_proj_gb300 import workloads as WL  # noqa: E402

METRIC = "fused QKV+norm+RoPE+scatter tokens/s & % bf16 TC peak; pack/merge GB/s % HBM"
WORKLOAD = WL.FUSED_WORKLOADS[WL.BENCH_FUSED]
SMALL_FUSED = WL.FUSED_WORKLOADS[WL.BENCH_FUSED_SMALL]
HEADCHUNK = WL.HEADCHUNK_WORKLOADS[WL.BENCH_HEADCHUNK]
SCHEDULE = WL.BENCH_SCHEDULE
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# the fused kernel and the host code that sets its launch shape and raster
FUSED_SOURCES = ["ulysses_qkv_proj_gb300/csrc/fused_qkv.cu", "ulysses_qkv_proj_gb300/csrc/fused_qkv.cuh",
                 "ulysses_qkv_proj_gb300/csrc/ptx.cuh", "ulysses_qkv_proj_gb300/csrc/qnre_api.cu"]
TRAFFIC_FILE = "profiles/traffic.json"


def fused_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in FUSED_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM read + write bytes per launch of the fused kernel on `workload`, from the
    committed ncu counters, or None when they were taken on other kernel sources."""
    path = os.path.join(ROOT, TRAFFIC_FILE)
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get("fused_qkv_kernel", {}).get(workload)
    if not rec or rec.get("kernel_source_hash") != fused_source_hash():
        return None
    return int(rec["dram_bytes_per_launch"])


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def refuse_multi_gpu(args) -> None:
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world > 1 or args.gpus > 1:
        sys.stderr.write(f"bench.py: one GPU only (WORLD_SIZE={world}, --gpus={args.gpus}): the fused kernel's "
                         "two-pair clusters multicast W within a cluster, and this path has no exchange "
                         "between GPUs\n")
        raise SystemExit(2)


# ----------------------------------------------------------------------------
# clocks sampled during the timed regions (read-only queries)
# ----------------------------------------------------------------------------
class ClockSampler:
    """Polls the GPU's SM clock, power and clock-event reasons every `period_s`
    through NVML (ctypes on the driver's libnvidia-ml), else through
    `nvidia-smi -lms`, while the benchmark runs.  `section(name)` records the
    wall-clock interval of a timed region; `summary(name)` reduces the samples
    inside it.  Nothing here sets or resets any GPU setting."""

    REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                   0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
    SMI_FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
                  "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                  "clocks_event_reasons.sw_power_cap")

    def __init__(self, pci_bus_id: str, period_s: float = 0.005):
        self.pci = pci_bus_id
        self.period = period_s
        self.samples = []        # (t, sm_mhz, max_mhz, power_w, reasons frozenset)
        self.sections = {}
        self.source = None
        self._stop = threading.Event()
        self._thread = None
        self._proc = None
        self._nvml = None
        self._h = None

    # -- NVML
    def _nvml_open(self) -> bool:
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return False
            h = ctypes.c_void_p()
            for bus in (self.pci, self.pci[4:]):
                if lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) == 0:
                    break
            else:
                return False
            self._nvml, self._h = lib, h
            self._reason_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                lib.nvmlDeviceGetCurrentClocksThrottleReasons
            return self._nvml_sample() is not None
        except (OSError, AttributeError):
            return False

    def _nvml_sample(self):
        lib, h = self._nvml, self._h
        sm, mx, pw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(sm)) != 0:   # NVML_CLOCK_SM
            return None
        lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))
        lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(pw))
        self._reason_fn(h, ctypes.byref(rs))
        reasons = frozenset(n for bit, n in self.REASON_BITS.items() if rs.value & bit)
        return (time.perf_counter(), float(sm.value), float(mx.value), pw.value / 1000.0, reasons)

    def _nvml_loop(self):
        while not self._stop.is_set():
            s = self._nvml_sample()
            if s is not None:
                self.samples.append(s)
            time.sleep(self.period)

    # -- nvidia-smi fallback
    def _smi_loop(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self._proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm, mx, pw = float(parts[0]), float(parts[1]), float(parts[2])
            except ValueError:
                continue
            reasons = frozenset(n for n, v in zip(names, parts[3:7]) if v.lower() == "active")
            self.samples.append((time.perf_counter(), sm, mx, pw, reasons))

    def start(self):
        if self._nvml_open():
            self.source = f"NVML every {self.period * 1e3:g} ms"
            self._thread = threading.Thread(target=self._nvml_loop, daemon=True)
        else:
            try:
                self._proc = subprocess.Popen(
                    ["nvidia-smi", "-i", self.pci, f"--query-gpu={self.SMI_FIELDS}", "--format=csv,noheader,nounits",
                     "-lms", "10"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except OSError:
                self.source = "unavailable"
                return self
            self.source = "nvidia-smi -lms 10"
            self._thread = threading.Thread(target=self._smi_loop, daemon=True)
        self._thread.start()
        return self

    def stop(self):
        self._stop.set()
        if self._proc is not None:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self._proc.kill()
        if self._thread is not None:
            self._thread.join(timeout=2)
        if self._nvml is not None:
            self._nvml.nvmlShutdown()

    @contextlib.contextmanager
    def section(self, name: str):
        t0 = time.perf_counter()
        try:
            yield
        finally:
            self.sections[name] = (t0, time.perf_counter())

    def summary(self, name: str):
        if name not in self.sections or self.source == "unavailable":
            return {"sm_mhz": None, "sm_max_mhz": None, "samples": 0, "reasons": [], "source": self.source}
        t0, t1 = self.sections[name]
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        reasons = sorted(set().union(*[s[4] for s in inside])) if inside else []
        sm = [s[1] for s in inside]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(s[2] for s in inside) if inside else None,
                "sm_mhz_min": min(sm) if sm else None,
                "power_w_max": round(max(s[3] for s in inside), 1) if inside else None,
                "samples": len(inside), "reasons": reasons, "source": self.source,
                "region_s": round(t1 - t0, 4)}


def pci_bus_id(torch, dev) -> str:
    """PCI bus id of the CUDA device as NVML and nvidia-smi name it (domain:bus:device.0)."""
    props = torch.cuda.get_device_properties(dev)
    return "%08x:%02x:%02x.0" % (getattr(props, "pci_domain_id", 0), getattr(props, "pci_bus_id", 0),
                                 getattr(props, "pci_device_id", 0))


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------
class Gpu:
    """Device helpers shared by the timed sections."""

    def __init__(self, torch, dev):
        self.torch = torch
        self.dev = dev
        self.flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.int32, device=dev)
        khz = getattr(torch.cuda.get_device_properties(dev), "clock_rate", 0) or 2_000_000
        self.sleep_cycles = int(2e-3 * khz * 1e3)  # about 2 ms of GPU time

    def bf16(self, a):
        t = self.torch
        return t.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(t.bfloat16).to(self.dev)

    def timed_alone(self, fn, steps: int, warmup: int):
        """Mean and median CUDA-event time (ms) of fn() on the current stream, L2
        flushed between repetitions (outside the events).  Each repetition is queued
        behind a 2 ms GPU sleep, so fn's launches run back to back on the device
        however long the host takes to enqueue them: the events time the kernels,
        not the Python calls between them."""
        torch = self.torch
        for _ in range(warmup):
            fn()
            self.flush.zero_()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for a, b in evs:
            torch.cuda._sleep(self.sleep_cycles)
            a.record()
            fn()
            b.record()
            self.flush.zero_()
        torch.cuda.synchronize()
        ms = [a.elapsed_time(b) for a, b in evs]
        return statistics.mean(ms), statistics.median(ms)


def fused_setup(gpu, qb, wl, inp=None):
    torch = gpu.torch
    inp = inp or WL.make_fused_inputs(wl)
    d = {"x": gpu.bf16(inp.x), "w": gpu.bf16(inp.w), "qw": gpu.bf16(inp.q_norm_w), "kw": gpu.bf16(inp.k_norm_w),
         "cs": torch.from_numpy(inp.cos_sin).to(gpu.dev), "pos": torch.from_numpy(inp.positions).to(gpu.dev)}
    plan = qb.Plan(wl.hidden, wl.num_heads, wl.P, wl.layout, max_tokens=wl.B * wl.S, rope_style=wl.rope_style)
    return inp, d, plan


def time_fused_alone(gpu, qb, wl, peaks, peak_src, steps, warmup, inp=None):
    """The fused op alone on `wl`; fraction of the burst tensor peak."""
    _, d, plan = fused_setup(gpu, qb, wl, inp)
    out = qb.alloc_outputs(plan, wl.B, wl.S, gpu.dev)
    ms, med = gpu.timed_alone(lambda: qb.qnre_forward(plan, d["x"], d["w"], d["qw"], d["kw"], d["cs"], d["pos"], out),
                              steps, warmup)
    if plan.device_status() != 0:
        raise RuntimeError("device status raised")
    info = plan.describe(wl.B, wl.S)
    plan.destroy()
    tflops = wl.flops() / (ms * 1e-3) / 1e12
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    return {"workload": wl.name, "tokens": wl.T, "ms": round(ms, 5), "ms_median": round(med, 5),
            "tflops": round(tflops, 1), "tokens_per_s": round(wl.T / (ms * 1e-3), 1),
            "frac": round(tflops / peak, 4), "peak": peak, "peak_source": f"{peak_src} bf16_tflops (burst)",
            "clusters": info["clusters"], "pairs_per_cluster": info["pairs_per_cluster"],
            "launches": steps, "timing": "alone, launch queued behind a GPU sleep, L2 flushed between launches"}


def unfused_torch_forward(torch, wl, d, out):
    """The same operator as separate PyTorch ops (a per-operator path like the pages'
    baselines): a cuBLAS bf16 GEMM, RMSNorm and rotate-half RoPE of q and k in fp32,
    a bf16 cast, and the band scatter as one permuted copy per q/k/v.  A comparator
    timed beside the fused kernel, not part of the library."""
    P, B, S, H, D, L = wl.P, wl.B, wl.S, wl.num_heads, 128, wl.H_local
    T = wl.T
    y = torch.matmul(d["x"].view(T, wl.hidden), d["w"]).view(T, 3, H, D)
    qk = y[:, :2].float()
    rinv = torch.rsqrt(qk.pow(2).mean(-1, keepdim=True) + 1e-6)
    n = qk * rinv * torch.stack([d["qw"], d["kw"]]).float().view(1, 2, 1, D)
    cs = d["cs"][d["pos"].view(-1).long()]
    cos, sin = cs[:, None, None, :64], cs[:, None, None, 64:]
    n1, n2 = n[..., :64], n[..., 64:]
    rot = torch.cat([n1 * cos - n2 * sin, n2 * cos + n1 * sin], -1).to(torch.bfloat16)
    # token (r_s, b, s), head h = r * L + hl -> band r, batch b, global row r_s * S + s, local head hl
    for g, src in (("q", rot[:, 0]), ("k", rot[:, 1]), ("v", y[:, 2])):
        out[g].view(P, B, P, S, L, D).copy_(src.reshape(P, B, S, P, L, D).permute(3, 1, 0, 2, 4, 5))


def time_unfused_alone(gpu, qb, wl, fused_ms, steps, warmup, inp=None):
    """The per-operator PyTorch path on `wl`, checked against the fused kernel's
    output, and the fused kernel's speedup over it."""
    torch = gpu.torch
    _, d, plan = fused_setup(gpu, qb, wl, inp)
    ref = qb.alloc_outputs(plan, wl.B, wl.S, gpu.dev)
    qb.qnre_forward(plan, d["x"], d["w"], d["qw"], d["kw"], d["cs"], d["pos"], ref)
    out = {g: torch.empty_like(t) for g, t in ref.items()}
    ms, med = gpu.timed_alone(lambda: unfused_torch_forward(torch, wl, d, out), steps, warmup)
    # the two paths round differently (bf16 GEMM output before the norm here): compare loosely
    err = max(float((out[g].float() - ref[g].float()).abs().max()) for g in ref)
    if not err < 0.25:
        raise RuntimeError(f"per-operator path disagrees with the fused kernel (max |diff| {err})")
    plan.destroy()
    return {"ms": round(ms, 5), "ms_median": round(med, 5), "speedup_of_fused": round(ms / fused_ms, 3),
            "max_abs_diff_vs_fused": round(err, 5),
            "ops": "torch.matmul (cuBLAS bf16) + fp32 RMSNorm and rotate-half RoPE of q, k + bf16 cast + "
                   "one permuted copy per q/k/v into the bands",
            "timing": "alone, launches queued behind a GPU sleep, L2 flushed between repetitions; the speedup "
                      "divides by the fused kernel alone on the same workload (fused_alone)"}


def time_headchunk_alone(gpu, qb, wl, peaks, peak_src, steps, warmup):
    """Pack and merge over the pages' head-chunk shape: every chunk of the schedule
    for every virtual rank, per chunk (one launch each) and as schedule calls (one
    launch per rank); then the ordinary and composed exchanges and Sage2 over the
    same q/k/v."""
    torch = gpu.torch
    buf = gpu.bf16(WL.make_headchunk_buffer(wl.B, wl.S_global, wl.num_heads, wl.D))
    W, L, D, S, P = wl.P, wl.H_local, wl.D, wl.S, wl.P
    views = [(buf[:, r * S:(r + 1) * S, 0], buf[:, r * S:(r + 1) * S, 1], buf[:, r * S:(r + 1) * S, 2])
             for r in range(P)]
    packed = [[torch.empty((wl.B, S, W * cnt, 3 * D), dtype=torch.bfloat16, device=gpu.dev) for _, cnt in wl.schedule]
              for _ in range(P)]
    merged = [torch.empty((wl.B, S, wl.num_heads, D), dtype=torch.bfloat16, device=gpu.dev) for _ in range(P)]
    offs = [off for off, _ in wl.schedule]
    n_chunks = len(wl.schedule)
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))

    def row(ms, med, nbytes, launches, form):
        g = nbytes / (ms * 1e-3) / 1e9
        return {"ms": round(ms, 5), "ms_median": round(med, 5), "bytes": nbytes, "GB/s": round(g, 1),
                "frac_hbm": round(g / hbm, 4), "peak": hbm, "peak_source": f"{peak_src} hbm_gbs",
                "launches": launches, "form": form,
                "timing": "alone, launches queued behind a GPU sleep, L2 flushed between repetitions"}

    def pack_chunks():
        for r, (q, k, v) in enumerate(views):
            for i, (off, cnt) in enumerate(wl.schedule):
                qb.ulysses_pack_head_chunk(q, k, v, W, off, cnt, packed[r][i])

    # the merge input of each chunk: the gathered output band, contiguous
    # [B, S, W*cnt, D] as the pages define it (here the packed q slice, so pack then
    # merge reproduces q)
    received = [[None] * n_chunks for _ in range(P)]

    def merge_chunks():
        for r in range(P):
            for i, off in enumerate(offs):
                qb.ulysses_merge_output_head_chunk(received[r][i], W, L, off, merged[r])

    def pack_sched():
        for r, (q, k, v) in enumerate(views):
            qb.ulysses_pack_head_chunk_schedule(q, k, v, W, wl.schedule, packed[r])

    def merge_sched():
        for r in range(P):
            qb.ulysses_merge_output_head_chunk_schedule(received[r], W, L, offs, merged[r])

    pack_bytes = sum(2 * wl.B * S * W * cnt * 3 * D * 2 for _, cnt in wl.schedule) * P
    merge_bytes = sum(2 * wl.B * S * W * cnt * D * 2 for _, cnt in wl.schedule) * P
    res = {}
    ms, med = gpu.timed_alone(pack_chunks, steps, warmup)
    for r in range(P):
        for i in range(n_chunks):
            received[r][i] = packed[r][i][..., :D].contiguous()
    res["pack_per_chunk"] = row(ms, med, pack_bytes, P * n_chunks, "ulysses_pack_head_chunk, one launch per chunk "
                                                                   "and virtual rank")
    ms, med = gpu.timed_alone(merge_chunks, steps, warmup)
    res["merge_per_chunk"] = row(ms, med, merge_bytes, P * n_chunks, "ulysses_merge_output_head_chunk, one launch "
                                                                     "per chunk and virtual rank")
    for r in range(P):
        if not torch.equal(merged[r], views[r][0]):
            raise RuntimeError("pack -> merge did not reproduce q")
        merged[r].zero_()
    ms, med = gpu.timed_alone(pack_sched, steps, warmup)
    res["pack_schedule"] = row(ms, med, pack_bytes, P, "ulysses_pack_head_chunk_schedule, one launch per virtual "
                                                       "rank for all chunks")
    ms, med = gpu.timed_alone(merge_sched, steps, warmup)
    res["merge_schedule"] = row(ms, med, merge_bytes, P, "ulysses_merge_output_head_chunk_schedule, one launch "
                                                         "per virtual rank for all chunks")
    for r in range(P):
        if not torch.equal(merged[r], views[r][0]):
            raise RuntimeError("schedule pack -> merge did not reproduce q")

    # ordinary and composed exchanges over the same P virtual ranks
    ranks = buf.view(P, S, 3, wl.num_heads, D)                 # [P*B, S, 3, H, D] with B = 1
    q5 = ranks[:, :, 0].contiguous().view(P, 1, S, wl.num_heads, D)
    y5 = torch.empty((P, 1, P * S, L, D), dtype=torch.bfloat16, device=gpu.dev)
    g5 = torch.empty_like(q5)
    pays = [torch.empty((P, 1, P * S, cnt, 3 * D), dtype=torch.bfloat16, device=gpu.dev) for _, cnt in wl.schedule]
    outs = torch.empty_like(q5)
    seq = [torch.empty((P, 1, S, cnt, D), dtype=torch.bfloat16, device=gpu.dev) for _, cnt in wl.schedule]
    qbytes = 2 * q5.numel() * 2
    ms, med = gpu.timed_alone(lambda: qb.ulysses_scatter_heads(q5, y5), steps, warmup)
    res["scatter_heads"] = row(ms, med, qbytes, 1, "ulysses_scatter_heads of q")
    ms, med = gpu.timed_alone(lambda: qb.ulysses_gather_heads(y5, g5), steps, warmup)
    res["gather_heads"] = row(ms, med, qbytes, 1, "ulysses_gather_heads of q")
    bands = [y5[:, :, :, off:off + cnt].contiguous() for off, cnt in wl.schedule]

    def sqkv():
        for i, (off, cnt) in enumerate(wl.schedule):
            qb.ulysses_scatter_qkv_head_chunk(ranks[:, :, 0], ranks[:, :, 1], ranks[:, :, 2], P, off, cnt, pays[i])

    def gout():
        for i, (off, cnt) in enumerate(wl.schedule):
            qb.ulysses_gather_output_head_chunk(bands[i], L, off, outs)

    def seqp():
        for i, (off, cnt) in enumerate(wl.schedule):
            qb.ulysses_pack_output_sequence_chunk(bands[i][0], P, seq[i])

    ms, med = gpu.timed_alone(sqkv, steps, warmup)
    res["scatter_qkv_head_chunk"] = row(ms, med, 3 * qbytes, n_chunks, "one launch per chunk, all ranks")
    ms, med = gpu.timed_alone(gout, steps, warmup)
    res["gather_output_head_chunk"] = row(ms, med, qbytes, n_chunks, "one launch per chunk, all ranks")
    ms, med = gpu.timed_alone(seqp, steps, warmup)
    res["pack_output_sequence_chunk"] = row(ms, med, qbytes // P, n_chunks, "one launch per chunk of one rank")
    if not (torch.equal(g5, q5) and torch.equal(outs, q5)):
        raise RuntimeError("scatter -> gather did not reproduce q")
    # Sage2 quantise-and-exchange of the same q/k/v (whole sequence used)
    sage = qb.sage2_outputs(P, 1, S, wl.num_heads, D, P * S)
    ms, med = gpu.timed_alone(lambda: qb.ulysses_sage2_scatter_qkv(ranks[:, :, 0], ranks[:, :, 1], ranks[:, :, 2],
                                                                   P, P * S, sage), steps, warmup)
    n_el = 3 * P * S * wl.num_heads * D
    sg = row(ms, med, n_el * 2 + n_el, 3, "ulysses_sage2_scatter_qkv (3 kernels)")
    sg["moved_bytes"] = n_el * 2 + n_el + (2 * n_el // 3) * 2   # + K and V read again by the statistics
    sg["note"] = "GB/s on algorithmic bytes (q/k/v read once, codes written); the statistics read K and V again"
    res["sage2_scatter_qkv"] = sg
    return res


def run_gpu(args):
    import torch

    from ulysses_qkv_proj_gb300 import binding as qb

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    clocks = ClockSampler(pci_bus_id(torch, dev)).start()
    gpu = Gpu(torch, dev)
    wl = WORKLOAD
    peaks, peak_src = load_peaks()

    inp, d, plan = fused_setup(gpu, qb, wl)
    x_host = torch.from_numpy(inp.x.view(np.int16)).view(torch.bfloat16).pin_memory()
    reserved = 0 if args.no_overlap else args.reserve_sms
    plan.reserve_sms(reserved)
    out = qb.alloc_outputs(plan, wl.B, wl.S, dev)
    info = plan.describe(wl.B, wl.S)

    # head-chunk inputs of the step: q/k/v views of a [P*B, S, 3, H, D] projection buffer
    PB, S, H, D, W, L = wl.P * wl.B, wl.S, wl.num_heads, 128, wl.P, wl.H_local
    qkv_np = WL.make_headchunk_buffer(PB, S, H, D)
    qkv_host = torch.from_numpy(qkv_np.view(np.int16)).view(torch.bfloat16).pin_memory()
    qkv = qkv_host.to(dev)
    packed = [torch.empty((PB, S, W * cnt, 3 * D), dtype=torch.bfloat16, device=dev) for _, cnt in SCHEDULE]
    merged = torch.empty((PB, S, H, D), dtype=torch.bfloat16, device=dev)
    side = torch.cuda.Stream(device=dev)
    primary = {"out": out, "packed": packed, "merged": merged}
    offs = [off for off, _ in SCHEDULE]

    def step(x_in, qkv_in, ev=None, bufs=None):
        """ev = [start, fused done, pack done, merge done, step done] or None."""
        bufs = bufs or primary
        o_, p_, m_ = bufs["out"], bufs["packed"], bufs["merged"]
        main = torch.cuda.current_stream()
        start = ev[0] if ev else torch.cuda.Event()
        start.record(main)
        qb.qnre_forward(plan, x_in, d["w"], d["qw"], d["kw"], d["cs"], d["pos"], o_, stream=main)
        if ev:
            ev[1].record(main)
        tail = main if args.no_overlap else side
        if tail is side:
            side.wait_event(start)
        q, k, v = qkv_in[:, :, 0], qkv_in[:, :, 1], qkv_in[:, :, 2]
        qb.ulysses_pack_head_chunk_schedule(q, k, v, W, SCHEDULE, p_, stream=tail)
        if ev:
            ev[2].record(tail)
        qb.ulysses_merge_output_head_chunk_schedule([pk[..., :D] for pk in p_], W, L, offs, m_, stream=tail)
        if ev:
            ev[3].record(tail)
        if tail is side:
            main.wait_stream(side)
        if ev:
            ev[4].record(main)

    launches_per_step = 3  # fused, pack schedule, merge schedule
    for _ in range(args.warmup):
        step(d["x"], qkv)
        gpu.flush.zero_()
    torch.cuda.synchronize()
    if plan.device_status() != 0:
        raise RuntimeError("device status raised during warm-up")
    if not torch.equal(merged, qkv[:, :, 0]):
        raise RuntimeError("pack -> merge did not reproduce q")

    # ---- device-resident timed region
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    torch.cuda.synchronize()
    with clocks.section("step"):
        for i in range(args.steps):
            step(d["x"], qkv, evs[i])
            gpu.flush.zero_()
        torch.cuda.synchronize()
    fused_ms = [e[0].elapsed_time(e[1]) for e in evs]
    step_ms = [e[0].elapsed_time(e[4]) for e in evs]
    pack_end = [e[0].elapsed_time(e[2]) for e in evs]
    merge_end = [e[0].elapsed_time(e[3]) for e in evs]
    ms_per_step = sum(step_ms) / args.steps
    value = wl.T / (ms_per_step * 1e-3)

    # ---- the same step with a warm L2 (no flush between steps), medians
    n_warm = min(args.steps, 200)
    evw = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(n_warm)]
    for _ in range(args.warmup):
        step(d["x"], qkv)
    torch.cuda.synchronize()
    with clocks.section("warm_l2"):
        for i in range(n_warm):
            step(d["x"], qkv, evw[i])
        torch.cuda.synchronize()
    warm = {"steps": n_warm,
            "ms_per_step_median": round(statistics.median(e[0].elapsed_time(e[4]) for e in evw), 5),
            "fused_ms_median": round(statistics.median(e[0].elapsed_time(e[1]) for e in evw), 5),
            "note": "no L2 flush between steps (the step's 2.1 GB of inputs exceed L2 anyway)"}

    # ---- end to end: every step copies its inputs from pinned host memory and its
    # results back.  Three device buffer sets and separate copy streams let step
    # i's device->host copy and the next steps' host->device copies overlap the
    # compute, with a step of slack either way.
    n_sets = 3
    sets = [primary] + [{"out": {g: torch.empty_like(t) for g, t in out.items()},
                         "packed": [torch.empty_like(t) for t in packed], "merged": torch.empty_like(merged)}
                        for _ in range(n_sets - 1)]
    dev_in = [(torch.empty_like(d["x"]), torch.empty_like(qkv)) for _ in range(n_sets)]
    host_out = ({g: torch.empty_like(t, device="cpu").pin_memory() for g, t in out.items()},
                torch.empty_like(merged, device="cpu").pin_memory())
    h2d = x_host.numel() * 2 + qkv_host.numel() * 2
    d2h = sum(t.numel() * 2 for t in out.values()) + merged.numel() * 2
    h2d_s, d2h_s = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    main = torch.cuda.current_stream()

    def e2e_pass(n):
        """n pipelined steps with their host copies; returns the device time (ms) of all n."""
        ev_in = [torch.cuda.Event() for _ in range(n)]
        ev_comp = [torch.cuda.Event() for _ in range(n)]
        ev_out = [torch.cuda.Event() for _ in range(n)]
        e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e_start.record(main)
        h2d_s.wait_event(e_start)
        for i in range(n):
            b = i % n_sets
            xin, qin = dev_in[b]
            if i >= n_sets:
                h2d_s.wait_event(ev_comp[i - n_sets])   # the step before has finished reading this input set
            with torch.cuda.stream(h2d_s):
                xin.copy_(x_host, non_blocking=True)
                qin.copy_(qkv_host, non_blocking=True)
            ev_in[i].record(h2d_s)
            main.wait_event(ev_in[i])
            if i >= n_sets:
                main.wait_event(ev_out[i - n_sets])     # this output set has been copied out
            step(xin, qin, bufs=sets[b])
            ev_comp[i].record(main)
            d2h_s.wait_event(ev_comp[i])
            ho, hm = host_out
            with torch.cuda.stream(d2h_s):
                for g, t in sets[b]["out"].items():
                    ho[g].copy_(t, non_blocking=True)
                hm.copy_(sets[b]["merged"], non_blocking=True)
            ev_out[i].record(d2h_s)
        main.wait_stream(d2h_s)
        e_end.record(main)
        torch.cuda.synchronize()
        return e_start.elapsed_time(e_end)

    # the first copy from or into a freshly pinned buffer pays its mapping (tens
    # of ms): warm-up passes touch every buffer before the timed one
    e2e_pass(max(n_sets, args.warmup))
    n = args.steps
    with clocks.section("e2e"):
        e2e_total = e2e_pass(n)
    e2e_ms = e2e_total / n
    if not torch.equal(host_out[1], qkv_host[:, :, 0]):
        raise RuntimeError("end-to-end result differs")
    if not torch.equal(host_out[0]["q"], out["q"].cpu()):
        raise RuntimeError("end-to-end projection differs from the device-resident one")
    e2e_value = wl.T / (e2e_ms * 1e-3)

    # the host link alone on this machine: the same copies as one step, no compute
    def copies_only():
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(main)
        h2d_s.wait_event(e0)
        d2h_s.wait_event(e0)
        xin, qin = dev_in[0]
        with torch.cuda.stream(h2d_s):
            xin.copy_(x_host, non_blocking=True)
            qin.copy_(qkv_host, non_blocking=True)
        ho, hm = host_out
        with torch.cuda.stream(d2h_s):
            for g, t in sets[1]["out"].items():
                ho[g].copy_(t, non_blocking=True)
            hm.copy_(sets[1]["merged"], non_blocking=True)
        main.wait_stream(h2d_s)
        main.wait_stream(d2h_s)
        e1.record(main)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    link_ms = min(copies_only() for _ in range(3))
    plan.destroy()
    del sets, dev_in, host_out, packed, merged, qkv, out, d
    torch.cuda.empty_cache()

    # ---- rows timed alone
    with clocks.section("alone"):
        small = time_fused_alone(gpu, qb, SMALL_FUSED, peaks, peak_src, max(args.steps, 20), args.warmup)
        hc = time_headchunk_alone(gpu, qb, HEADCHUNK, peaks, peak_src, max(args.steps, 20), args.warmup)
        fused_alone = time_fused_alone(gpu, qb, wl, peaks, peak_src, max(args.steps, 10), args.warmup, inp)
        unfused = time_unfused_alone(gpu, qb, wl, fused_alone["ms"], max(args.steps, 10), args.warmup, inp)
    clocks.stop()

    # ---- rooflines
    flops = wl.flops()
    fused_avg = statistics.mean(fused_ms)
    tflops = flops / (fused_avg * 1e-3) / 1e12
    burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    sustained = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    alg_bytes = 2 * (wl.T * wl.hidden + wl.hidden * wl.N + wl.T * wl.N) + 512 * wl.n_pos + 512
    step_pack_bytes = sum(2 * PB * S * W * cnt * 3 * D * 2 for _, cnt in SCHEDULE)
    step_merge_bytes = sum(2 * PB * S * W * cnt * D * 2 for _, cnt in SCHEDULE)
    cpu = None
    if not args.no_cpu_baseline:
        cpu_inputs(inp, qkv_np)
        cpu = cpu_baseline(args.cpu_sample_tokens)
    step_clk = clocks.summary("step")
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) activations, N(0,1/hidden) weights, 1+0.1N(0,1) norm weights)",
        "config": headline_config(),
        "execution": {"streams": "one" if args.no_overlap else "fused on the main stream, pack/merge on a second",
                      "reserved_sms": reserved, "fused_clusters": info["clusters"],
                      "pairs_per_cluster": info["pairs_per_cluster"], "parallelism": "one GPU"},
        "roofline": {"bound": "tensor", "achieved": round(tflops, 1), "peak": sustained, "unit": "TFLOP/s",
                     "frac": round(tflops / sustained, 4), "traffic": profiled_traffic(wl.name),
                     "kernel": "fused_qkv_kernel", "flops_per_launch": flops,
                     "algorithmic_bytes_per_launch": alg_bytes,
                     "peak_source": f"{peak_src} bf16_tflops_sustained (the kernel runs inside a step loop under "
                                    f"the power cap)",
                     "peak_burst": burst, "frac_burst": round(tflops / burst, 4),
                     "ms_mean": round(fused_avg, 5), "ms_median": round(statistics.median(fused_ms), 5)},
        "ms_per_step_median": round(statistics.median(step_ms), 5),
        "warm_l2": warm,
        "pack": dict(hc["pack_per_chunk"], workload=HEADCHUNK.name),
        "merge": dict(hc["merge_per_chunk"], workload=HEADCHUNK.name),
        "pack_schedule": dict(hc["pack_schedule"], workload=HEADCHUNK.name),
        "merge_schedule": dict(hc["merge_schedule"], workload=HEADCHUNK.name),
        "pack_output_sequence_chunk": dict(hc["pack_output_sequence_chunk"], workload=HEADCHUNK.name),
        "layout_rows": {k: dict(hc[k], workload=HEADCHUNK.name)
                        for k in ("scatter_heads", "gather_heads", "scatter_qkv_head_chunk",
                                  "gather_output_head_chunk")},
        "sage2": dict(hc["sage2_scatter_qkv"], workload=HEADCHUNK.name),
        "fused_h4096_p4_s4096": small,
        "fused_alone": fused_alone,
        "unfused_torch": unfused,
        "step_copies": {"pack_bytes": step_pack_bytes, "merge_bytes": step_merge_bytes,
                        "pack_end_ms": round(statistics.mean(pack_end), 5),
                        "merge_end_ms": round(statistics.mean(merge_end), 5),
                        "note": "end times from the step's start; the copies run beside the fused kernel on the "
                                "SMs it leaves, so these are not HBM fractions of the copy kernel"
                                if not args.no_overlap else "end times from the step's start, one stream"},
        "e2e": {"value": round(e2e_value, 1), "unit": "tokens/s", "ms_per_step": round(e2e_ms, 4),
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "link_ms_per_step": round(link_ms, 4), "frac_of_link": round(link_ms / e2e_ms, 4),
                "note": "pipelined: step i's D2H and step i+1's H2D overlap compute; link_ms_per_step is the "
                        "same copies alone (both directions at once, no compute), the floor on this box"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": step_clk,
        "clocks_sections": {k: clocks.summary(k) for k in ("warm_l2", "e2e", "alone")},
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------
# CPU oracle (baseline leg and the reference arm)
# ----------------------------------------------------------------------------
_CPU_CACHE = {}


def stratified_tokens(wl, n: int, seed: int = 123) -> np.ndarray:
    """n token ids of wl: the first and last token of every (rank, batch) segment
    and of every 256-row tile, the rest drawn at random."""
    rng = np.random.default_rng(seed)
    picks = set()
    for t0 in range(0, wl.T, wl.S):
        picks.update({t0, t0 + wl.S - 1})
    for t0 in range(0, wl.T, 256):
        picks.update({t0, min(wl.T - 1, t0 + 255)})
    picks = sorted(picks)
    if len(picks) >= n:
        idx = np.linspace(0, len(picks) - 1, n).round().astype(int)
        return np.array(sorted({picks[i] for i in idx}))
    rest = np.setdiff1d(np.arange(wl.T), picks)
    extra = rng.choice(rest, size=min(n - len(picks), len(rest)), replace=False)
    return np.sort(np.concatenate([np.array(picks), extra]))


def cpu_inputs(inp=None, qkv=None):
    """The headline workload's host inputs (drawn once; the GPU arm passes its own)."""
    wl = WORKLOAD
    if inp is not None:
        _CPU_CACHE["inp"] = inp
    if qkv is not None:
        _CPU_CACHE["qkv"] = qkv
    if "inp" not in _CPU_CACHE:
        _CPU_CACHE["inp"] = WL.make_fused_inputs(wl)
    if "qkv" not in _CPU_CACHE:
        _CPU_CACHE["qkv"] = WL.make_headchunk_buffer(wl.P * wl.B, wl.S, wl.num_heads, 128)
    return _CPU_CACHE["inp"], _CPU_CACHE["qkv"]


def cpu_sample_step(n_tokens: int):
    """One step of the workload on the CPU oracle over n_tokens of its tokens; returns
    (tokens, seconds).  The token subset is stratified (stratified_tokens) and goes
    through projection, RMSNorm, RoPE and band placement; pack/merge of the same
    share of the step's rows follows."""
    import oracle
    wl = WORKLOAD
    inp, qkv = cpu_inputs()
    tok = stratified_tokens(wl, min(n_tokens, wl.T))
    rows = max(1, round(wl.S * len(tok) / wl.T))
    sub = qkv[:, :rows]
    t0 = time.perf_counter()
    x2 = inp.x.reshape(wl.T, wl.hidden)
    O = oracle.project_norm_rope(x2[tok], inp.w, inp.q_norm_w, inp.k_norm_w, inp.cos_sin,
                                 inp.positions.reshape(-1)[tok], wl.num_heads, wl.rope_style)
    dest = [oracle.band_destination(*oracle.token_coords(int(t), wl.P, wl.B, wl.S), h, wl.P, wl.B, wl.S,
                                    wl.num_heads) for t in tok for h in range(wl.num_heads)]
    assert O.shape[0] == len(tok) and len(dest) == len(tok) * wl.num_heads
    merged = np.zeros((wl.P * wl.B, rows, wl.num_heads, 128), np.uint16)
    for off, cnt in SCHEDULE:
        pk = oracle.pack_head_chunk(sub[:, :, 0], sub[:, :, 1], sub[:, :, 2], wl.P, off, cnt)
        merged = oracle.merge_output_head_chunk(pk[..., :128], wl.P, wl.H_local, off, merged)
    dt = time.perf_counter() - t0
    return len(tok), dt


def cpu_cores() -> int:
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var):
            return int(os.environ[var])
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(n_tokens: int):
    cpu_sample_step(16)  # warm the caches and BLAS
    tok, dt = cpu_sample_step(n_tokens)
    return {"value": round(tok / dt, 2), "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
            "sample": f"{tok} of {WORKLOAD.T} tokens of {WORKLOAD.name} (first and last token of every segment and "
                      f"256-row tile, the rest random) through the fp64 oracle (projection, RMSNorm, RoPE, band "
                      f"placement) plus pack+merge of the same share of the step's rows; tokens/s extrapolated "
                      f"from the sample to the workload; numpy BLAS threads = cores",
            "extrapolated": True, "seconds": round(dt, 3)}


def headline_config():
    """The headline workload, as both arms report it."""
    wl = WORKLOAD
    sched = [list(b) for b in SCHEDULE]
    return {"workload": f"{wl.name}: P={wl.P} B={wl.B} S_local={wl.S} S_global={wl.S_global} "
                        f"hidden={wl.hidden} heads={wl.num_heads} layout={wl.layout} rope={wl.rope_style}; "
                        f"pack/merge schedule {sched} over H_local={wl.H_local}",
            "tokens_per_step": wl.T, "P": wl.P, "B": wl.B, "S_local": wl.S, "hidden": wl.hidden,
            "num_heads": wl.num_heads, "layout": wl.layout, "schedule": sched,
            "l2": "inputs (2.1 GB) larger than L2, and L2 flushed (512 MB write) between steps"}


def run_reference(args):
    if int(os.environ.get("RANK", "0")) != 0:
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    cpu_inputs()
    # size each step so that warm-up + timed steps take about ref_budget_s of CPU time
    n_cal, dt_cal = cpu_sample_step(32)
    per_token = dt_cal / n_cal
    budget = args.ref_budget_s / max(1, args.steps + args.warmup)
    n = int(max(8, min(WORKLOAD.T, budget / per_token)))
    for _ in range(args.warmup):
        cpu_sample_step(n)
    times = []
    for _ in range(args.steps):
        tok, dt = cpu_sample_step(n)
        times.append(dt)
    ms_per_step = 1e3 * sum(times) / len(times)
    value = tok / (ms_per_step * 1e-3)
    wl = WORKLOAD
    sample = (f"{tok} of {wl.T} tokens of {wl.name} per step (stratified) through the fp64 oracle, plus "
              f"pack+merge of the same share of the step's rows; tokens/s extrapolated to the workload")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": headline_config(),
        "execution": {"parallelism": "host cores", "tokens_per_step_sample": tok},
        "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def run_gpu_workload(args):
    """One row alone on a named workload (not the headline step): the fused op on a
    fused workload (with the readiness-word forms), or every copy row and Sage2 on a
    head-chunk workload."""
    import torch

    from ulysses_qkv_proj_gb300 import binding as qb

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    gpu = Gpu(torch, dev)
    clocks = ClockSampler(pci_bus_id(torch, dev)).start()
    peaks, peak_src = load_peaks()
    name = args.workload
    if name in WL.FUSED_WORKLOADS:
        wl = WL.FUSED_WORKLOADS[name]
        with clocks.section("alone"):
            res = time_fused_alone(gpu, qb, wl, peaks, peak_src, args.steps, args.warmup)
        line = {"metric": "fused QKV+norm+RoPE+scatter tokens/s", "value": res["tokens_per_s"], "unit": "tokens/s",
                "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["ms"],
                "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
                "config": {"workload": name, "tokens": wl.T, "hidden": wl.hidden, "layout": wl.layout,
                           "l2": "flushed between launches"},
                "roofline": {"bound": "tensor", "achieved": res["tflops"], "peak": res["peak"], "unit": "TFLOP/s",
                             "frac": res["frac"], "traffic": profiled_traffic(name),
                             "peak_source": res["peak_source"]},
                "fused": res, "gpu_launches": args.steps}
        if args.readiness:
            _, d, plan = fused_setup(gpu, qb, wl)
            out = qb.alloc_outputs(plan, wl.B, wl.S, dev)
            ready = torch.zeros((wl.P,), dtype=torch.int32, device=dev)
            target = qb.qnre_ready_target(plan, wl.B, wl.S)
            consumer = torch.cuda.Stream(device=dev)
            fwd = (plan, d["x"], d["w"], d["qw"], d["kw"], d["cs"], d["pos"], out)

            def publish_and_wait():
                main = torch.cuda.current_stream()
                qb.qnre_forward_publish(*fwd, ready, stream=main)
                consumer.wait_stream(main)
                qb.qnre_wait_ready(plan, ready, target, 1_000_000_000, stream=consumer)
                main.wait_stream(consumer)
            ms_pub, _ = gpu.timed_alone(lambda: qb.qnre_forward_publish(*fwd, ready), args.steps, args.warmup)
            ms_pw, _ = gpu.timed_alone(publish_and_wait, args.steps, args.warmup)
            if plan.device_status() != 0 or ready.cpu().tolist() != [target] * wl.P:
                raise RuntimeError("readiness words did not reach their target")
            line["readiness"] = {"forward_publish_ms": round(ms_pub, 5), "publish_and_wait_ms": round(ms_pw, 5),
                                 "publish_overhead_pct": round(100 * (ms_pub / res["ms"] - 1), 2)}
            plan.destroy()
    elif name in WL.HEADCHUNK_WORKLOADS:
        wl = WL.HEADCHUNK_WORKLOADS[name]
        with clocks.section("alone"):
            res = time_headchunk_alone(gpu, qb, wl, peaks, peak_src, args.steps, args.warmup)
        p = res["pack_per_chunk"]
        line = {"metric": "head-chunk pack/merge GB/s", "value": p["GB/s"], "unit": "GB/s", "n_gpus": 1,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": p["ms"], "higher_is_better": True,
                "dtype": "bf16", "data": "synthetic",
                "config": {"workload": name, "schedule": [list(b) for b in wl.schedule], "P": wl.P,
                           "l2": "flushed between repetitions"},
                "roofline": {"bound": "hbm", "achieved": p["GB/s"], "peak": p["peak"], "unit": "GB/s",
                             "frac": p["frac_hbm"], "peak_source": p["peak_source"]}}
        line.update(res)
    else:
        raise SystemExit(f"unknown workload {name!r}")
    clocks.stop()
    line["clocks"] = clocks.summary("alone")
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1, help="must be 1: this benchmark runs on one GPU")
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-sample-tokens", type=int, default=8192,
                    help="tokens of the headline workload the CPU-oracle baseline runs")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the CPU-oracle baseline leg")
    ap.add_argument("--ref-budget-s", type=float, default=90.0,
                    help="CPU seconds the reference arm spreads over warm-up + timed steps")
    ap.add_argument("--no-overlap", action="store_true",
                    help="run pack/merge after the fused op on one stream instead of beside it")
    ap.add_argument("--reserve-sms", type=int, default=0,
                    help="SMs the fused kernel leaves to the concurrent pack/merge (overlapped step only)")
    ap.add_argument("--workload", default=None,
                    help="time one row alone on this workload instead of the headline step")
    ap.add_argument("--readiness", action="store_true",
                    help="with a fused --workload: also time the readiness-word forward and its wait")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
        return
    refuse_multi_gpu(args)
    if args.workload:
        run_gpu_workload(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
