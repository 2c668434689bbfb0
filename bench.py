"""Benchmark of the Ulysses QKV front end on one GB300 (or N independent replicas).

One step = one pass of the whole hot path over one batch of the workload
"h4096_p4_s4096" (P=4 virtual ranks x B=1 x S_local=1024 tokens, hidden 4096,
32 heads, bshd):
  1. qnre_forward: fused QKV projection + RMSNorm + RoPE + band scatter of all
     4096 tokens into the 4 ranks' [B, S_global, 8, 128] bands;
  2. the head-chunk pack of every band of the uneven schedule
     [(0,2),(2,4),(6,2)] over H_local = 8, on strided q/k/v views of a
     [P*B, S_local, 3, 32, 128] projection buffer (all virtual ranks, all bands
     in one ulysses_pack_head_chunk_schedule launch);
  3. the merge of each packed band's q slice back into a [P*B, S_local, 32, 128]
     output (one ulysses_merge_output_head_chunk_schedule launch; pack then
     merge reproduces q).
Steps 2-3 do not depend on step 1, so they run on a second stream beside it
(the memory-bound copies fill what the tensor-bound projection leaves idle).
A copy CTA does not share an SM with a CTA of the persistent fused kernel
(%smid stamps: none of a step's 4096 copy blocks started beside one); the
copies run on the SMs its four-CTA clusters leave (12 here: the plan launches
35 clusters, as many rounds as 36) and on SMs as the fused kernel's clusters
retire.  --reserve-sms N (default 0) leaves N more SMs
to them: qnre_plan_reserve_sms.  --no-overlap runs everything on one stream with every
SM given to the fused kernel.
The L2 (129 MB) is flushed with a 512 MB write between timed steps.

value = tokens per second of the whole step (all ranks' tokens / step time).

`--impl reference` times the CPU oracle on the host cores instead: every step
is a bounded sample of the same workload (a stratified token subset through the
fp64 projection/norm/RoPE/placement and the same rows through pack/merge).
"""
from __future__ import annotations

import argparse
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
SCHEDULE = WL.BENCH_SCHEDULE
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


FUSED_SOURCES = ["ulysses_qkv_proj_gb300/csrc/fused_qkv.cu", "ulysses_qkv_proj_gb300/csrc/fused_qkv.cuh",
                 "ulysses_qkv_proj_gb300/csrc/ptx.cuh"]
FUSED_PROFILE = "profiles/fused_qkv_kernel_h4096_p4_s4096.md"


def fused_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in FUSED_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the current kernel source."""
    path = os.path.join(ROOT, FUSED_PROFILE)
    if not os.path.exists(path):
        return None
    fields = {}
    for line in open(path):
        if ":" in line and not line.startswith(("|", "#", " ")):
            k, v = line.split(":", 1)
            fields[k.strip()] = v.strip()
    if fields.get("kernel-source-hash") != fused_source_hash():
        return None
    try:
        return int(fields["traffic-bytes-per-launch"])
    except (KeyError, ValueError):
        return None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def max_over_ranks(x: float) -> float:
    """Largest x over the process group (the slowest rank's time); x itself with one rank."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


# ----------------------------------------------------------------------------
# clocks sampling during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self._t.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None, "samples": len(sm), "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------
def run_gpu(args):
    import torch
    import torch.distributed as dist

    from ulysses_qkv_proj_gb300 import binding as qb

    rank, world, local_rank = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl = WORKLOAD
    peaks, peak_src = load_peaks()

    def t16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    inp = WL.make_fused_inputs(wl)
    x_host = torch.from_numpy(inp.x.view(np.int16)).view(torch.bfloat16).pin_memory()
    x = x_host.to(dev)
    w = t16(inp.w)
    qw, kw = t16(inp.q_norm_w), t16(inp.k_norm_w)
    cs = torch.from_numpy(inp.cos_sin).to(dev)
    pos = torch.from_numpy(inp.positions).to(dev)
    plan = qb.Plan(wl.hidden, wl.num_heads, wl.P, wl.layout, max_tokens=wl.B * wl.S, rope_style=wl.rope_style)
    reserved = 0 if args.no_overlap else args.reserve_sms
    plan.reserve_sms(reserved)
    out = qb.alloc_outputs(plan, wl.B, wl.S, dev)

    # head-chunk inputs: q/k/v views of a [P*B, S, 3, H, D] projection buffer
    PB, S, H, D, W, L = wl.P * wl.B, wl.S, wl.num_heads, 128, wl.P, wl.H_local
    qkv_host_np = WL.make_headchunk_buffer(PB, S, H, D)
    qkv_host = torch.from_numpy(qkv_host_np.view(np.int16)).view(torch.bfloat16).pin_memory()
    qkv = qkv_host.to(dev)
    packed = [torch.empty((PB, S, W * cnt, 3 * D), dtype=torch.bfloat16, device=dev) for _, cnt in SCHEDULE]
    merged = torch.empty((PB, S, H, D), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    side = torch.cuda.Stream(device=dev)

    primary = {"out": out, "packed": packed, "merged": merged}

    def step(x_in, qkv_in, ev=None, bufs=None):
        """ev = [start, fused done, pack done, merge done, step done] or None.

        The fused op runs on the current stream; pack and merge (independent of it)
        run on a second stream so they fill the SMs' spare issue slots and DRAM
        bandwidth while the tensor cores work (--no-overlap serialises them)."""
        bufs = bufs or primary
        o_, p_, m_ = bufs["out"], bufs["packed"], bufs["merged"]
        main = torch.cuda.current_stream()
        start = ev[0] if ev else torch.cuda.Event()
        start.record(main)
        qb.qnre_forward(plan, x_in, w, qw, kw, cs, pos, o_, stream=main)
        if ev:
            ev[1].record(main)
        tail = main if args.no_overlap else side
        if tail is side:
            side.wait_event(start)
        q, k, v = qkv_in[:, :, 0], qkv_in[:, :, 1], qkv_in[:, :, 2]
        qb.ulysses_pack_head_chunk_schedule(q, k, v, W, SCHEDULE, p_, stream=tail)
        if ev:
            ev[2].record(tail)
        qb.ulysses_merge_output_head_chunk_schedule([pk[..., :D] for pk in p_], W, L, [off for off, _ in SCHEDULE],
                                                    m_, stream=tail)
        if ev:
            ev[3].record(tail)
        if tail is side:
            main.wait_stream(side)
        if ev:
            ev[4].record(main)

    launches_per_step = 3  # fused, pack schedule, merge schedule
    for _ in range(args.warmup):
        step(x, qkv)
        flush.zero_()
    torch.cuda.synchronize()
    if plan.device_status() != 0:
        raise RuntimeError("device status raised during warm-up")
    if not torch.equal(merged, qkv[:, :, 0]):
        raise RuntimeError("pack -> merge did not reproduce q")

    # ---- device-resident timed region
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    clocks = ClockSampler(local_rank)
    clocks.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    for i in range(args.steps):
        step(x, qkv, evs[i])
        flush.zero_()
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    clk = clocks.stop()
    fused_ms = [e[0].elapsed_time(e[1]) for e in evs]
    pack_ms = [(e[1] if args.no_overlap else e[0]).elapsed_time(e[2]) for e in evs]
    merge_ms = [e[2].elapsed_time(e[3]) for e in evs]
    step_ms = [e[0].elapsed_time(e[4]) for e in evs]
    total_ms = max_over_ranks(sum(step_ms))
    ms_per_step = total_ms / args.steps
    tokens_per_step = wl.T
    value = tokens_per_step * world / (ms_per_step * 1e-3)

    # ---- the same step with a warm L2 (no flush between steps), reported beside
    # the flushed number as the pages report both; medians over the steps
    n_warm = min(args.steps, 200)
    evw = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(n_warm)]
    for _ in range(args.warmup):
        step(x, qkv)
    torch.cuda.synchronize()
    for i in range(n_warm):
        step(x, qkv, evw[i])
    torch.cuda.synchronize()
    warm = {"steps": n_warm,
            "ms_per_step_median": round(statistics.median(e[0].elapsed_time(e[4]) for e in evw), 5),
            "fused_ms_median": round(statistics.median(e[0].elapsed_time(e[1]) for e in evw), 5),
            "note": "no L2 flush between steps; value and roofline use the flushed run"}

    # ---- end to end: every step copies its inputs from pinned host memory and its
    # results back.  Two buffer sets and separate copy streams let step i's
    # device->host copy and step i+1's host->device copy overlap the compute.
    sets = [primary, {"out": {g: torch.empty_like(t) for g, t in out.items()},
                      "packed": [torch.empty_like(t) for t in packed], "merged": torch.empty_like(merged)}]
    dev_in = [(torch.empty_like(x), torch.empty_like(qkv)) for _ in range(2)]
    host_out = [({g: torch.empty_like(t, device="cpu").pin_memory() for g, t in out.items()},
                 torch.empty_like(merged, device="cpu").pin_memory()) for _ in range(2)]
    h2d = x_host.numel() * 2 + qkv_host.numel() * 2
    d2h = sum(t.numel() * 2 for t in out.values()) + merged.numel() * 2
    h2d_s, d2h_s = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    n = args.steps
    ev_in = [torch.cuda.Event() for _ in range(n)]
    ev_comp = [torch.cuda.Event() for _ in range(n)]
    ev_out = [torch.cuda.Event() for _ in range(n)]
    e2e_start, e2e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    main = torch.cuda.current_stream()
    torch.cuda.synchronize()
    e2e_start.record(main)
    h2d_s.wait_event(e2e_start)
    for i in range(n):
        b = i % 2
        xin, qin = dev_in[b]
        if i >= 2:
            h2d_s.wait_event(ev_comp[i - 2])   # step i-2 has finished reading this input set
        with torch.cuda.stream(h2d_s):
            xin.copy_(x_host, non_blocking=True)
            qin.copy_(qkv_host, non_blocking=True)
        ev_in[i].record(h2d_s)
        main.wait_event(ev_in[i])
        if i >= 2:
            main.wait_event(ev_out[i - 2])     # this output set has been copied out
        step(xin, qin, bufs=sets[b])
        ev_comp[i].record(main)
        d2h_s.wait_event(ev_comp[i])
        ho, hm = host_out[b]
        with torch.cuda.stream(d2h_s):
            for g, t in sets[b]["out"].items():
                ho[g].copy_(t, non_blocking=True)
            hm.copy_(sets[b]["merged"], non_blocking=True)
        ev_out[i].record(d2h_s)
    main.wait_stream(d2h_s)
    e2e_end.record(main)
    torch.cuda.synchronize()
    e2e_ms = e2e_start.elapsed_time(e2e_end) / n
    if not torch.equal(host_out[(n - 1) % 2][1], qkv_host[:, :, 0]):
        raise RuntimeError("end-to-end result differs")
    e2e_ms = max_over_ranks(e2e_ms)
    e2e_value = tokens_per_step * world / (e2e_ms * 1e-3)

    # ---- rooflines
    flops = wl.flops()
    fused_avg = statistics.mean(fused_ms)
    tflops = flops / (fused_avg * 1e-3) / 1e12
    tc_peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    elt = 2
    pack_bytes = sum(2 * PB * S * W * cnt * 3 * D * elt for _, cnt in SCHEDULE)
    merge_bytes = sum(2 * PB * S * W * cnt * D * elt for _, cnt in SCHEDULE)
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    pack_gbs = pack_bytes / (statistics.mean(pack_ms) * 1e-3) / 1e9
    merge_gbs = merge_bytes / (statistics.mean(merge_ms) * 1e-3) / 1e9

    if rank == 0:
        cpu = cpu_baseline(args.cpu_sample_tokens) if world == 1 else None
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) activations, N(0,1/hidden) weights)",
            "config": {"workload": f"{wl.name}: P={wl.P} B={wl.B} S_local={wl.S} hidden={wl.hidden} "
                                   f"heads={wl.num_heads} layout={wl.layout} rope={wl.rope_style}; "
                                   f"pack/merge schedule {list(SCHEDULE)} over H_local={L}",
                       "tokens_per_step": tokens_per_step, "P": wl.P, "B": wl.B, "S_local": wl.S,
                       "hidden": wl.hidden, "num_heads": wl.num_heads, "layout": wl.layout,
                       "schedule": [list(b) for b in SCHEDULE], "l2": "flushed (512 MB write) between steps",
                       "streams": "one" if args.no_overlap else "fused on the main stream, pack/merge on a second",
                       "reserved_sms": reserved,
                       "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "tensor", "achieved": round(tflops, 1), "peak": tc_peak, "unit": "TFLOP/s",
                         "frac": round(tflops / tc_peak, 4), "traffic": profiled_traffic(),
                         "kernel": "fused_qkv_kernel", "peak_source": f"{peak_src} bf16_tflops (burst)",
                         "flops_per_launch": flops},
            "fused": {"ms": round(fused_avg, 5), "ms_median": round(statistics.median(fused_ms), 5),
                      "tflops": round(tflops, 1), "tokens_per_s": round(wl.T / (fused_avg * 1e-3), 1)},
            "ms_per_step_median": round(statistics.median(step_ms), 5),
            "warm_l2": warm,
            "pack": {"ms": round(statistics.mean(pack_ms), 5), "bytes": pack_bytes, "GB/s": round(pack_gbs, 1),
                     "frac_hbm": round(pack_gbs / hbm_peak, 4), "launches": 1, "chunks": len(SCHEDULE)},
            "merge": {"ms": round(statistics.mean(merge_ms), 5), "bytes": merge_bytes, "GB/s": round(merge_gbs, 1),
                      "frac_hbm": round(merge_gbs / hbm_peak, 4), "launches": 1, "chunks": len(SCHEDULE)},
            "e2e": {"value": round(e2e_value, 1), "unit": "tokens/s", "ms_per_step": round(e2e_ms, 4),
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "note": "pipelined: step i's D2H and step i+1's H2D overlap compute; 268 MB of "
                            "per-step copies exceed L2"},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk,
            "wall_s_timed": round(t_wall, 4),
        }
        if cpu is not None:
            line["cpu_baseline"] = cpu
        print(json.dumps(line), flush=True)
    plan.destroy()
    if world > 1:
        dist.destroy_process_group()


# ----------------------------------------------------------------------------
# CPU oracle (baseline leg and the reference arm)
# ----------------------------------------------------------------------------
_CPU_CACHE = {}


def _cpu_inputs():
    if "inp" not in _CPU_CACHE:
        wl = WORKLOAD
        _CPU_CACHE["inp"] = WL.make_fused_inputs(wl)
        _CPU_CACHE["qkv"] = WL.make_headchunk_buffer(wl.P * wl.B, wl.S, wl.num_heads, 128)
    return _CPU_CACHE["inp"], _CPU_CACHE["qkv"]


def cpu_sample_step(n_tokens: int):
    """One step of the workload on the CPU oracle, on n_tokens of its tokens; returns (tokens, seconds).

    n_tokens >= T runs the whole workload (oracle.qnre_forward + pack/merge of every row);
    fewer tokens take a stratified random subset (projection/norm/RoPE of those tokens,
    their band destinations, and pack/merge of the same number of rows).
    """
    import oracle
    wl = WORKLOAD
    inp, qkv = _cpu_inputs()
    t0 = time.perf_counter()
    if n_tokens >= wl.T:
        n_tokens = wl.T
        res = oracle.qnre_forward(inp.x, inp.w, inp.q_norm_w, inp.k_norm_w, inp.cos_sin, inp.positions,
                                  wl.P, wl.num_heads, wl.layout, wl.rope_style)
        assert all(not np.isnan(a).any() for a in res.values())
        rows = wl.S
    else:
        rng = np.random.default_rng(123)
        tok = np.sort(rng.choice(wl.T, size=n_tokens, replace=False))
        x2 = inp.x.reshape(wl.T, wl.hidden)
        O = oracle.project_norm_rope(x2[tok], inp.w, inp.q_norm_w, inp.k_norm_w, inp.cos_sin,
                                     inp.positions.reshape(-1)[tok], wl.num_heads, wl.rope_style)
        dest = [oracle.band_destination(*oracle.token_coords(int(t), wl.P, wl.B, wl.S), h, wl.P, wl.B, wl.S,
                                        wl.num_heads) for t in tok for h in range(wl.num_heads)]
        assert O.shape[0] == n_tokens and len(dest) == n_tokens * wl.num_heads
        rows = max(1, n_tokens // (wl.P * wl.B))
    sub = qkv[:, :rows]
    merged = np.zeros((wl.P * wl.B, rows, wl.num_heads, 128), np.uint16)
    for off, cnt in SCHEDULE:
        pk = oracle.pack_head_chunk(sub[:, :, 0], sub[:, :, 1], sub[:, :, 2], wl.P, off, cnt)
        merged = oracle.merge_output_head_chunk(pk[..., :128], wl.P, wl.H_local, off, merged)
    dt = time.perf_counter() - t0
    return n_tokens, dt


def cpu_cores() -> int:
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var):
            return int(os.environ[var])
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(n_tokens: int):
    cpu_sample_step(32)  # warm the input cache and BLAS
    tok, dt = cpu_sample_step(n_tokens)
    what = ("the whole workload" if tok >= WORKLOAD.T else f"{tok} of {WORKLOAD.T} tokens (stratified random)")
    return {"value": round(tok / dt, 2), "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
            "sample": f"{what} of {WORKLOAD.name} through the fp64 oracle (projection, RMSNorm, RoPE, band "
                      f"placement) plus pack+merge of the matching rows over the same schedule; numpy BLAS "
                      f"threads = cores",
            "seconds": round(dt, 3)}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    _cpu_inputs()
    # size each step so that warm-up + timed steps take about 90 s of CPU time
    n_cal, dt_cal = cpu_sample_step(64)
    per_token = dt_cal / n_cal
    budget = args.ref_budget_s / max(1, args.steps + args.warmup)
    n = int(max(1, min(WORKLOAD.T, budget / per_token)))
    for _ in range(args.warmup):
        cpu_sample_step(n)
    times = []
    for _ in range(args.steps):
        tok, dt = cpu_sample_step(n)
        times.append(dt)
    ms_per_step = 1e3 * sum(times) / len(times)
    value = tok / (ms_per_step * 1e-3)
    wl = WORKLOAD
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": wl.name, "tokens_per_step_sample": tok,
                                        "parallelism": "host cores"},
        "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": f"{tok} of {wl.T} tokens per step (stratified random) through the fp64 "
                                   f"oracle, plus pack+merge of the matching rows"},
        "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def run_gpu_workload(args):
    """One row of the hot path alone on a named workload (not the headline step):
    the fused op on a FUSED_WORKLOADS shape, or pack + merge over a HEADCHUNK_WORKLOADS shape."""
    import torch

    from ulysses_qkv_proj_gb300 import binding as qb

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    peaks, peak_src = load_peaks()
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.int32, device=dev)

    def t16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    def timed(fn):
        for _ in range(args.warmup):
            fn()
            flush.zero_()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        clocks = ClockSampler(0)
        clocks.start()
        for a, b in evs:
            a.record()
            fn()
            b.record()
            flush.zero_()
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in evs), clocks.stop()

    name = args.workload
    if name in WL.FUSED_WORKLOADS:
        wl = WL.FUSED_WORKLOADS[name]
        inp = WL.make_fused_inputs(wl)
        x, w = t16(inp.x), t16(inp.w)
        qw, kw = t16(inp.q_norm_w), t16(inp.k_norm_w)
        cs = torch.from_numpy(inp.cos_sin).to(dev)
        pos = torch.from_numpy(inp.positions).to(dev)
        plan = qb.Plan(wl.hidden, wl.num_heads, wl.P, wl.layout, max_tokens=wl.B * wl.S, rope_style=wl.rope_style)
        out = qb.alloc_outputs(plan, wl.B, wl.S, dev)
        ms, clk = timed(lambda: qb.qnre_forward(plan, x, w, qw, kw, cs, pos, out))
        if plan.device_status() != 0:
            raise RuntimeError("device status raised")
        # readiness words: the publishing forward, then the bounded wait on a consumer
        # stream ordered after it, joined back into the main stream
        ready = torch.zeros((wl.P,), dtype=torch.int32, device=dev)
        target = qb.qnre_ready_target(plan, wl.B, wl.S)
        consumer = torch.cuda.Stream(device=dev)

        def publish_and_wait():
            main = torch.cuda.current_stream()
            qb.qnre_forward_publish(plan, x, w, qw, kw, cs, pos, out, ready, stream=main)
            consumer.wait_stream(main)
            qb.qnre_wait_ready(plan, ready, target, 1_000_000_000, stream=consumer)
            main.wait_stream(consumer)
        ms_pub, _ = timed(lambda: qb.qnre_forward_publish(plan, x, w, qw, kw, cs, pos, out, ready))
        ms_pw, _ = timed(publish_and_wait)
        if plan.device_status() != 0 or ready.cpu().tolist() != [target] * wl.P:
            raise RuntimeError("readiness words did not reach their target")
        tflops = wl.flops() / (ms * 1e-3) / 1e12
        peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
        line = {"metric": "fused QKV+norm+RoPE+scatter tokens/s", "value": round(wl.T / (ms * 1e-3), 1),
                "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(ms, 5), "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
                "config": {"workload": name, "tokens": wl.T, "hidden": wl.hidden, "layout": wl.layout,
                           "l2": "flushed between launches"},
                "roofline": {"bound": "tensor", "achieved": round(tflops, 1), "peak": peak, "unit": "TFLOP/s",
                             "frac": round(tflops / peak, 4), "peak_source": f"{peak_src} bf16_tflops (burst)"},
                "readiness": {"forward_publish_ms": round(ms_pub, 5), "publish_and_wait_ms": round(ms_pw, 5),
                              "publish_overhead_pct": round(100 * (ms_pub / ms - 1), 2),
                              "note": "the wait kernel runs after the producer on a consumer stream"},
                "gpu_launches": args.steps, "clocks": clk}
        plan.destroy()
    elif name in WL.HEADCHUNK_WORKLOADS:
        wl = WL.HEADCHUNK_WORKLOADS[name]
        buf = t16(WL.make_headchunk_buffer(wl.B, wl.S_global, wl.num_heads, wl.D))
        W, L, D, S = wl.P, wl.H_local, wl.D, wl.S
        views = [(buf[:, r * S:(r + 1) * S, 0], buf[:, r * S:(r + 1) * S, 1], buf[:, r * S:(r + 1) * S, 2])
                 for r in range(wl.P)]
        packed = [[torch.empty((wl.B, S, W * cnt, 3 * D), dtype=torch.bfloat16, device=dev) for _, cnt in wl.schedule]
                  for _ in range(wl.P)]
        merged = [torch.empty((wl.B, S, wl.num_heads, D), dtype=torch.bfloat16, device=dev) for _ in range(wl.P)]

        def pack_all():
            for r, (q, k, v) in enumerate(views):
                for i, (off, cnt) in enumerate(wl.schedule):
                    qb.ulysses_pack_head_chunk(q, k, v, W, off, cnt, packed[r][i])

        def merge_all():
            for r in range(wl.P):
                for i, (off, cnt) in enumerate(wl.schedule):
                    qb.ulysses_merge_output_head_chunk(packed[r][i][..., :D], W, L, off, merged[r])

        ms_p, clk = timed(pack_all)
        ms_m, _ = timed(merge_all)
        for r in range(wl.P):
            if not torch.equal(merged[r], views[r][0]):
                raise RuntimeError("pack -> merge did not reproduce q")

        # the same schedule through the schedule calls: one launch per rank each
        def pack_sched():
            for r, (q, k, v) in enumerate(views):
                qb.ulysses_pack_head_chunk_schedule(q, k, v, W, wl.schedule, packed[r])

        def merge_sched():
            for r in range(wl.P):
                qb.ulysses_merge_output_head_chunk_schedule([pk[..., :D] for pk in packed[r]], W, L,
                                                            [off for off, _ in wl.schedule], merged[r])
        for r in range(wl.P):
            merged[r].zero_()
        ms_ps, _ = timed(pack_sched)
        ms_ms, _ = timed(merge_sched)
        for r in range(wl.P):
            if not torch.equal(merged[r], views[r][0]):
                raise RuntimeError("schedule pack -> merge did not reproduce q")

        # ordinary and composed exchanges over the same P virtual ranks
        P = wl.P
        ranks = buf.view(P, S, 3, wl.num_heads, D)                 # [P*B, S, 3, H, D] with B = 1
        q5 = ranks[:, :, 0].contiguous().view(P, 1, S, wl.num_heads, D)
        y5 = torch.empty((P, 1, P * S, L, D), dtype=torch.bfloat16, device=dev)
        g5 = torch.empty_like(q5)
        pays = [torch.empty((P, 1, P * S, cnt, 3 * D), dtype=torch.bfloat16, device=dev) for _, cnt in wl.schedule]
        outs = torch.empty_like(q5)
        seq = [torch.empty((P, 1, S, cnt, D), dtype=torch.bfloat16, device=dev) for _, cnt in wl.schedule]
        ms_sc, _ = timed(lambda: qb.ulysses_scatter_heads(q5, y5))
        ms_ga, _ = timed(lambda: qb.ulysses_gather_heads(y5, g5))
        bands = [y5[:, :, :, off:off + cnt].contiguous() for off, cnt in wl.schedule]  # after y5 is filled

        def sqkv():
            for i, (off, cnt) in enumerate(wl.schedule):
                qb.ulysses_scatter_qkv_head_chunk(ranks[:, :, 0], ranks[:, :, 1], ranks[:, :, 2], P, off, cnt, pays[i])

        def gout():
            for i, (off, cnt) in enumerate(wl.schedule):
                qb.ulysses_gather_output_head_chunk(bands[i], L, off, outs)

        def seqp():
            for i, (off, cnt) in enumerate(wl.schedule):
                qb.ulysses_pack_output_sequence_chunk(bands[i][0], P, seq[i])

        ms_sq, _ = timed(sqkv)
        ms_go, _ = timed(gout)
        ms_sp, _ = timed(seqp)
        if not (torch.equal(g5, q5) and torch.equal(outs, q5)):
            raise RuntimeError("scatter -> gather did not reproduce q")
        qbytes = 2 * q5.numel() * 2

        def row(ms, nbytes, launches):
            g = nbytes / (ms * 1e-3) / 1e9
            return {"ms": round(ms, 5), "bytes": nbytes, "GB/s": round(g, 1), "frac_hbm": round(g / float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])), 4),
                    "launches": launches}
        # Sage2 quantise-and-exchange of the same q/k/v (whole sequence used)
        sage = qb.sage2_outputs(P, 1, S, wl.num_heads, D, P * S)
        ms_sg, _ = timed(lambda: qb.ulysses_sage2_scatter_qkv(ranks[:, :, 0], ranks[:, :, 1], ranks[:, :, 2], P,
                                                              P * S, sage))
        n_el = 3 * P * S * wl.num_heads * D
        extra_sage = row(ms_sg, n_el * 2 + n_el, 3)   # read bf16 q/k/v once, write 1-byte codes (scales < 0.1 %)
        extra_sage["moved_bytes"] = n_el * 2 + n_el + (2 * n_el // 3) * 2   # + K and V read again by the statistics
        extra_sage["note"] = "GB/s on algorithmic bytes; the statistics pass reads K and V a second time"
        elt_b = 2
        pk_bytes = sum(2 * wl.B * S * W * cnt * 3 * D * elt_b for _, cnt in wl.schedule) * wl.P
        mg_bytes = sum(2 * wl.B * S * W * cnt * D * elt_b for _, cnt in wl.schedule) * wl.P
        extra = {"pack_schedule_call": row(ms_ps, pk_bytes, wl.P), "merge_schedule_call": row(ms_ms, mg_bytes, wl.P),
                 "sage2_scatter_qkv": extra_sage,
                 "scatter_heads": row(ms_sc, qbytes, 1), "gather_heads": row(ms_ga, qbytes, 1),
                 "scatter_qkv_head_chunk": row(ms_sq, 3 * qbytes, len(wl.schedule)),
                 "gather_output_head_chunk": row(ms_go, qbytes, len(wl.schedule)),
                 "pack_output_sequence_chunk": row(ms_sp, qbytes // P, len(wl.schedule))}
        elt = 2
        pack_bytes = sum(2 * wl.B * S * W * cnt * 3 * D * elt for _, cnt in wl.schedule) * wl.P
        merge_bytes = sum(2 * wl.B * S * W * cnt * D * elt for _, cnt in wl.schedule) * wl.P
        hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        gp, gm = pack_bytes / (ms_p * 1e-3) / 1e9, merge_bytes / (ms_m * 1e-3) / 1e9
        launches = wl.P * len(wl.schedule)
        line = {"metric": "head-chunk pack/merge GB/s", "value": round(gp, 1), "unit": "GB/s", "n_gpus": 1,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_p + ms_m, 5),
                "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
                "config": {"workload": name, "schedule": [list(b) for b in wl.schedule], "P": wl.P,
                           "l2": "flushed between steps"},
                "roofline": {"bound": "hbm", "achieved": round(gp, 1), "peak": hbm, "unit": "GB/s",
                             "frac": round(gp / hbm, 4), "peak_source": f"{peak_src} hbm_gbs"},
                "pack": {"ms": round(ms_p, 5), "bytes": pack_bytes, "GB/s": round(gp, 1), "frac_hbm": round(gp / hbm, 4),
                         "launches": launches},
                "merge": {"ms": round(ms_m, 5), "bytes": merge_bytes, "GB/s": round(gm, 1),
                          "frac_hbm": round(gm / hbm, 4), "launches": launches},
                "gpu_launches": 2 * launches * args.steps, "clocks": clk}
        line.update(extra)
    else:
        raise SystemExit(f"unknown workload {name!r}")
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-sample-tokens", type=int, default=4096)
    ap.add_argument("--ref-sample-tokens", type=int, default=128)
    ap.add_argument("--ref-budget-s", type=float, default=90.0,
                    help="CPU seconds the reference arm spreads over warm-up + timed steps")
    ap.add_argument("--no-overlap", action="store_true",
                    help="run pack/merge after the fused op on one stream instead of beside it")
    ap.add_argument("--reserve-sms", type=int, default=0,
                    help="SMs the fused kernel leaves to the concurrent pack/merge (overlapped step only)")
    ap.add_argument("--workload", default=None,
                    help="time one row alone on this workload instead of the headline step")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.workload:
        run_gpu_workload(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
