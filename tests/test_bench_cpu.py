"""CPU checks of the benchmark's host logic: it runs on one GPU only and refuses a
multi-process launch (as torchrun starts it, and with --gpus > 1) before touching
any GPU; under torchrun only rank 0 runs and prints the reference arm; the token
sample of the CPU baseline covers every segment and 256-row tile edge; the clock
summary reduces only the samples inside a timed region; the profiled traffic is
used only while the kernel sources still hash to the value it was taken on."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _no_gpu_env(**extra):
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    env.update(extra)
    return env


def test_refuses_two_ranks_under_torchrun():
    """The driver's multi-GPU launch: both gloo-free ranks exit non-zero before any
    process group or GPU work, and no JSON line is printed."""
    port = _free_port()
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", str(port),
                        os.path.join(ROOT, "bench.py"), "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       capture_output=True, text=True, env=_no_gpu_env(), timeout=300)
    assert r.returncode != 0
    assert "one GPU only" in r.stderr
    assert "{" not in r.stdout


@pytest.mark.parametrize("env,flags", [({"WORLD_SIZE": "2", "RANK": "0", "LOCAL_RANK": "0"}, []),
                                       ({}, ["--gpus", "4"])])
def test_refuses_more_than_one_gpu(env, flags):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "1"] + flags,
                       capture_output=True, text=True, env=_no_gpu_env(**env), timeout=120)
    assert r.returncode == 2 and "one GPU only" in r.stderr and r.stdout.strip() == ""


def test_reference_arm_only_rank0_prints():
    env = _no_gpu_env(RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], capture_output=True, text=True, env=env, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""


@pytest.mark.slow
def test_reference_arm_line_rank0():
    env = _no_gpu_env(RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                        "--warmup", "3", "--ref-budget-s", "5"], capture_output=True, text=True, env=env,
                       timeout=900)
    assert r.returncode == 0, r.stderr[-800:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "tokens/s"
    # the same config object as the GPU arm's line, so the two lines compare like for like
    assert line["config"] == bench.headline_config()
    assert line["config"]["workload"].startswith(bench.WORKLOAD.name + ":")
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


@pytest.mark.parametrize("n", [64, 300, 1024])
def test_stratified_tokens_cover_segments_and_tile_edges(n):
    for wl in (bench.WORKLOAD, bench.SMALL_FUSED):
        t = bench.stratified_tokens(wl, n)
        assert len(t) == len(set(t.tolist())) and t.min() >= 0 and t.max() < wl.T
        need = {e for t0 in range(0, wl.T, wl.S) for e in (t0, t0 + wl.S - 1)}
        need |= {e for t0 in range(0, wl.T, 256) for e in (t0, min(wl.T - 1, t0 + 255))}
        if n >= len(need):
            assert need <= set(t.tolist()) and len(t) == n
        else:
            assert len(t) <= n and {0, wl.T - 1} <= set(t.tolist())


def test_clock_summary_uses_only_samples_inside_the_region():
    cs = bench.ClockSampler("00000000:00:00.0")
    cs.source = "test"
    cs.sections["a"] = (10.0, 11.0)
    cs.samples = [(9.9, 500.0, 2070.0, 100.0, frozenset()),
                  (10.1, 2000.0, 2070.0, 1300.0, frozenset({"sw_power_cap"})),
                  (10.5, 1900.0, 2070.0, 1390.0, frozenset()),
                  (10.9, 1800.0, 2070.0, 1350.0, frozenset()),
                  (11.2, 400.0, 2070.0, 90.0, frozenset({"hw_slowdown"}))]
    s = cs.summary("a")
    assert s["samples"] == 3 and s["sm_mhz"] == 1900.0 and s["sm_mhz_min"] == 1800.0
    assert s["reasons"] == ["sw_power_cap"] and s["power_w_max"] == 1390.0
    assert cs.summary("missing")["samples"] == 0


def test_profiled_traffic_is_gated_by_the_kernel_source_hash(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    for f in bench.FUSED_SOURCES:
        p = tmp_path / f
        p.parent.mkdir(parents=True, exist_ok=True)
        p.write_bytes(open(os.path.join(ROOT, f), "rb").read())
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    rec = {"fused_qkv_kernel": {"w": {"kernel_source_hash": bench.fused_source_hash(),
                                      "dram_bytes_per_launch": 1234}}}
    (tmp_path / bench.TRAFFIC_FILE).write_text(json.dumps(rec))
    assert bench.profiled_traffic("w") == 1234
    assert bench.profiled_traffic("other") is None
    with open(tmp_path / bench.FUSED_SOURCES[0], "a") as f:
        f.write("// changed\n")
    assert bench.profiled_traffic("w") is None


def test_committed_traffic_record_is_well_formed():
    path = os.path.join(ROOT, bench.TRAFFIC_FILE)
    if not os.path.exists(path):
        pytest.skip("no traffic record committed")
    rec = json.load(open(path))
    for wl, r in rec["fused_qkv_kernel"].items():
        assert isinstance(r["dram_bytes_per_launch"], int) and r["dram_bytes_per_launch"] > 0
        assert len(r["kernel_source_hash"]) == 16 and r["command"]
