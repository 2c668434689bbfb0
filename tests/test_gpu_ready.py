"""Readiness words: the fused epilogue publishes per-destination counts, and a one-CTA
bounded wait acquires them.  The wait is also the GPU failure-detection case: with a
word that nothing ever sets it gives up after its limit, raises a status bit that the
host reads, and leaves the context usable."""
import time

import numpy as np
import pytest

import oracle
from ulysses_qkv_proj_gb300 import workloads as WL
from _util import assert_fused_close, to_dev_bf16, to_host_bits, to_host_f64

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from ulysses_qkv_proj_gb300 import binding as qb  # noqa: E402


def _expected_count(wl):
    """Publications each destination rank receives in a complete forward, from the
    tile geometry: tokens are processed in 256-row tiles, each stored by 8 epilogue
    warps (4 in each CTA of the pair, 32 rows apiece), and a warp publishes once per
    head it stores; rank r is the destination of 3 * H_local heads (its q, k and v
    bands) of every token."""
    row_tiles = -(-wl.T // 256)
    return row_tiles * 8 * 3 * wl.H_local


def _setup(wl, with_host=False):
    inp = WL.make_fused_inputs(wl)
    d = dict(x=to_dev_bf16(inp.x), w=to_dev_bf16(inp.w), qw=to_dev_bf16(inp.q_norm_w),
             kw=to_dev_bf16(inp.k_norm_w), cs=torch.from_numpy(inp.cos_sin).cuda(),
             pos=torch.from_numpy(inp.positions).cuda())
    plan = qb.Plan(wl.hidden, wl.num_heads, wl.P, wl.layout, max_tokens=wl.B * wl.S, rope_style=wl.rope_style)
    return (plan, d, inp) if with_host else (plan, d)


@pytest.mark.parametrize("wl", [
    WL.FusedWorkload("ready_a", P=4, B=2, S=96, num_heads=8),                 # 3 row tiles (odd)
    WL.FusedWorkload("ready_b", P=2, B=1, S=200, num_heads=6, layout="fused"),
    WL.FusedWorkload("ready_c", P=2, B=2, S=512, num_heads=4),                # 8 row tiles, two-pair clusters
])
def test_publish_reaches_target_and_wait_passes(wl):
    plan, d, inp = _setup(wl, with_host=True)
    ref = qb.alloc_outputs(plan, wl.B, wl.S)
    qb.qnre_forward(plan, d["x"], d["w"], d["qw"], d["kw"], d["cs"], d["pos"], ref)
    out = qb.alloc_outputs(plan, wl.B, wl.S)
    ready = torch.full((wl.P,), 12345, dtype=torch.int32, device="cuda")  # the call zeroes it first
    qb.qnre_forward_publish(plan, d["x"], d["w"], d["qw"], d["kw"], d["cs"], d["pos"], out, ready)
    target = _expected_count(wl)
    assert qb.qnre_ready_target(plan, wl.B, wl.S) == target
    done = torch.cuda.Event()
    done.record()
    consumer = torch.cuda.Stream()
    consumer.wait_event(done)               # the wait runs after the producer, never beside it
    qb.qnre_wait_ready(plan, ready, target, 1_000_000_000, stream=consumer)
    torch.cuda.synchronize()
    assert ready.cpu().tolist() == [target] * wl.P
    assert plan.device_status() == 0
    want = oracle.qnre_forward(inp.x, inp.w, inp.q_norm_w, inp.k_norm_w, inp.cos_sin, inp.positions,
                               wl.P, wl.num_heads, wl.layout, wl.rope_style)
    for g in ref:
        assert np.array_equal(to_host_bits(out[g]), to_host_bits(ref[g]))
        assert_fused_close(to_host_f64(out[g]), want[g], what=f"{wl.name}/{g}")


def test_wait_gives_up_when_nothing_publishes():
    wl = WL.FusedWorkload("ready_e", P=2, B=1, S=64, num_heads=2)
    plan, d = _setup(wl)
    ready = torch.zeros((wl.P,), dtype=torch.int32, device="cuda")  # nothing will ever add to it
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    qb.qnre_wait_ready(plan, ready, 1, 50_000_000)  # 50 ms
    bits = plan.device_status()                     # waits for the stream, then reads the word
    elapsed = time.perf_counter() - t0
    assert bits & qb.DEVICE_READY_TIMEOUT
    assert 0.04 < elapsed < 5.0
    # the context is still usable: a normal forward runs and reports a clean status
    out = qb.alloc_outputs(plan, wl.B, wl.S)
    qb.qnre_forward(plan, d["x"], d["w"], d["qw"], d["kw"], d["cs"], d["pos"], out)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    assert not bool(torch.isnan(out["q"]).any())


def test_publish_rejects_bad_ready_buffer():
    wl = WL.FusedWorkload("ready_d", P=2, B=1, S=64, num_heads=2)
    plan, d = _setup(wl)
    out = qb.alloc_outputs(plan, wl.B, wl.S)
    with pytest.raises(qb.QnreError) as e:   # the words may not live inside an output
        qb.qnre_forward_publish(plan, d["x"], d["w"], d["qw"], d["kw"], d["cs"], d["pos"], out,
                                out["v"].view(torch.int32).view(-1)[:2])
    assert e.value.status == 4
    with pytest.raises(qb.QnreError) as e:
        qb.qnre_wait_ready(plan, torch.zeros(2, dtype=torch.int32, device="cuda"), 1, 0)
    assert e.value.status == 1
