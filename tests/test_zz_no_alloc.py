"""The allocation-free forward (qnre_forward_noalloc) against the plan-based qnre_forward
and the CPU oracle.

qnre_forward_noalloc serves callers that cannot call cudaMalloc when they run
the projection (a memory pool that forbids raw allocations, a runtime that owns
all device memory, a server that must not allocate once running): it needs no
plan and keeps its status word in the library's static device scratch.  This
file is collected last so that a run stopping at the first failure has already
run every other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest

import oracle
from ulysses_qkv_proj_gb300 import workloads as WL
from _util import assert_fused_close, to_dev_bf16, to_host_bits, to_host_f64

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from ulysses_qkv_proj_gb300 import binding as qb  # noqa: E402


def _noalloc():
    lib = qb.load_library()
    fn = lib.qnre_forward_noalloc
    c_int, c_vp = ctypes.c_int, ctypes.c_void_p
    fn.restype = c_int
    fn.argtypes = [c_int, c_int, c_int, c_int, c_int, ctypes.c_uint, c_int, c_int,
                   c_vp, c_vp, c_vp, c_vp, c_vp, ctypes.c_int64, c_vp, ctypes.POINTER(qb._Out), c_vp, c_vp]
    return fn


def _host_inputs(wl, bad_positions=()):
    inp = WL.make_fused_inputs(wl)
    if bad_positions:
        inp.positions = inp.positions.copy()
        flat = inp.positions.reshape(-1)
        for t in bad_positions:
            flat[t] = wl.n_pos + 5
    return inp


def _inputs(wl, bad_positions=(), inp=None):
    inp = inp or _host_inputs(wl, bad_positions)
    return dict(x=to_dev_bf16(inp.x), w=to_dev_bf16(inp.w), qw=to_dev_bf16(inp.q_norm_w),
                kw=to_dev_bf16(inp.k_norm_w), cs=torch.from_numpy(inp.cos_sin).cuda(),
                pos=torch.from_numpy(inp.positions).cuda())


def _call_noalloc(fn, wl, d, out, status):
    o = qb._Out(*(out[g].data_ptr() if g in out else None for g in ("q", "k", "v", "fused")))
    return fn(wl.hidden, wl.num_heads, wl.P, qb.LAYOUTS[wl.layout], qb.ROPE_STYLES[wl.rope_style], 0,
              wl.B, wl.S, d["x"].data_ptr(), d["w"].data_ptr(), d["qw"].data_ptr(), d["kw"].data_ptr(),
              d["cs"].data_ptr(), d["cs"].shape[0], d["pos"].data_ptr(), ctypes.byref(o), status.data_ptr(),
              torch.cuda.current_stream().cuda_stream)


def test_noalloc_forward_matches_plan_forward_on_two_calls_in_a_row():
    """Two calls in a row.  Each output equals, bit for bit, a plan forward that takes
    the same one-pair-per-cluster form (QNRE_FLAG_ONE_PAIR), and the CPU oracle
    element by element within max(2 bf16 ulp, 2e-2)."""
    fn = _noalloc()
    calls = [
        # first call: one token with a position outside the table -> its q/k rows are NaN
        (WL.FusedWorkload("noalloc_a", P=2, B=2, S=200, num_heads=4), (37,)),
        # second call, straight after: another geometry; its status must not carry the first call's bit
        (WL.FusedWorkload("noalloc_b", P=4, B=1, S=96, num_heads=8, layout="fused",
                          rope_style="interleaved"), ()),
    ]
    status = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    results = []
    for i, (wl, bad) in enumerate(calls):
        inp = _host_inputs(wl, bad)
        d = _inputs(wl, inp=inp)
        plan = qb.Plan(wl.hidden, wl.num_heads, wl.P, wl.layout, max_tokens=wl.B * wl.S,
                       rope_style=wl.rope_style, flags=qb.FLAG_ONE_PAIR)
        ref = qb.alloc_outputs(plan, wl.B, wl.S)
        qb.qnre_forward(plan, d["x"], d["w"], d["qw"], d["kw"], d["cs"], d["pos"], ref)
        out = qb.alloc_outputs(plan, wl.B, wl.S)
        for t in out.values():
            t.view(torch.int16).fill_(-1)
        st = _call_noalloc(fn, wl, d, out, status[i:i + 1])
        assert st == 0, qb.STATUS_NAMES.get(st, st)
        torch.cuda.synchronize()
        plan_bits = plan.device_status()
        results.append((wl, inp, ref, out, plan_bits))
    bits = status.cpu().tolist()
    assert bits[0] == qb.DEVICE_BAD_POSITION and results[0][4] == qb.DEVICE_BAD_POSITION
    assert bits[1] == 0 and results[1][4] == 0
    for wl, inp, ref, out, _ in results:
        want = oracle.qnre_forward(inp.x, inp.w, inp.q_norm_w, inp.k_norm_w, inp.cos_sin, inp.positions,
                                   wl.P, wl.num_heads, wl.layout, wl.rope_style)
        for g in ref:
            assert np.array_equal(to_host_bits(out[g]), to_host_bits(ref[g])), f"{wl.name}/{g}"
            assert_fused_close(to_host_f64(out[g]), want[g], what=f"{wl.name}/{g}")


def test_noalloc_rejects_before_enqueueing():
    fn = _noalloc()
    wl = WL.FusedWorkload("noalloc_c", P=2, B=1, S=64, num_heads=4)
    d = _inputs(wl)
    out = {g: torch.empty((2, 1, 128, 2, 128), dtype=torch.bfloat16, device="cuda") for g in "qkv"}
    status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    o = qb._Out(out["q"].data_ptr(), out["k"].data_ptr(), out["v"].data_ptr(), None)
    stream = torch.cuda.current_stream().cuda_stream
    args = [d["x"].data_ptr(), d["w"].data_ptr(), d["qw"].data_ptr(), d["kw"].data_ptr(), d["cs"].data_ptr(),
            d["cs"].shape[0], d["pos"].data_ptr(), ctypes.byref(o), status.data_ptr(), stream]
    assert fn(500, 4, 2, 0, 0, 0, 1, 64, *args) == 1             # hidden != heads * 128
    assert fn(512, 4, 3, 0, 0, 0, 1, 64, *args) == 1             # heads % P != 0
    assert fn(512, 4, 2, 0, 0, 0, 1 << 20, 1 << 12, *args) == 5  # tokens beyond the kernel's range
    torch.cuda.synchronize()
    assert status.item() == 12345                                # nothing was enqueued


def test_noalloc_forward_replays_in_a_cuda_graph():
    """After its first call on the device, the call can be captured: a CUDA graph of
    one no-alloc forward, replayed on fresh inputs copied into the captured buffers,
    gives the same bits as a one-pair plan forward on those inputs each time."""
    fn = _noalloc()
    wl = WL.FusedWorkload("noalloc_g", P=2, B=1, S=160, num_heads=4)
    inp = _host_inputs(wl)
    d = _inputs(wl, inp=inp)
    plan = qb.Plan(wl.hidden, wl.num_heads, wl.P, wl.layout, max_tokens=wl.B * wl.S, flags=qb.FLAG_ONE_PAIR)
    out = qb.alloc_outputs(plan, wl.B, wl.S)
    status = torch.zeros((1,), dtype=torch.int32, device="cuda")
    assert _call_noalloc(fn, wl, d, out, status) == 0           # set-up call, outside the capture
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        assert _call_noalloc(fn, wl, d, out, status) == 0
    rng = np.random.default_rng(3)
    for rep in range(2):
        x_new = rng.standard_normal(inp.x.shape).astype(np.float32)
        d["x"].copy_(to_dev_bf16(WL.f32_to_bf16_bits(x_new)))
        for t in out.values():
            t.view(torch.int16).fill_(-1)
        graph.replay()
        torch.cuda.synchronize()
        ref = qb.alloc_outputs(plan, wl.B, wl.S)
        qb.qnre_forward(plan, d["x"], d["w"], d["qw"], d["kw"], d["cs"], d["pos"], ref)
        torch.cuda.synchronize()
        assert status.item() == 0 and plan.device_status() == 0
        for g in ref:
            assert np.array_equal(to_host_bits(out[g]), to_host_bits(ref[g])), f"replay {rep}/{g}"
