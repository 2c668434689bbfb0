"""The debug build (libqnre_debug.so, QNRE_DEBUG_BOUNDS=1): every load and store of
the layout and Sage2 kernels and every head-row store of the fused epilogue is
checked against its buffer's byte range, and an access outside it is counted and
skipped.  Each entry point runs in a child process once on the release library
and once on the debug library: the debug run must count nothing, raise no
status bit and give the same bytes.  A positive control takes 256 bytes off the
end of every output range (QNRE_DEBUG_SHRINK_OUTPUT, a hook of the debug build
alone): the stores there are then counted and skipped, so those bytes keep
their fill value while every other byte still matches."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = os.path.dirname(os.path.abspath(__file__))
FILL = 0x55
SHRINK = 256


# ---------------------------------------------------------------- child side
def _filled(shape, dtype):
    t = torch.empty(shape, dtype=dtype, device="cuda")
    t.view(torch.uint8).fill_(FILL)
    return t


def _calls(which):
    """(name, thunk) pairs; each thunk runs one entry point and returns
    (outputs, device status bits or None)."""
    from ulysses_qkv_proj_gb300 import binding as qb
    from ulysses_qkv_proj_gb300 import workloads as WL

    def bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()

    def fused(layout, mode):
        wl = WL.FusedWorkload("dbg", P=2, B=1, S=320, num_heads=4, layout=layout)  # 640 tokens: a ragged tile
        inp = WL.make_fused_inputs(wl)
        x, w, qw, kw = bf16(inp.x), bf16(inp.w), bf16(inp.q_norm_w), bf16(inp.k_norm_w)
        cs = torch.from_numpy(inp.cos_sin).cuda()
        pos = torch.from_numpy(inp.positions).cuda()
        shapes = ({g: (wl.P, wl.B, wl.P * wl.S, wl.H_local, 128) for g in "qkv"} if layout == "bshd"
                  else {"fused": (wl.P, wl.B, wl.P * wl.S, wl.H_local, 384)})
        out = {g: _filled(s, torch.bfloat16) for g, s in shapes.items()}
        if mode == "noalloc":
            st = torch.zeros(1, dtype=torch.int32, device="cuda")
            qb.qnre_forward_noalloc(wl.hidden, wl.num_heads, wl.P, x, w, qw, kw, cs, pos, out, layout=layout,
                                    device_status=st)
            torch.cuda.synchronize()
            return list(out.values()), int(st.item())
        plan = qb.Plan(wl.hidden, wl.num_heads, wl.P, layout, max_tokens=wl.B * wl.S)
        if mode == "publish":
            ready = torch.zeros(wl.P, dtype=torch.int32, device="cuda")
            qb.qnre_forward_publish(plan, x, w, qw, kw, cs, pos, out, ready)
            qb.qnre_wait_ready(plan, ready, qb.qnre_ready_target(plan, wl.B, wl.S), 1_000_000_000)
        else:
            qb.qnre_forward(plan, x, w, qw, kw, cs, pos, out)
        torch.cuda.synchronize()
        return list(out.values()), plan.device_status()

    # q/k/v as slices of one [B, S_global, 3, H, D] buffer (strided views)
    B, Sg, H, D, W = 2, 200, 8, 128, 2
    buf = bf16(WL.make_headchunk_buffer(B, Sg, H, D))
    q, k, v = buf[:, :, 0], buf[:, :, 1], buf[:, :, 2]
    qe, ke, ve = q[..., ::2], k[..., ::2], v[..., ::2]  # innermost stride 2: the element path

    def pack(views, off, cnt):
        d = views[0].shape[-1]
        out = _filled((B, Sg, W * cnt, 3 * d), torch.bfloat16)
        qb.ulysses_pack_head_chunk(*views, W, off, cnt, out)
        return [out], None

    def pack_schedule():
        sched = [(0, 1), (1, 2), (3, 1)]
        outs = [_filled((B, Sg, W * c, 3 * D), torch.bfloat16) for _, c in sched]
        qb.ulysses_pack_head_chunk_schedule(q, k, v, W, sched, outs)
        return outs, None

    L_heads = H // W
    recv = bf16(WL.make_received(B, Sg, W * 2, D))

    def merge():
        out = _filled((B, Sg, W * L_heads, D), torch.bfloat16)
        qb.ulysses_merge_output_head_chunk(recv, W, L_heads, 1, out)
        return [out], None

    def merge_schedule():
        out = _filled((B, Sg, W * L_heads, D), torch.bfloat16)
        r0 = bf16(WL.make_received(B, Sg, W * 1, D, seed=7))
        r1 = bf16(WL.make_received(B, Sg, W * 3, D, seed=8))
        qb.ulysses_merge_output_head_chunk_schedule([r0, r1], W, L_heads, [0, 1], out)
        return [out], None

    P, Bs, S_l, Hs = 4, 2, 37, 8
    xs = bf16(np.random.default_rng(3).integers(0, 1 << 16, (P, Bs, S_l, Hs, D)).astype(np.uint16))

    def scatter_heads():
        y = _filled((P, Bs, P * S_l, Hs // P, D), torch.bfloat16)
        qb.ulysses_scatter_heads(xs, y)
        return [y], None

    def gather_heads():
        y = bf16(np.random.default_rng(6).integers(0, 1 << 16, (P, Bs, P * S_l, Hs // P, D)).astype(np.uint16))
        back = _filled(xs.shape, torch.bfloat16)
        qb.ulysses_gather_heads(y, back)
        return [back], None

    def seq_pack():
        x = recv[:, :, 1:3]  # a head-strided view [B, S_global, 2, D]
        out = _filled((W, B, Sg // W, 2, D), torch.bfloat16)
        qb.ulysses_pack_output_sequence_chunk(x, W, out)
        return [out], None

    def gather_out_chunk():
        x = bf16(np.random.default_rng(4).integers(0, 1 << 16, (P, Bs, P * S_l, 1, D)).astype(np.uint16))
        out = _filled((P, Bs, S_l, P * 2, D), torch.bfloat16)
        qb.ulysses_gather_output_head_chunk(x, 2, 1, out)
        return [out], None

    def scatter_qkv(views):
        # views [B, S, H, d] read as 2 virtual ranks of B // 2 = 1 batch row each; heads 1..2 of every band
        d = views[0].shape[-1]
        out = _filled((2, B // 2, 2 * Sg, 2, 3 * d), torch.bfloat16)
        qb.ulysses_scatter_qkv_head_chunk(*views, 2, 1, 2, out)
        return [out], None

    def sage2(dtype, D2, U):
        P2, B2, L2, H2 = 2, 1, 150, 4
        rng = np.random.default_rng(5)
        a = torch.from_numpy(rng.standard_normal((P2 * B2, L2, 3, H2, D2)).astype(np.float32)).cuda().to(dtype)
        out = qb.sage2_outputs(P2, B2, L2, H2, D2, U)
        for t in out.values():
            t.view(torch.uint8).fill_(FILL)
        qb.ulysses_sage2_scatter_qkv(a[:, :, 0], a[:, :, 1], a[:, :, 2], P2, U, out)
        return [out[n] for n in ("q", "k", "v", "q_scale", "k_scale", "v_scale")], None

    calls = [
        ("forward_bshd", lambda: fused("bshd", "plan")),
        ("forward_fused", lambda: fused("fused", "plan")),
        ("forward_publish", lambda: fused("bshd", "publish")),
        ("forward_noalloc", lambda: fused("fused", "noalloc")),
        ("pack_vector", lambda: pack((q, k, v), 1, 2)),
        ("pack_element", lambda: pack((qe, ke, ve), 0, 3)),
        ("pack_schedule", pack_schedule),
        ("merge", merge),
        ("merge_schedule", merge_schedule),
        ("scatter_heads", scatter_heads),
        ("gather_heads", gather_heads),
        ("pack_sequence_chunk", seq_pack),
        ("gather_output_head_chunk", gather_out_chunk),
        ("scatter_qkv_vector", lambda: scatter_qkv((q, k, v))),
        ("scatter_qkv_element", lambda: scatter_qkv((qe, ke, ve))),
        ("sage2_bf16_d128", lambda: sage2(torch.bfloat16, 128, 260)),
        ("sage2_fp16_d64", lambda: sage2(torch.float16, 64, 300)),
    ]
    if which == "control":
        keep = {"forward_bshd", "forward_fused", "pack_vector", "pack_element", "scatter_heads",
                "gather_heads", "sage2_bf16_d128"}
        calls = [c for c in calls if c[0] in keep]
    return calls


def child_main(out_path: str, which: str) -> None:
    """Run the calls on the library QNRE_LIB names; save every output's bytes to
    out_path (.npz) and print one JSON line of statuses and violation counts."""
    from ulysses_qkv_proj_gb300 import binding as qb
    debug = os.environ.get("QNRE_LIB", "") == qb.DEBUG_LIB_PATH
    if debug:
        qb.debug_bounds(reset=True)
    arrays, report = {}, {}
    for name, thunk in _calls(which):
        outs, status = thunk()
        torch.cuda.synchronize()
        for i, t in enumerate(outs):
            arrays[f"{name}.{i}"] = t.contiguous().view(torch.uint8).cpu().numpy().reshape(-1)
        report[name] = {"status": status, "violations": qb.debug_bounds(reset=True) if debug else None}
    np.savez(out_path, **arrays)
    print(json.dumps(report))


# --------------------------------------------------------------- parent side
@pytest.fixture(scope="module")
def debug_lib():
    from ulysses_qkv_proj_gb300 import build
    return build.build(debug_bounds=True)


def _child(tmp_path, lib, which, shrink=None):
    env = dict(os.environ, QNRE_LIB=lib, PYTHONPATH=os.pathsep.join([ROOT, TESTS]))
    env.pop("QNRE_DEBUG_SHRINK_OUTPUT", None)
    if shrink is not None:
        env["QNRE_DEBUG_SHRINK_OUTPUT"] = str(shrink)
    tag = f"{os.path.basename(lib)}_{which}_{shrink}"
    path = str(tmp_path / f"{tag}.npz")
    code = "import sys, test_gpu_debug_bounds as t; t.child_main(sys.argv[1], sys.argv[2])"
    res = subprocess.run([sys.executable, "-c", code, path, which], cwd=ROOT, env=env, capture_output=True,
                         text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-3000:]
    report = json.loads(res.stdout.strip().splitlines()[-1])
    return report, dict(np.load(path))


def test_debug_build_counts_nothing_and_matches_release(tmp_path, debug_lib):
    from ulysses_qkv_proj_gb300 import binding as qb
    rel_report, rel = _child(tmp_path, qb.LIB_PATH, "all")
    dbg_report, dbg = _child(tmp_path, debug_lib, "all")
    assert set(rel) == set(dbg)
    for name, r in dbg_report.items():
        assert r["violations"] == 0, (name, r)
        assert r["status"] in (None, 0), (name, r)
        assert rel_report[name]["status"] in (None, 0), (name, rel_report[name])
    for key in rel:
        assert np.array_equal(rel[key], dbg[key]), key
    # every output was written somewhere (the fill value is not what the calls leave)
    for key, a in dbg.items():
        assert (a != FILL).any(), key


def test_shrunk_ranges_skip_exactly_the_tail(tmp_path, debug_lib):
    """Positive control: with SHRINK bytes taken off every output range, stores to
    each output's last SHRINK bytes are counted and skipped, the rest is unchanged."""
    from ulysses_qkv_proj_gb300 import binding as qb
    _, rel = _child(tmp_path, qb.LIB_PATH, "control")
    report, got = _child(tmp_path, debug_lib, "control", shrink=SHRINK)
    for name, r in report.items():
        if name.startswith("forward"):
            assert r["status"] == qb.DEVICE_BOUNDS, (name, r)   # the fused epilogue reports in the status word
            assert r["violations"] == 0, (name, r)
        else:
            assert r["violations"] > 0, (name, r)
    scales = {"sage2_bf16_d128.3", "sage2_bf16_d128.4", "sage2_bf16_d128.5"}  # scale outputs are not shrunk
    for key in rel:
        a, b = rel[key], got[key]
        if key in scales:
            assert np.array_equal(a, b), key
            continue
        assert np.array_equal(a[:-SHRINK], b[:-SHRINK]), key
        assert (b[-SHRINK:] == FILL).all(), key
        assert (a[-SHRINK:] != FILL).any(), key
