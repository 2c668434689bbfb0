"""A prepared forward and the head-chunk copies captured in a CUDA graph and replayed
with fresh inputs ("QKV projection + RMSNorm + RoPE overlapped with the Ulysses head
exchange", Tests: checks after CUDA-graph replays with fresh inputs; [FUSED]: a
prepared call allocates nothing and runs no host collective, so it can be captured)."""
import numpy as np
import pytest

import oracle
from ulysses_qkv_proj_gb300 import workloads as WL
from _sage2 import assert_sage2_matches, sage2_oracle
from _util import assert_fused_close, to_dev_bf16, to_host_bits, to_host_f64

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from ulysses_qkv_proj_gb300 import binding as qb  # noqa: E402


def test_forward_and_pack_merge_replay_with_fresh_inputs():
    # 1024 tokens = 4 row tiles: the plan takes clusters of two pairs sharing W (multicast)
    wl = WL.FusedWorkload("graph", P=2, B=2, S=256, num_heads=4, layout="fused", rope_style="interleaved")
    plan = qb.Plan(wl.hidden, wl.num_heads, wl.P, wl.layout, max_tokens=wl.B * wl.S, rope_style=wl.rope_style)
    base = WL.make_fused_inputs(wl)
    x = to_dev_bf16(base.x)
    w = to_dev_bf16(base.w)
    qw, kw = to_dev_bf16(base.q_norm_w), to_dev_bf16(base.k_norm_w)
    cs = torch.from_numpy(base.cos_sin).cuda()
    pos = torch.from_numpy(base.positions).cuda()
    out = qb.alloc_outputs(plan, wl.B, wl.S)
    B2, S2, H2, D, W = 1, 48, 8, 128, 2
    buf = torch.empty((B2, S2, 3, H2, D), dtype=torch.bfloat16, device="cuda")
    packed = torch.empty((B2, S2, W * 2, 3 * D), dtype=torch.bfloat16, device="cuda")
    merged = torch.zeros((B2, S2, H2, D), dtype=torch.bfloat16, device="cuda")

    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):  # one eager call first (device set-up happens outside capture)
        qb.qnre_forward(plan, x, w, qw, kw, cs, pos, out, stream=stream)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        s = torch.cuda.current_stream()
        qb.qnre_forward(plan, x, w, qw, kw, cs, pos, out, stream=s)
        qb.ulysses_pack_head_chunk(buf[:, :, 0], buf[:, :, 1], buf[:, :, 2], W, 1, 2, packed, stream=s)
        qb.ulysses_merge_output_head_chunk(packed[..., :D], W, H2 // W, 1, merged, stream=s)

    rng = np.random.default_rng(5)
    for replay in range(3):
        xs = WL.f32_to_bf16_bits(rng.standard_normal(base.x.shape).astype(np.float32))
        bs = rng.integers(0, 1 << 16, size=(B2, S2, 3, H2, D)).astype(np.uint16)
        x.copy_(to_dev_bf16(xs))
        buf.copy_(to_dev_bf16(bs))
        for t in out.values():
            t.view(torch.int16).fill_(-1)
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert plan.device_status() == 0
        ref = oracle.qnre_forward(xs, base.w, base.q_norm_w, base.k_norm_w, base.cos_sin, base.positions,
                                  wl.P, wl.num_heads, wl.layout, wl.rope_style)
        assert_fused_close(to_host_f64(out["fused"]), ref["fused"], what=f"replay {replay}")
        want = oracle.pack_head_chunk(bs[:, :, 0], bs[:, :, 1], bs[:, :, 2], W, 1, 2)
        assert np.array_equal(to_host_bits(packed), want)
        got_m = to_host_bits(merged)
        band = np.zeros(H2, bool)
        for r in range(W):
            band[r * (H2 // W) + 1: r * (H2 // W) + 3] = True
        assert np.array_equal(got_m[:, :, band], bs[:, :, 0][:, :, band])


def test_sage2_replay_with_fresh_inputs():
    """The Sage2 encoding captured once (after one eager call, which makes the
    per-device set-up) and replayed on new q/k/v: every code and scale bit equals
    the oracle's on each replay."""
    P, B, L, H, D, U = 2, 1, 96, 4, 128, 180
    buf = torch.zeros((P * B, L, 3, H, D), dtype=torch.bfloat16, device="cuda")
    q, k, v = buf[:, :, 0], buf[:, :, 1], buf[:, :, 2]
    enc = qb.sage2_outputs(P, B, L, H, D, U)
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        qb.ulysses_sage2_scatter_qkv(q, k, v, P, U, enc, stream=stream)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        qb.ulysses_sage2_scatter_qkv(q, k, v, P, U, enc, stream=torch.cuda.current_stream())
    rng = np.random.default_rng(8)
    live = (np.arange(P * L) < U).reshape(P * B, L, 1, 1, 1)
    for replay in range(3):
        a = (rng.standard_normal((P * B, L, 3, H, D)) * (1 + replay)).astype(np.float32)
        a[:, :, 1] += 1.5                                       # K offset: the mean removal matters
        bits = WL.f32_to_bf16_bits(np.where(live, a, 0))
        buf.copy_(to_dev_bf16(bits))
        for t in enc.values():
            if t is not enc["workspace"]:
                t.view(torch.uint8).fill_(0x55)
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        ranks = bits.reshape(P, B, L, 3, H, D)
        assert_sage2_matches(enc, sage2_oracle(ranks, U, "bf16"), P)
