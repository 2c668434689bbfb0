"""Stream order through the whole front end on one stream, against the oracle.

The layout copies are programmatic dependent launches: their blocks may be
scheduled while the previous kernel in the stream drains, and must wait for it
before they read.  Here every copy reads what the kernel right before it wrote,
with nothing in between: the fused forward's bands go straight into the ordinary
gather (the inverse exchange), which gives every source rank its own tokens'
q/k/v with all heads; those feed the head-chunk pack of an uneven schedule, its
merge and the ordinary scatter.  Each stage is compared with the oracle applied
to the previous stage's expected result.
"""
import numpy as np
import pytest

import oracle
from ulysses_qkv_proj_gb300 import workloads as WL
from _util import assert_fused_close, to_dev_bf16, to_host_bits, to_host_f64

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from ulysses_qkv_proj_gb300 import binding as qb  # noqa: E402


@pytest.mark.parametrize("P,B,S,H,sched", [
    (4, 1, 512, 8, [(0, 1), (1, 1)]),       # 2048 tokens: eight 256-row tiles, TMA-stored bands
    (2, 2, 200, 6, [(0, 2), (2, 1)]),       # segments of 200: warps at segment edges store rows
])
def test_copies_read_the_projection_in_stream_order(P, B, S, H, sched):
    wl = WL.FusedWorkload("pipeline", P=P, B=B, S=S, num_heads=H)
    inp = WL.make_fused_inputs(wl)
    L, D = wl.H_local, 128
    plan = qb.Plan(wl.hidden, H, P, "bshd", max_tokens=B * S)
    out = qb.alloc_outputs(plan, B, S)
    gathered = {g: torch.empty((P, B, S, H, D), dtype=torch.bfloat16, device="cuda") for g in "qkv"}
    packed = [torch.empty((P * B, S, P * cnt, 3 * D), dtype=torch.bfloat16, device="cuda") for _, cnt in sched]
    merged = torch.full((P * B, S, H, D), -1.0, dtype=torch.bfloat16, device="cuda")
    rescattered = torch.empty((P, B, P * S, L, D), dtype=torch.bfloat16, device="cuda")
    x, w = to_dev_bf16(inp.x), to_dev_bf16(inp.w)
    qw, kw = to_dev_bf16(inp.q_norm_w), to_dev_bf16(inp.k_norm_w)
    cs, pos = torch.from_numpy(inp.cos_sin).cuda(), torch.from_numpy(inp.positions).cuda()
    torch.cuda.synchronize()

    # one stream, no synchronisation between the launches
    qb.qnre_forward(plan, x, w, qw, kw, cs, pos, out)
    for g in "qkv":
        qb.ulysses_gather_heads(out[g], gathered[g])
    q, k, v = (gathered[g].view(P * B, S, H, D) for g in "qkv")
    for (off, cnt), pk in zip(sched, packed):
        qb.ulysses_pack_head_chunk(q, k, v, P, off, cnt, pk)
    for (off, cnt), pk in zip(sched, packed):
        qb.ulysses_merge_output_head_chunk(pk[..., :D], P, L, off, merged)
    qb.ulysses_scatter_heads(gathered["q"], rescattered)
    torch.cuda.synchronize()
    assert plan.device_status() == 0

    # the fused bands, gathered back to each source rank: the per-token result
    O = oracle.project_norm_rope(inp.x.reshape(wl.T, wl.hidden), inp.w, inp.q_norm_w, inp.k_norm_w,
                                 inp.cos_sin, inp.positions.reshape(-1), H)             # [T, 3, H, D]
    for gi, g in enumerate("qkv"):
        assert_fused_close(to_host_f64(gathered[g]).reshape(wl.T, H, D), O[:, gi], what=f"gathered {g}")
    # pack / merge / scatter of exactly those bits
    gb = {g: to_host_bits(gathered[g]).reshape(P * B, S, H, D) for g in "qkv"}
    want_m = np.full((P * B, S, H, D), 0xBF80, np.uint16)                               # bf16 -1.0
    for (off, cnt), pk in zip(sched, packed):
        want = oracle.pack_head_chunk(gb["q"], gb["k"], gb["v"], P, off, cnt)
        assert np.array_equal(to_host_bits(pk), want), f"pack ({off}, {cnt})"
        want_m = oracle.merge_output_head_chunk(want[..., :D], P, L, off, want_m)
    assert np.array_equal(to_host_bits(merged), want_m)
    assert np.array_equal(to_host_bits(rescattered), oracle.scatter_heads(gb["q"].reshape(P, B, S, H, D)))
    assert np.array_equal(to_host_bits(rescattered), to_host_bits(out["q"]))          # scatter inverts gather
