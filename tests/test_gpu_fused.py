"""GPU parity of the fused QKV projection + RMSNorm + RoPE + band scatter against the oracle.

Values: |gpu - oracle| <= max(2 bf16 ulp(oracle), 2e-2) per element.
Placement: bit-exact, checked with integer-coded inputs (QNRE_FLAG_EPILOGUE_OFF)
whose projection is exact in every precision.
"""
import dataclasses

import numpy as np
import pytest

import oracle
from ulysses_qkv_proj_gb300 import workloads as WL
from _util import assert_fused_close, dest_index, sample_tokens, to_dev_bf16, to_host_bits, to_host_f64

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from ulysses_qkv_proj_gb300 import binding as qb  # noqa: E402


def _dev_inputs(inp):
    return dict(x=to_dev_bf16(inp.x), w=to_dev_bf16(inp.w), qw=to_dev_bf16(inp.q_norm_w),
                kw=to_dev_bf16(inp.k_norm_w), cs=torch.from_numpy(inp.cos_sin).cuda(),
                pos=torch.from_numpy(inp.positions).cuda())


def _run(wl, d, flags=0, positions="given", poison=True, stream=None):
    plan = qb.Plan(wl.hidden, wl.num_heads, wl.P, wl.layout, max_tokens=wl.B * wl.S,
                   rope_style=wl.rope_style, flags=flags)
    out = qb.alloc_outputs(plan, wl.B, wl.S)
    if poison:
        for t in out.values():
            t.view(torch.int16).fill_(-1)  # 0xFFFF: a NaN; every element must be rewritten
    pos = d["pos"] if positions == "given" else None
    qb.qnre_forward(plan, d["x"], d["w"], d["qw"], d["kw"], d["cs"], pos, out, stream=stream)
    torch.cuda.synchronize()
    status = plan.device_status()
    return plan, out, status


def _full_compare(wl, inp, out, positions=None):
    ref = oracle.qnre_forward(inp.x, inp.w, inp.q_norm_w, inp.k_norm_w, inp.cos_sin,
                              inp.positions if positions is None else positions,
                              wl.P, wl.num_heads, wl.layout, wl.rope_style)
    for g in ref:
        assert_fused_close(to_host_f64(out[g]), ref[g], what=f"{wl.name}/{g}")


def _wl(name, P, B, S, H, layout="bshd", rope="rotate_half"):
    return WL.FusedWorkload(name, P=P, B=B, S=S, num_heads=H, layout=layout, rope_style=rope)


def test_tiny_workload_full():
    wl = WL.FUSED_WORKLOADS["tiny_p2_s64_h4"]
    inp = WL.make_fused_inputs(wl)
    _, out, status = _run(wl, _dev_inputs(inp))
    assert status == 0
    _full_compare(wl, inp, out)


@pytest.mark.parametrize("layout", ["bshd", "fused"])
@pytest.mark.parametrize("rope", ["rotate_half", "interleaved"])
def test_ragged_multi_tile(layout, rope):
    # 800 tokens = 6.25 row tiles, segments of 200 straddle tile edges; 6 column tiles.
    wl = _wl("ragged", P=2, B=2, S=200, H=4, layout=layout, rope=rope)
    inp = WL.make_fused_inputs(wl)
    _, out, status = _run(wl, _dev_inputs(inp))
    assert status == 0
    _full_compare(wl, inp, out)


@pytest.mark.parametrize("P,B,S,H,layout", [
    (1, 1, 96, 2, "bshd"),      # one 256-row tile, three full 32-token warps stored by TMA, the rest past T
    (2, 3, 32, 4, "fused"),     # every segment one warp long
    (4, 1, 224, 8, "bshd"),     # 896 tokens: a ragged last pair tile, two-pair clusters
])
def test_tma_store_boxes_with_a_ragged_end(P, B, S, H, layout):
    """S a multiple of 32, so every full warp's 32 tokens lie in one segment and
    go out as TMA store boxes, while the problem ends inside a row tile."""
    wl = _wl("tma_tail", P=P, B=B, S=S, H=H, layout=layout)
    inp = WL.make_fused_inputs(wl)
    _, out, status = _run(wl, _dev_inputs(inp))
    assert status == 0
    _full_compare(wl, inp, out)


def test_odd_head_count_column_tail():
    # 3 heads -> N = 1152 = 4.5 tiles of 256 columns; P = 3 ranks of one head each.
    wl = _wl("oddh", P=3, B=1, S=50, H=3)
    inp = WL.make_fused_inputs(wl)
    _, out, status = _run(wl, _dev_inputs(inp))
    assert status == 0
    _full_compare(wl, inp, out)


def test_single_rank_and_many_ranks():
    for wl in (_wl("p1", P=1, B=3, S=70, H=2), _wl("p8", P=8, B=1, S=16, H=8, layout="fused")):
        inp = WL.make_fused_inputs(wl)
        _, out, status = _run(wl, _dev_inputs(inp))
        assert status == 0
        _full_compare(wl, inp, out)


def test_null_positions_use_token_index():
    wl = _wl("nullpos", P=2, B=2, S=40, H=2)
    inp = WL.make_fused_inputs(wl)
    inp.cos_sin = WL.rope_table(wl.T)  # rows for every token index
    _, out, status = _run(wl, _dev_inputs(inp), positions=None)
    assert status == 0
    _full_compare(wl, inp, out, positions=np.arange(wl.T))


@pytest.mark.parametrize("layout,rope", [("bshd", "rotate_half"), ("fused", "interleaved")])
def test_random_positions_into_a_larger_table(layout, rope):
    """Each token's cos/sin row is positions[token], anywhere in a table longer
    than the sequence: the rows must follow the given positions, not the token
    index or the global sequence index."""
    wl = _wl("randpos", P=2, B=2, S=96, H=4, layout=layout, rope=rope)
    inp = WL.make_fused_inputs(wl)
    rng = np.random.default_rng(17)
    inp.cos_sin = WL.rope_table(5000)
    inp.positions = rng.integers(0, 5000, size=(wl.P, wl.B, wl.S)).astype(np.int32)
    _, out, status = _run(wl, _dev_inputs(inp))
    assert status == 0
    _full_compare(wl, inp, out)


def test_bad_position_gives_nan_rows_and_status():
    wl = _wl("badpos", P=2, B=1, S=64, H=2)
    inp = WL.make_fused_inputs(wl)
    inp.positions = inp.positions.copy()
    inp.positions.reshape(-1)[[5, 70]] = [wl.n_pos, -3]
    plan, out, status = _run(wl, _dev_inputs(inp))
    assert status & qb.DEVICE_BAD_POSITION
    assert plan.device_status() == 0  # cleared by the first read
    _full_compare(wl, inp, out)        # NaN rows where the oracle has NaN, values elsewhere


def _exact_projection(x2, w_bits):
    """Closed form of x W for rows with one or two nonzeros: a sum of scaled W rows."""
    rows, cols = np.nonzero(x2)
    T = x2.shape[0]
    count = np.bincount(rows, minlength=T)
    assert count.min() >= 1 and count.max() <= 2
    first = np.searchsorted(rows, np.arange(T))
    second = np.minimum(first + 1, len(rows) - 1)
    v1 = oracle.bf16_to_f64(x2[rows[first], cols[first]]).astype(np.float32)
    v2 = np.where(count == 2, oracle.bf16_to_f64(x2[rows[second], cols[second]]), 0).astype(np.float32)
    wf = oracle.bf16_to_f64(w_bits).astype(np.float32)
    return wf[cols[first]] * v1[:, None] + wf[cols[second]] * v2[:, None]


def _exact_placement(wl):
    inp = WL.make_exact_fused_inputs(wl)
    _, out, status = _run(wl, _dev_inputs(inp), flags=qb.FLAG_EPILOGUE_OFF)
    assert status == 0
    # exact projection: Y[t] = W[c1(t)] + W[c2(t)], integers with |y| <= 128 (exact in bf16)
    x2 = inp.x.reshape(wl.T, wl.hidden)
    y = _exact_projection(x2, inp.w)
    some = np.unique(np.linspace(0, wl.T - 1, 8).astype(int))
    assert np.array_equal(oracle.qkv_projection(x2[some], inp.w), y[some].astype(np.float64))
    bits = WL.f32_to_bf16_bits(y)
    assert np.array_equal(oracle.bf16_to_f64(bits), y.astype(np.float64))  # representable exactly
    del y
    O = bits.reshape(wl.T, 3, wl.num_heads, 128)
    ref = oracle.place_bands(O, wl.P, wl.B, wl.S, wl.num_heads, wl.layout)
    for g in ref:
        got = to_host_bits(out[g])
        assert np.array_equal(got, ref[g]), f"{wl.name}/{g}: placement differs"


@pytest.mark.parametrize("layout", ["bshd", "fused"])
def test_exact_placement_small(layout):
    _exact_placement(_wl("exact", P=4, B=2, S=96, H=8, layout=layout))


def test_capacity_and_empty_call():
    wl = _wl("cap", P=2, B=1, S=32, H=2)
    inp = WL.make_fused_inputs(wl)
    d = _dev_inputs(inp)
    plan = qb.Plan(wl.hidden, wl.num_heads, wl.P, "bshd", max_tokens=16)
    out = qb.alloc_outputs(plan, 1, 32)
    with pytest.raises(qb.QnreError) as e:
        qb.qnre_forward(plan, d["x"], d["w"], d["qw"], d["kw"], d["cs"], d["pos"], out)
    assert e.value.status == 5
    empty = d["x"][:, :, :0]
    for t in out.values():
        t.view(torch.int16).fill_(7)
    qb.qnre_forward(plan, empty, d["w"], d["qw"], d["kw"], d["cs"], None, out)
    torch.cuda.synchronize()
    for t in out.values():
        assert bool((t.view(torch.int16) == 7).all())


def test_output_alias_rejected():
    wl = _wl("alias", P=2, B=1, S=32, H=2)
    inp = WL.make_fused_inputs(wl)
    d = _dev_inputs(inp)
    plan = qb.Plan(wl.hidden, wl.num_heads, wl.P, "bshd", max_tokens=32)
    out = qb.alloc_outputs(plan, 1, 32)
    out["k"] = out["q"]
    with pytest.raises(qb.QnreError) as e:
        qb.qnre_forward(plan, d["x"], d["w"], d["qw"], d["kw"], d["cs"], d["pos"], out)
    assert e.value.status == 4


def test_side_stream_and_two_plans():
    wl1 = _wl("s1", P=2, B=1, S=128, H=4)
    wl2 = _wl("s2", P=4, B=1, S=64, H=8, layout="fused", rope="interleaved")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    res = []
    for wl in (wl1, wl2):
        inp = WL.make_fused_inputs(wl)
        d = _dev_inputs(inp)
        torch.cuda.synchronize()
        plan = qb.Plan(wl.hidden, wl.num_heads, wl.P, wl.layout, max_tokens=wl.B * wl.S, rope_style=wl.rope_style)
        out = qb.alloc_outputs(plan, wl.B, wl.S)
        with torch.cuda.stream(s):
            qb.qnre_forward(plan, d["x"], d["w"], d["qw"], d["kw"], d["cs"], d["pos"], out, stream=s)
        res.append((wl, inp, plan, out))
    s.synchronize()
    for wl, inp, plan, out in res:
        assert plan.device_status() == 0
        _full_compare(wl, inp, out)


# ---------------------------------------------------------------------------
# The full-size workloads: sampled values against the oracle, full coverage,
# and full bit-exact placement.
# ---------------------------------------------------------------------------
FULL = ["h4096_p4_s4096", "h7168_p4_s37888_fused", "h8192_p8_b2_s16384"]


@pytest.mark.slow
@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled_values(name):
    wl = WL.FUSED_WORKLOADS[name]
    inp = WL.make_fused_inputs(wl)
    _, out, status = _run(wl, _dev_inputs(inp))
    assert status == 0
    for t in out.values():  # every element rewritten (poisoned with NaN before)
        assert not bool(torch.isnan(t).any())
    tok = sample_tokens(wl.T, wl.S, n=640)
    assert len(tok) >= 512
    x2 = inp.x.reshape(wl.T, wl.hidden)
    O = oracle.project_norm_rope(x2[tok], inp.w, inp.q_norm_w, inp.k_norm_w, inp.cos_sin,
                                 inp.positions.reshape(-1)[tok], wl.num_heads, wl.rope_style)
    idx = torch.from_numpy(dest_index(tok, wl.P, wl.B, wl.S, wl.num_heads)).cuda()
    for gi, g in enumerate("qkv"):
        if wl.layout == "bshd":
            got = out[g][idx[0], idx[1], idx[2], idx[3]]
        else:
            got = out["fused"][idx[0], idx[1], idx[2], idx[3]][..., gi * 128:(gi + 1) * 128]
        assert_fused_close(to_host_f64(got), O[:, gi], what=f"{name}/{g}")


@pytest.mark.slow
@pytest.mark.parametrize("name", ["h7168_p4_s37888_fused", "h8192_p8_b2_s16384"])
def test_full_size_v_of_every_token(name):
    """v is the bare projection, so for a random z and every token t,
    sum_d v[t, h, d] z_d = x_t . (W_vh z) exactly up to v's rounding: this checks
    the v rows of three heads for every token of the full-size workload (the
    per-token sample above covers all heads of 640 tokens).  The bound is the
    per-element bar summed: |sum_d z_d e_d| <= sum_d |z_d| max(2 ulp(v_d), 2e-2)."""
    wl = WL.FUSED_WORKLOADS[name]
    inp = WL.make_fused_inputs(wl)
    _, out, status = _run(wl, _dev_inputs(inp))
    assert status == 0
    H, L, D, S, B, P = wl.num_heads, wl.H_local, 128, wl.S, wl.B, wl.P
    rng = np.random.default_rng(5)
    z = rng.standard_normal(D)
    heads = [0, H // 2 + 1, H - 1]
    w = inp.w
    U = np.stack([oracle.bf16_to_f64(w[:, (2 * H + h) * D:(2 * H + h + 1) * D]) @ z for h in heads], 1)   # [K, 3]
    x2 = inp.x.reshape(wl.T, wl.hidden)
    want = np.concatenate([oracle.bf16_to_f64(x2[i:i + 4096]) @ U for i in range(0, wl.T, 4096)])        # [T, 3]
    t = np.arange(wl.T)
    r_s, b, s = t // (B * S), (t // S) % B, t % S
    zg = torch.from_numpy(z).cuda()
    for j, h in enumerate(heads):
        r, hl = h // L, h % L
        band = out["v"][r, :, :, hl] if wl.layout == "bshd" else out["fused"][r, :, :, hl, 2 * D:]   # [B, S_g, D]
        vf = band.double()
        got = (vf @ zg).cpu().numpy()[b, r_s * S + s]                                                   # token order
        ulp = torch.exp2(torch.floor(torch.log2(vf.abs().clamp_min(2.0 ** -126))) - 7)
        tol = (zg.abs() * torch.maximum(2 * ulp, torch.full_like(ulp, 2e-2))).sum(-1).cpu().numpy()[b, r_s * S + s]
        err = np.abs(got - want[:, j])
        assert np.all(err <= tol), f"{name} head {h}: {np.sum(err > tol)} tokens beyond the bound, worst {err.max():.4g}"


@pytest.mark.slow
@pytest.mark.parametrize("name", ["h7168_p4_s37888_fused", "h8192_p8_b2_s16384"])
def test_full_size_qk_norms_of_every_token(name):
    """With unit norm weights RMSNorm leaves every q and k head row with mean square 1
    (less eps / (ms + eps)) and RoPE turns each pair without changing its norm, so
    every q and k row of every token has sum of squares 128 up to the bf16 rounding
    of its elements (at most 2^-8 relative each, so 2^-7 relative on each square
    and on the sum: |S - 128| <= 1, with 0.01 for eps and the fp32 arithmetic)."""
    wl = WL.FUSED_WORKLOADS[name]
    inp = WL.make_fused_inputs(wl)
    one = np.full(128, 0x3F80, np.uint16)                    # bf16 1.0
    inp = dataclasses.replace(inp, q_norm_w=one, k_norm_w=one)
    _, out, status = _run(wl, _dev_inputs(inp))
    assert status == 0
    for gi, g in enumerate("qk"):
        t = out[g] if wl.layout == "bshd" else out["fused"][..., gi * 128:(gi + 1) * 128]
        dev = (t.double().square().sum(-1) - 128.0).abs()    # [P, B, S_global, H_local]
        worst = dev.max().item()
        assert worst <= 1.01, f"{name}/{g}: {int((dev > 1.01).sum())} rows beyond the bound, worst {worst:.4g}"


@pytest.mark.slow
@pytest.mark.parametrize("name", FULL)
def test_full_size_exact_placement(name):
    _exact_placement(WL.FUSED_WORKLOADS[name])


def test_reserved_sms_give_identical_bits():
    """qnre_plan_reserve_sms changes only how many CTA pairs run the tiles: the output
    bits are the same for every setting, down to a single pair."""
    wl = _wl("reserve", P=4, B=1, S=1024, H=32)          # 768 pair tiles: many rounds, a short last round
    inp = WL.make_fused_inputs(wl)
    d = _dev_inputs(inp)
    plan = qb.Plan(wl.hidden, wl.num_heads, wl.P, wl.layout, max_tokens=wl.B * wl.S, rope_style=wl.rope_style)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    results = []
    for reserve in (0, 8, 16, 120, 0):                     # 120: 16 of the 76 pairs of a GB300 left
        plan.reserve_sms(reserve)
        out = qb.alloc_outputs(plan, wl.B, wl.S)
        for t in out.values():
            t.view(torch.int16).fill_(-1)
        qb.qnre_forward(plan, d["x"], d["w"], d["qw"], d["kw"], d["cs"], d["pos"], out)
        torch.cuda.synchronize()
        assert plan.device_status() == 0
        results.append({g: to_host_bits(t) for g, t in out.items()})
    for r in results[1:]:
        for g in r:
            assert np.array_equal(r[g], results[0][g]), g
    for bad in (-1, sms, 2 * sms):
        with pytest.raises(qb.QnreError) as e:
            plan.reserve_sms(bad)
        assert e.value.status == 1
    _full_compare(wl, inp, {g: to_dev_bf16(b) for g, b in results[0].items()})


@pytest.mark.parametrize("layout,rope", [("bshd", "interleaved"), ("fused", "rotate_half")])
def test_meets_the_pages_own_bar(layout, rope):
    """The pages' own acceptance test ("QKV projection + RMSNorm + RoPE overlapped
    with the Ulysses head exchange", Tests): against their fp32 step-by-step
    reference form, atol = rtol = 1e-2, with isolated 1-ulp bf16 flips classified;
    S_local = 200 is their tail row count."""
    import oracle.pages_mode as PM
    wl = _wl("pages_bar", P=2, B=1, S=200, H=8, layout=layout, rope=rope)
    inp = WL.make_fused_inputs(wl)
    _, out, status = _run(wl, _dev_inputs(inp))
    assert status == 0
    ref = PM.qnre_forward_pages_mode(inp.x, inp.w, inp.q_norm_w, inp.k_norm_w, inp.cos_sin, inp.positions,
                                     wl.P, wl.num_heads, wl.layout, wl.rope_style)
    exact = oracle.qnre_forward(inp.x, inp.w, inp.q_norm_w, inp.k_norm_w, inp.cos_sin, inp.positions,
                                wl.P, wl.num_heads, wl.layout, wl.rope_style)
    for g in ref:
        got, r = to_host_f64(out[g]), ref[g]
        ok = PM.pages_close(got, r)
        flips = ~ok & (np.abs(got - r) <= oracle.bf16_ulp(r))
        assert flips.mean() < 1e-3, f"{g}: {flips.sum()} one-ulp flips are not isolated"
        # The reference form rounds n and n*w to bf16 before RoPE, so where a pair's
        # rotation cancels it can sit a few hundredths from the exact result.  Past
        # the bar is allowed only there: where the kernel is the closer of the two
        # to the float64 oracle, and only at isolated elements.
        rest = ~(ok | flips)
        assert rest.mean() < 1e-4, f"{g}: {rest.sum()} elements beyond the pages' bar"
        closer = np.abs(got - exact[g]) < np.abs(r - exact[g])
        assert np.all(closer[rest]), f"{g}: beyond the bar where the reference form is the closer one"


@pytest.mark.parametrize("P,H,S,B,layout,rope", [
    (8, 24, 64, 1, "bshd", "interleaved"),    # hidden 3072 over 8 ranks: a band is 3 heads, pair tiles straddle bands
    (2, 48, 96, 2, "fused", "rotate_half"),   # hidden 6144 over 2 ranks
    (4, 64, 32, 1, "bshd", "rotate_half"),    # hidden 8192 over 4 ranks
    (8, 32, 48, 1, "fused", "interleaved"),   # hidden 4096 over 8 ranks
])
def test_pages_grid_shapes_sampled(P, H, S, B, layout, rope):
    """Shapes from the pages' measured grid (W in {2, 4, 8} x hidden in {3072, 4096,
    6144, 8192}, head_dim 128) at short sequences: sampled tokens against the oracle,
    every element written."""
    wl = _wl("grid", P=P, B=B, S=S, H=H, layout=layout, rope=rope)
    inp = WL.make_fused_inputs(wl)
    _, out, status = _run(wl, _dev_inputs(inp))
    assert status == 0
    for t in out.values():
        assert not bool(torch.isnan(t).any())
    tok = sample_tokens(wl.T, wl.S, n=96)
    x2 = inp.x.reshape(wl.T, wl.hidden)
    O = oracle.project_norm_rope(x2[tok], inp.w, inp.q_norm_w, inp.k_norm_w, inp.cos_sin,
                                 inp.positions.reshape(-1)[tok], wl.num_heads, wl.rope_style)
    idx = torch.from_numpy(dest_index(tok, wl.P, wl.B, wl.S, wl.num_heads)).cuda()
    for gi, g in enumerate("qkv"):
        if wl.layout == "bshd":
            got = out[g][idx[0], idx[1], idx[2], idx[3]]
        else:
            got = out["fused"][idx[0], idx[1], idx[2], idx[3]][..., gi * 128:(gi + 1) * 128]
        assert_fused_close(to_host_f64(got), O[:, gi], what=f"grid P{P} H{H}/{g}")


@pytest.mark.parametrize("S,B,H,P,layout,rope", [
    (300, 1, 4, 2, "bshd", "rotate_half"),     # 600 tokens = 3 row tiles: the second pair of the last cluster idles
    (200, 2, 8, 4, "fused", "interleaved"),    # 1600 tokens = 7 row tiles, 12 column tiles
    (1024, 1, 32, 4, "bshd", "rotate_half"),   # the benchmarked shape: 16 row tiles, 48 column tiles
])
def test_w_multicast_bit_identical(S, B, H, P, layout, rope):
    """Clusters of two CTA pairs sharing W through TMA multicast give the same bits as
    one pair per cluster, and the same readiness counts (the 1600-token case ends
    in a short round of half tiles)."""
    wl = _wl("mcast", P=P, B=B, S=S, H=H, layout=layout, rope=rope)
    inp = WL.make_fused_inputs(wl)
    d = _dev_inputs(inp)
    outs = []
    for flags in (qb.FLAG_ONE_PAIR, qb.FLAG_W_MULTICAST):
        plan = qb.Plan(wl.hidden, wl.num_heads, wl.P, wl.layout, max_tokens=wl.B * wl.S, rope_style=wl.rope_style,
                       flags=flags)
        out = qb.alloc_outputs(plan, wl.B, wl.S)
        for t in out.values():
            t.view(torch.int16).fill_(-1)
        ready = torch.zeros((wl.P,), dtype=torch.int32, device="cuda")
        qb.qnre_forward_publish(plan, d["x"], d["w"], d["qw"], d["kw"], d["cs"], d["pos"], out, ready)
        torch.cuda.synchronize()
        assert plan.device_status() == 0
        assert ready.cpu().tolist() == [qb.qnre_ready_target(plan, wl.B, wl.S)] * wl.P
        outs.append({g: to_host_bits(t) for g, t in out.items()})
    for g in outs[0]:
        assert np.array_equal(outs[1][g], outs[0][g]), g
    if wl.T <= 1600:
        _full_compare(wl, inp, {g: to_dev_bf16(b) for g, b in outs[1].items()})


def test_plan_describe_reports_the_form_that_runs():
    """qnre_plan_describe agrees with the launch rules: one pair per cluster for an
    odd handful of row tiles, two pairs sharing W for the benchmarked shape, the
    flags force either form, and reserved SMs shrink the grid."""
    tiny = WL.FUSED_WORKLOADS["tiny_p2_s64_h4"]
    plan = qb.Plan(tiny.hidden, tiny.num_heads, tiny.P, tiny.layout, max_tokens=tiny.B * tiny.S)
    d = plan.describe(tiny.B, tiny.S)
    assert d["pairs_per_cluster"] == 1 and d["row_tiles"] == 1 and d["col_tiles"] == 6
    assert d["half_items"] == d["work_items"] == 12                  # a small problem runs in halves
    assert plan.describe(0, 0)["clusters"] == 0
    with pytest.raises(qb.QnreError) as e:
        plan.describe(tiny.B, tiny.S + 1)
    assert e.value.status == 5
    wl = WL.FUSED_WORKLOADS["h4096_p4_s4096"]
    for flags, ppc in ((0, 2), (qb.FLAG_ONE_PAIR, 1), (qb.FLAG_W_MULTICAST, 2)):
        p = qb.Plan(wl.hidden, wl.num_heads, wl.P, wl.layout, max_tokens=wl.B * wl.S, flags=flags)
        d = p.describe(wl.B, wl.S)
        assert d["pairs_per_cluster"] == ppc and d["row_tiles"] == 16 and d["col_tiles"] == 48
        assert d["sms"] == d["clusters"] * 2 * ppc and d["launches"] == 1 and d["clusters"] >= 1
        full = d["work_items"] - d["half_items"]
        assert full + d["half_items"] // 2 == (768 if ppc == 1 else 384)   # every tile (or tile pair) once
        total = torch.cuda.get_device_properties(0).multi_processor_count
        p.reserve_sms(16)
        assert p.describe(wl.B, wl.S)["sms"] <= total - 16


def _plan_work(tiles, units):
    """The work list's split rule (whole tiles, and a short last round in halves)."""
    if 2 * tiles <= units:
        return 0, 2 * tiles
    rem = tiles % units
    if rem > 0 and 2 * rem <= units:
        return tiles - rem, tiles + rem
    return tiles, tiles


def _makespan_halves(full, work, units):
    loads = [0] * units
    for w in range(work):
        loads[w % units] += 2 if w < full else 1
    return max(loads)


@pytest.mark.parametrize("flags", [0, qb.FLAG_ONE_PAIR])
def test_fewest_clusters_for_the_same_makespan(flags):
    """A forward launches the fewest clusters that finish in as many rounds as one
    cluster fewer could not: for the 4096-token shape the last round would leave
    clusters idle, and those are not launched."""
    wl = WL.FUSED_WORKLOADS["h4096_p4_s4096"]
    p = qb.Plan(wl.hidden, wl.num_heads, wl.P, wl.layout, max_tokens=wl.B * wl.S, flags=flags)
    d = p.describe(wl.B, wl.S)
    c = d["clusters"]
    tiles = 384 if d["pairs_per_cluster"] == 2 else 768
    full, work = d["work_items"] - d["half_items"], d["work_items"]
    assert (full, work) == _plan_work(tiles, c) or c == work
    span = _makespan_halves(full, work, c)
    for fewer in range(1, c):
        f, w = _plan_work(tiles, fewer)
        assert _makespan_halves(f, w, min(w, fewer)) > span, fewer
    per_cluster = 2 * d["pairs_per_cluster"]
    sm_count = torch.cuda.get_device_properties(0).multi_processor_count
    assert c * per_cluster <= sm_count

