"""Pins for the CPU oracle: facts fixed by the pages and by mathematics, not by the oracle.

Each check below fails on a plausible mistake in one oracle step (a dropped
term, a wrong sign, a wrong index, a transposed operand); `test_pins_catch_*`
plants such mistakes in the oracle on the CPU and asserts that a pin fails.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle.qnre_oracle as Q
from ulysses_qkv_proj_gb300 import workloads as WL

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _bf16(vals):
    return WL.f32_to_bf16_bits(np.asarray(vals, dtype=np.float32))


def _rand_bf16(rng, shape, std=1.0):
    return WL.f32_to_bf16_bits(rng.standard_normal(shape).astype(np.float32) * np.float32(std))


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


# ----------------------------------------------------------------------------
# bf16 decoding: IEEE bf16 = the high 16 bits of a float32
# ----------------------------------------------------------------------------
def check_bf16_decode():
    bits = np.array([0x3F80, 0xC000, 0x3F81, 0x0000, 0x8000, 0x4049], dtype=np.uint16)
    want = [1.0, -2.0, 1.0 + 2.0 ** -7, 0.0, -0.0, 3.140625]
    assert Q.bf16_to_f64(bits).tolist() == want


def check_rne_rounding_of_generator():
    # 1 + 2^-8 is halfway between bf16 1.0 and 1.0078125: ties go to even (1.0);
    # 1 + 3*2^-8 is halfway between 1.0078125 and 1.015625: ties go to even (1.015625).
    bits = WL.f32_to_bf16_bits(np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -8 + 2 ** -20], np.float32))
    assert bits.tolist() == [0x3F80, 0x3F82, 0x3F81]


# ----------------------------------------------------------------------------
# Step 1: projection
# ----------------------------------------------------------------------------
def check_projection_one_hot():
    rng = np.random.default_rng(11)
    K, N, T = 6, 10, 4
    w = _rand_bf16(rng, (K, N))
    x = np.zeros((T, K), np.uint16)
    pick = [3, 0, 5, 3]
    for t, k in enumerate(pick):
        x[t, k] = 0x3F80  # 1.0
    y = Q.qkv_projection(x, w)
    assert y.shape == (T, N)
    assert np.array_equal(y, Q.bf16_to_f64(w)[pick])


def check_projection_brute_force():
    rng = np.random.default_rng(12)
    T, K, N = 3, 5, 4
    x = _rand_bf16(rng, (T, K))
    w = _rand_bf16(rng, (K, N))
    xf = [[float(np.float32(np.uint32(int(b) << 16).view(np.float32))) for b in row] for row in x]
    wf = [[float(np.float32(np.uint32(int(b) << 16).view(np.float32))) for b in row] for row in w]
    y = Q.qkv_projection(x, w)
    for t in range(T):
        for c in range(N):
            s = math.fsum(xf[t][k] * wf[k][c] for k in range(K))
            assert abs(y[t, c] - s) <= 1e-12 * max(1.0, abs(s))


def check_split_heads_column_order():
    H, D, T = 3, 4, 2
    y = np.tile(np.arange(3 * H * D, dtype=np.float64), (T, 1))
    s = Q.split_qkv_heads(y, H, head_dim=D)
    for g in range(3):
        for h in range(H):
            for d in range(D):
                assert s[1, g, h, d] == g * H * D + h * D + d


# ----------------------------------------------------------------------------
# Step 2: RMSNorm
# ----------------------------------------------------------------------------
def check_rms_norm_closed_forms():
    D = 128
    ones = _bf16(np.ones(D))
    # constant row a: n_d = a / sqrt(a^2 + eps)
    for a in (3.0, -0.5, 1e-3):
        n = Q.rms_norm(np.full((1, D), a), ones)
        assert np.allclose(n, a / math.sqrt(a * a + 1e-6), rtol=1e-14, atol=0)
    # eps sits inside the square root: a^2 = eps gives 1/sqrt(2)
    n = Q.rms_norm(np.full((1, D), 1e-3), ones)
    assert abs(n[0, 0] - 1 / math.sqrt(2)) < 1e-12
    # zero row stays zero
    assert np.all(Q.rms_norm(np.zeros((1, D)), ones) == 0)
    # the mean is over the head axis: one spike of size sqrt(D) has mean square 1
    y = np.zeros((1, D))
    y[0, 5] = math.sqrt(D)
    n = Q.rms_norm(y, ones)
    assert abs(n[0, 5] - math.sqrt(D) / math.sqrt(1 + 1e-6)) < 1e-12


def check_rms_norm_weight_indexing():
    D = 128
    rng = np.random.default_rng(13)
    y = rng.standard_normal((2, D))
    w = np.zeros(D, np.float32)
    w[7] = 2.0
    n = Q.rms_norm(y, _bf16(w))
    rinv = 1 / np.sqrt(np.mean(y * y, axis=-1) + 1e-6)
    assert np.all(n[:, np.arange(D) != 7] == 0)
    assert np.allclose(n[:, 7], y[:, 7] * rinv * 2.0, rtol=1e-14)


def check_rms_norm_invariant():
    rng = np.random.default_rng(14)
    D = 128
    y = rng.standard_normal((5, D)) * np.array([[0.01], [0.1], [1], [10], [100]])
    wv = (1 + 0.1 * rng.standard_normal(D)).astype(np.float32)
    wb = _bf16(wv)
    n = Q.rms_norm(y, wb)
    ms = np.mean(y * y, axis=-1)
    rms = np.sqrt(np.mean((n / Q.bf16_to_f64(wb)) ** 2, axis=-1))
    assert np.allclose(rms, np.sqrt(ms / (ms + 1e-6)), rtol=1e-12)


# ----------------------------------------------------------------------------
# Step 3: RoPE
# ----------------------------------------------------------------------------
def _cs_row(angles):
    a = np.asarray(angles, np.float64)
    return np.concatenate([np.cos(a), np.sin(a)])[None, :]


def check_rope_identity_at_zero():
    rng = np.random.default_rng(15)
    n = rng.standard_normal((1, 3, 128))
    cs = _cs_row(np.zeros(64))
    for style in ("rotate_half", "interleaved"):
        assert np.array_equal(Q.apply_rope(n, cs, style), n)


def check_rope_rotate_half_unit_vectors():
    ang = 0.3 + 0.05 * np.arange(64)
    cs = _cs_row(ang)
    for i in (0, 17, 63):
        e = np.zeros((1, 1, 128))
        e[0, 0, i] = 1
        o = Q.apply_rope(e, cs, "rotate_half")[0, 0]
        want = np.zeros(128)
        want[i], want[i + 64] = math.cos(ang[i]), math.sin(ang[i])
        assert np.allclose(o, want, atol=1e-15)
        e = np.zeros((1, 1, 128))
        e[0, 0, i + 64] = 1
        o = Q.apply_rope(e, cs, "rotate_half")[0, 0]
        want = np.zeros(128)
        want[i], want[i + 64] = -math.sin(ang[i]), math.cos(ang[i])
        assert np.allclose(o, want, atol=1e-15)


def check_rope_interleaved_unit_vectors():
    ang = 0.2 + 0.07 * np.arange(64)
    cs = _cs_row(ang)
    for i in (0, 9, 63):
        e = np.zeros((1, 1, 128))
        e[0, 0, 2 * i] = 1
        o = Q.apply_rope(e, cs, "interleaved")[0, 0]
        want = np.zeros(128)
        want[2 * i], want[2 * i + 1] = math.cos(ang[i]), math.sin(ang[i])
        assert np.allclose(o, want, atol=1e-15)
        e = np.zeros((1, 1, 128))
        e[0, 0, 2 * i + 1] = 1
        o = Q.apply_rope(e, cs, "interleaved")[0, 0]
        want = np.zeros(128)
        want[2 * i], want[2 * i + 1] = -math.sin(ang[i]), math.cos(ang[i])
        assert np.allclose(o, want, atol=1e-15)


def check_rope_norm_and_composition():
    rng = np.random.default_rng(16)
    tab = WL.rope_table(64).astype(np.float64)
    n = rng.standard_normal((1, 2, 128))
    for style, pairs in (("rotate_half", [(i, i + 64) for i in range(64)]),
                         ("interleaved", [(2 * i, 2 * i + 1) for i in range(64)])):
        o = Q.apply_rope(n, tab[[23]], style)
        for i, (a, b) in enumerate(pairs):
            c, s = tab[23, i], tab[23, 64 + i]
            lhs = o[..., a] ** 2 + o[..., b] ** 2
            rhs = (n[..., a] ** 2 + n[..., b] ** 2) * (c * c + s * s)
            assert abs(lhs - rhs).max() < 1e-12
        # rotating by position 7 then 16 equals rotating by position 23 (fp32 table error only)
        o2 = Q.apply_rope(Q.apply_rope(n, tab[[7]], style), tab[[16]], style)
        assert np.abs(o2 - o).max() < 1e-4


def check_rope_table():
    tab = WL.rope_table(3)
    assert tab.dtype == np.float32 and tab.shape == (3, 128)
    assert np.all(tab[0, :64] == 1) and np.all(tab[0, 64:] == 0)
    assert tab[1, 0] == np.float32(math.cos(1.0)) and tab[1, 64] == np.float32(math.sin(1.0))
    f1 = 1e4 ** (-2.0 / 128)
    assert tab[2, 1] == np.float32(math.cos(2 * f1)) and tab[2, 65] == np.float32(math.sin(2 * f1))
    f63 = 1e4 ** (-126.0 / 128)
    assert tab[1, 63] == np.float32(math.cos(f63))


# ----------------------------------------------------------------------------
# Steps 1-3 together: brute force on a tiny problem with the math module only
# ----------------------------------------------------------------------------
def _f(b):
    return float(np.uint32(int(b) << 16).view(np.float32))


def _brute_token(x_row, w, qw, kw, cs_row, H, style):
    D = 128
    K = len(x_row)
    y = [[[math.fsum(_f(x_row[k]) * _f(w[k][g * H * D + h * D + d]) for k in range(K))
           for d in range(D)] for h in range(H)] for g in range(3)]
    out = [[None] * H for _ in range(3)]
    for g in range(3):
        for h in range(H):
            v = y[g][h]
            if g == 2:
                out[g][h] = v
                continue
            wt = qw if g == 0 else kw
            ms = math.fsum(a * a for a in v) / D
            r = 1.0 / math.sqrt(ms + 1e-6)
            nv = [v[d] * r * _f(wt[d]) for d in range(D)]
            o = [0.0] * D
            for i in range(64):
                c, s = float(cs_row[i]), float(cs_row[64 + i])
                a_i, b_i = (i, i + 64) if style == "rotate_half" else (2 * i, 2 * i + 1)
                o[a_i] = nv[a_i] * c - nv[b_i] * s
                o[b_i] = nv[b_i] * c + nv[a_i] * s
            out[g][h] = o
    return np.array(out)


@pytest.mark.parametrize("style", ["rotate_half", "interleaved"])
def test_project_norm_rope_brute_force(style):
    rng = np.random.default_rng(17)
    H, K = 2, 64
    x = _rand_bf16(rng, (3, K))
    w = _rand_bf16(rng, (K, 3 * H * 128), std=0.125)
    qw = _bf16(1 + 0.1 * rng.standard_normal(128))
    kw = _bf16(1 + 0.1 * rng.standard_normal(128))
    tab = WL.rope_table(40)
    pos = np.array([0, 37, 5])
    O = Q.project_norm_rope(x, w, qw, kw, tab, pos, H, style)
    for t in range(3):
        want = _brute_token(x[t], w, qw, kw, tab[pos[t]], H, style)
        assert np.allclose(O[t], want, rtol=1e-10, atol=1e-12)


def test_v_is_bare_projection_and_bad_position_is_nan():
    rng = np.random.default_rng(18)
    H, K = 2, 256
    x = _rand_bf16(rng, (4, K))
    w = _rand_bf16(rng, (K, 3 * H * 128), std=1 / 16)
    qw = kw = _bf16(np.ones(128))
    tab = WL.rope_table(8)
    O = Q.project_norm_rope(x, w, qw, kw, tab, np.array([1, 8, -1, 7]), H)
    y = Q.qkv_projection(x, w).reshape(4, 3, H, 128)
    assert np.array_equal(O[:, 2], y[:, 2])
    assert np.isnan(O[1, :2]).all() and np.isnan(O[2, :2]).all()
    assert not np.isnan(O[[0, 3]]).any() and not np.isnan(O[:, 2]).any()


# ----------------------------------------------------------------------------
# Step 4: placement
# ----------------------------------------------------------------------------
def check_placement_golden(golden_dir):
    g = _load(golden_dir, "placement_p2_b2_s3_h4.json")
    P, B, S, H = g["P"], g["B"], g["S"], g["H"]
    T, D = P * B * S, 4
    O = np.zeros((T, 3, H, D))
    for t in range(T):
        for gi in range(3):
            for h in range(H):
                O[t, gi, h, :] = 1000 * t + 100 * gi + 10 * h + np.arange(D)
    out = Q.place_bands(O, P, B, S, H, "bshd")
    fused = Q.place_bands(O, P, B, S, H, "fused")["fused"]
    for case in g["cases"]:
        t, h = case["t"], case["h"]
        assert list(Q.token_coords(t, P, B, S)) == case["coords"]
        r_s, b, s = case["coords"]
        assert list(Q.band_destination(r_s, b, s, h, P, B, S, H)) == case["dest"]
        r, bb, row, hl = case["dest"]
        for gi, name in enumerate("qkv"):
            assert np.array_equal(out[name][r, bb, row, hl], O[t, gi, h])
            assert np.array_equal(fused[r, bb, row, hl, gi * D:(gi + 1) * D], O[t, gi, h])


def check_placement_p1_and_coverage():
    rng = np.random.default_rng(19)
    B, S, H, D = 2, 5, 3, 4
    O = rng.standard_normal((B * S, 3, H, D))
    out = Q.place_bands(O, 1, B, S, H, "bshd")
    for gi, name in enumerate("qkv"):
        assert np.array_equal(out[name][0], O[:, gi].reshape(B, S, H, D))
    P, B, S, H = 4, 2, 3, 8
    O = rng.standard_normal((P * B * S, 3, H, D))
    for layout in ("bshd", "fused"):
        res = Q.place_bands(O, P, B, S, H, layout)
        total = sum(a.size for a in res.values())
        assert total == O.size and not any(np.isnan(a).any() for a in res.values())
        vals = np.sort(np.concatenate([a.ravel() for a in res.values()]))
        assert np.array_equal(vals, np.sort(O.ravel()))


def check_placement_matches_scatter_heads():
    rng = np.random.default_rng(20)
    P, B, S, H, D = 2, 2, 3, 4, 4
    O = rng.standard_normal((P * B * S, 3, H, D))
    out = Q.place_bands(O, P, B, S, H, "bshd")
    for gi, name in enumerate("qkv"):
        assert np.array_equal(out[name], Q.scatter_heads(O[:, gi].reshape(P, B, S, H, D)))


def check_scatter_gather():
    rng = np.random.default_rng(21)
    x = rng.standard_normal((1, 2, 3, 4, 2))
    assert np.array_equal(Q.scatter_heads(x), x)  # world_size 1 is the identity
    x = rng.standard_normal((3, 2, 4, 6, 2))
    assert np.array_equal(Q.gather_heads(Q.scatter_heads(x)), x)


# ----------------------------------------------------------------------------
# Head-chunk pack / merge
# ----------------------------------------------------------------------------
def check_pack_golden(golden_dir):
    g = _load(golden_dir, "pack_w2_h4_d2.json")
    B, S, H, D = g["B"], g["S"], g["H"], g["D"]
    b, s, h, d = np.meshgrid(np.arange(B), np.arange(S), np.arange(H), np.arange(D), indexing="ij")
    q = 100 * h + 10 * s + d
    out = Q.pack_head_chunk(q, q + 1000, q + 2000, g["world_size"], g["head_offset"], g["head_count"])
    assert out.tolist() == g["expected"]


def check_merge_golden(golden_dir):
    g = _load(golden_dir, "merge_w2_l2_d2.json")
    B, S, D, W, L = g["B"], g["S"], g["D"], g["world_size"], g["local_heads"]
    b, s, slot, d = np.meshgrid(np.arange(B), np.arange(S), np.arange(W), np.arange(D), indexing="ij")
    rec = 100 * s + 10 * slot + d
    out = np.full((B, S, W * L, D), g["fill"])
    res = Q.merge_output_head_chunk(rec, W, L, g["head_offset"], out)
    assert res.tolist() == g["expected"]
    assert np.all(out == g["fill"])  # the input destination is not modified in place


def check_pack_merge_schedules(golden_dir):
    g = _load(golden_dir, "schedules.json")
    rng = np.random.default_rng(22)
    for sch in g["schedules"]:
        L = sch["local_heads"]
        covered = sorted(h for off, cnt in sch["bands"] for h in range(off, off + cnt))
        assert covered == list(range(L))
        W, B, S, D = 2, 2, 3, 4
        q, k, v = (rng.integers(0, 1 << 16, size=(B, S, W * L, D)).astype(np.uint16) for _ in range(3))
        outs = {c: np.zeros_like(q) for c in "qkv"}
        for off, cnt in sch["bands"]:
            pk = Q.pack_head_chunk(q, k, v, W, off, cnt)
            assert pk.shape == (B, S, W * cnt, 3 * D)
            for ci, c in enumerate("qkv"):
                outs[c] = Q.merge_output_head_chunk(pk[..., ci * D:(ci + 1) * D], W, L, off, outs[c])
        for c, X in zip("qkv", (q, k, v)):
            assert np.array_equal(outs[c], X)


def check_sequence_chunk_golden(golden_dir):
    g = _load(golden_dir, "seqchunk_w2_s4.json")
    B, S_g, cnt, D, W = g["B"], g["S_global"], g["head_count"], g["D"], g["world_size"]
    b, s, j, d = np.meshgrid(np.arange(B), np.arange(S_g), np.arange(cnt), np.arange(D), indexing="ij")
    x = 100 * s + 10 * j + d
    assert Q.pack_output_sequence_chunk(x, W).tolist() == g["expected"]


def check_all_to_all():
    sent = [[(r, r2) for r2 in range(3)] for r in range(3)]
    rec = Q.all_to_all(sent)
    for r2 in range(3):
        assert rec[r2] == [(r, r2) for r in range(3)]  # slot r on rank r2 holds rank r's chunk for r2


def check_head_chunk_exchanges_reconstruct_ordinary(golden_dir):
    """Every band of a complete schedule through the head-chunk exchanges rebuilds the
    ordinary scatter_heads / gather_heads results (the pages' reconstruction statements)."""
    g = _load(golden_dir, "schedules.json")
    rng = np.random.default_rng(23)
    for sch in g["schedules"][:2]:
        L = sch["local_heads"]
        P, B, S, D = 2, 2, 3, 4
        H = P * L
        q, k, v = (rng.integers(0, 1 << 16, size=(P, B, S, H, D)).astype(np.uint16) for _ in range(3))
        full = {c: Q.scatter_heads(X) for c, X in zip("qkv", (q, k, v))}   # [P, B, P*S, L, D]
        for off, cnt in sch["bands"]:
            res = Q.scatter_qkv_head_chunk(list(q), list(k), list(v), off, cnt)
            for r2 in range(P):
                assert res[r2].shape == (B, P * S, cnt, 3 * D)
                for ci, c in enumerate("qkv"):
                    assert np.array_equal(res[r2][..., ci * D:(ci + 1) * D], full[c][r2][:, :, off:off + cnt])
        # output side: attention output bands [P, B, P*S, L, D] back to [P, B, S, H, D]
        o = rng.integers(0, 1 << 16, size=(P, B, P * S, L, D)).astype(np.uint16)
        outs = [np.zeros((B, S, H, D), np.uint16) for _ in range(P)]
        for off, cnt in sch["bands"]:
            outs = Q.gather_output_head_chunk([o[r][:, :, off:off + cnt] for r in range(P)], L, off, outs)
        assert np.array_equal(np.stack(outs), Q.gather_heads(o))


def check_tolerance_rule():
    assert Q.bf16_ulp(np.array([1.0, 1.5, 3.0, -0.25]))[:].tolist() == [2 ** -7, 2 ** -7, 2 ** -6, 2 ** -9]
    tol = Q.fused_tolerance(np.array([0.5, 4.0, 100.0]))
    assert tol.tolist() == [2e-2, 2 * 2 ** -5, 2 * 2 ** -1]


# ----------------------------------------------------------------------------
# Tests
# ----------------------------------------------------------------------------
PLAIN_CHECKS = [
    check_bf16_decode, check_rne_rounding_of_generator, check_projection_one_hot,
    check_projection_brute_force, check_split_heads_column_order, check_rms_norm_closed_forms,
    check_rms_norm_weight_indexing, check_rms_norm_invariant, check_rope_identity_at_zero,
    check_rope_rotate_half_unit_vectors, check_rope_interleaved_unit_vectors,
    check_rope_norm_and_composition, check_rope_table, check_placement_p1_and_coverage,
    check_placement_matches_scatter_heads, check_scatter_gather, check_tolerance_rule,
    check_all_to_all,
]
GOLDEN_CHECKS = [check_placement_golden, check_pack_golden, check_merge_golden, check_pack_merge_schedules,
                 check_sequence_chunk_golden, check_head_chunk_exchanges_reconstruct_ordinary]


@pytest.mark.parametrize("check", PLAIN_CHECKS, ids=lambda f: f.__name__)
def test_pin(check):
    check()


@pytest.mark.parametrize("check", GOLDEN_CHECKS, ids=lambda f: f.__name__)
def test_golden_pin(check, golden_dir):
    check(golden_dir)


def test_oracle_forward_tiny_matches_step_by_step():
    """The composed forward equals placement of the per-token brute-force result."""
    wl = WL.FUSED_WORKLOADS["tiny_p2_s64_h4"]
    inp = WL.make_fused_inputs(wl)
    out = Q.qnre_forward(inp.x, inp.w, inp.q_norm_w, inp.k_norm_w, inp.cos_sin, inp.positions,
                         wl.P, wl.num_heads, "bshd")
    x2 = inp.x.reshape(wl.T, wl.hidden)
    for t in (0, 63, 64, 127):
        want = _brute_token(x2[t], inp.w, inp.q_norm_w, inp.k_norm_w,
                            inp.cos_sin[inp.positions.reshape(-1)[t]], wl.num_heads, "rotate_half")
        r_s, b, s = Q.token_coords(t, wl.P, wl.B, wl.S)
        for h in range(wl.num_heads):
            r, bb, row, hl = Q.band_destination(r_s, b, s, h, wl.P, wl.B, wl.S, wl.num_heads)
            for gi, g in enumerate("qkv"):
                assert np.allclose(out[g][r, bb, row, hl], want[gi, h], rtol=1e-10, atol=1e-12)


# ----------------------------------------------------------------------------
# Planted mistakes: every one of them must trip at least one pin
# ----------------------------------------------------------------------------
def _mut_projection_transposed(x_bits, w_bits):
    x = Q.bf16_to_f64(x_bits)
    w = Q.bf16_to_f64(w_bits)
    return x @ w.reshape(w.shape[1], w.shape[0]).T


def _mut_rms_no_eps(y, weight_bits, eps=Q.RMS_EPS):
    return y / np.sqrt(np.mean(y * y, axis=-1, keepdims=True)) * Q.bf16_to_f64(weight_bits)


def _mut_rms_sum_not_mean(y, weight_bits, eps=Q.RMS_EPS):
    return y / np.sqrt(np.sum(y * y, axis=-1, keepdims=True) + eps) * Q.bf16_to_f64(weight_bits)


def _mut_rms_eps_outside(y, weight_bits, eps=Q.RMS_EPS):
    return y / (np.sqrt(np.mean(y * y, axis=-1, keepdims=True)) + eps) * Q.bf16_to_f64(weight_bits)


def _mut_rms_weight_reversed(y, weight_bits, eps=Q.RMS_EPS):
    ms = np.mean(y * y, axis=-1, keepdims=True)
    return y / np.sqrt(ms + eps) * Q.bf16_to_f64(weight_bits)[::-1]


def _mut_rope_sign(n, cos, sin):
    half = n.shape[-1] // 2
    a, b = n[..., :half], n[..., half:]
    return np.concatenate([a * cos + b * sin, b * cos - a * sin], axis=-1)


def _mut_rope_dropped_term(n, cos, sin):
    half = n.shape[-1] // 2
    a, b = n[..., :half], n[..., half:]
    return np.concatenate([a * cos - b * sin, b * cos], axis=-1)


def _mut_interleaved_swapped(n, cos, sin):
    a, b = n[..., 0::2], n[..., 1::2]
    out = np.empty_like(n)
    out[..., 0::2] = a * cos - b * sin
    out[..., 1::2] = a * cos + b * sin
    return out


def _mut_place_swapped_ranks(O, P, B, S, num_heads, layout):
    res = Q.__dict__["_orig_place_bands"](O, P, B, S, num_heads, layout)
    return {k: v[::-1].copy() for k, v in res.items()}


def _mut_pack_wrong_head(q, k, v, world_size, head_offset, head_count):
    B, S, H, D = q.shape
    out = np.empty((B, S, world_size * head_count, 3 * D), dtype=q.dtype)
    for r in range(world_size):
        for j in range(head_count):
            h = r * head_count + head_offset + j
            for c, X in enumerate((q, k, v)):
                out[:, :, r * head_count + j, c * D:(c + 1) * D] = X[:, :, h, :]
    return out


def _mut_merge_wrong_slot(received, world_size, local_heads, head_offset, out):
    B, S, WC, D = received.shape
    cnt = WC // world_size
    res = out.copy()
    for r in range(world_size):
        for j in range(cnt):
            res[:, :, r * local_heads + head_offset + j, :] = received[:, :, j * world_size + r, :]
    return res


def _mut_split_heads_swapped(y, num_heads, head_dim=Q.HEAD_DIM):
    return y.reshape(y.shape[0], num_heads, 3, head_dim).transpose(0, 2, 1, 3)


def _mut_bf16_decode(bits):
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 15).view(np.float32).astype(np.float64)


def _mut_seqchunk_wrong_rows(x, world_size):
    B, S_g, cnt, D = x.shape
    S = S_g // world_size
    out = np.empty((world_size, B, S, cnt, D), dtype=x.dtype)
    for r in range(world_size):
        out[r] = x[:, r::world_size][:, :S]
    return out


def _mut_all_to_all_identity(sent):
    return [list(row) for row in sent]


def _mut_scatter_heads_swapped(x):
    P, B, S, H, D = x.shape
    H_local = H // P
    out = np.empty((P, B, P * S, H_local, D), dtype=x.dtype)
    for r in range(P):
        for r_s in range(P):
            out[r, :, r_s * S:(r_s + 1) * S] = x[r, :, :, r_s * H_local:(r_s + 1) * H_local]
    return out


def _mut_scatter_qkv_reversed_sources(q_ranks, k_ranks, v_ranks, head_offset, head_count):
    # the received blocks stacked in reverse source-rank order along the sequence
    P = len(q_ranks)
    packed = [Q.pack_head_chunk(q_ranks[r], k_ranks[r], v_ranks[r], P, head_offset, head_count) for r in range(P)]
    sent = [[packed[r][:, :, r2 * head_count:(r2 + 1) * head_count, :] for r2 in range(P)] for r in range(P)]
    received = Q.all_to_all(sent)
    return [np.concatenate(received[r2][::-1], axis=1) for r2 in range(P)]


def _mut_gather_output_slot_order(x_ranks, local_heads, head_offset, out_ranks):
    # received slots read head-major (j * P + src) instead of source-major
    P = len(x_ranks)
    staged = [Q.pack_output_sequence_chunk(x, P) for x in x_ranks]
    received = Q.all_to_all([[staged[r][r2] for r2 in range(P)] for r in range(P)])
    res = []
    for r2 in range(P):
        band = np.stack(received[r2], axis=0)
        _, B, S, cnt, D = band.shape
        rec = band.transpose(1, 2, 3, 0, 4).reshape(B, S, P * cnt, D)
        res.append(Q.merge_output_head_chunk(rec, P, local_heads, head_offset, out_ranks[r2]))
    return res


MUTANTS = [
    ("qkv_projection", _mut_projection_transposed),
    ("rms_norm", _mut_rms_no_eps),
    ("rms_norm", _mut_rms_sum_not_mean),
    ("rms_norm", _mut_rms_eps_outside),
    ("rms_norm", _mut_rms_weight_reversed),
    ("rope_rotate_half", _mut_rope_sign),
    ("rope_rotate_half", _mut_rope_dropped_term),
    ("rope_interleaved", _mut_interleaved_swapped),
    ("place_bands", _mut_place_swapped_ranks),
    ("pack_head_chunk", _mut_pack_wrong_head),
    ("merge_output_head_chunk", _mut_merge_wrong_slot),
    ("split_qkv_heads", _mut_split_heads_swapped),
    ("bf16_to_f64", _mut_bf16_decode),
    ("pack_output_sequence_chunk", _mut_seqchunk_wrong_rows),
    ("all_to_all", _mut_all_to_all_identity),
    ("scatter_heads", _mut_scatter_heads_swapped),
    ("scatter_qkv_head_chunk", _mut_scatter_qkv_reversed_sources),
    ("gather_output_head_chunk", _mut_gather_output_slot_order),
]


@pytest.mark.parametrize("name,mutant", MUTANTS, ids=[m[1].__name__ for m in MUTANTS])
def test_pins_catch_planted_mistake(name, mutant, monkeypatch, golden_dir):
    monkeypatch.setitem(Q.__dict__, "_orig_place_bands", Q.place_bands)
    monkeypatch.setattr(Q, name, mutant)
    tripped = []
    for check in PLAIN_CHECKS:
        try:
            check()
        except (AssertionError, ValueError, IndexError):
            tripped.append(check.__name__)
    for check in GOLDEN_CHECKS:
        try:
            check(golden_dir)
        except (AssertionError, ValueError, IndexError):
            tripped.append(check.__name__)
    for style in ("rotate_half", "interleaved"):
        try:
            test_project_norm_rope_brute_force(style)
        except (AssertionError, ValueError, IndexError):
            tripped.append("brute_force_" + style)
    assert tripped, f"no pin caught the planted mistake in {name}"
