"""Pins for the Sage2 oracle: the E4M3 and INT8 encoders against the formats' definitions,
the fixed-order K statistics against exact sums, and the encoding against invariants that
any correct grouped quantiser satisfies.  Planted mistakes must trip a pin."""
import json
import os

import numpy as np
import pytest

import oracle
import oracle.sage2_oracle as S2
from ulysses_qkv_proj_gb300 import workloads as WL


def _bf16(a):
    return WL.f32_to_bf16_bits(np.asarray(a, np.float32))


def _f(bits):
    return oracle.bf16_to_f64(bits)


def check_e4m3_fixture(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "e4m3_values.json")))
    for c in g["cases"]:
        code = int(c["code"], 16)
        assert S2.e4m3_decode(np.array([code]))[0] == c["value"]
        assert int(S2.e4m3_encode(np.array([c["value"]]))[0]) == code


def check_e4m3_rounding():
    codes = np.arange(256, dtype=np.uint8)
    vals = S2.e4m3_decode(codes)
    fin = ~np.isnan(vals)
    assert np.array_equal(S2.e4m3_encode(vals[fin]), codes[fin])        # every finite code round-trips
    assert np.isnan(vals[0x7F]) and np.isnan(vals[0xFF])
    enc = lambda v: int(S2.e4m3_encode(np.array([v]))[0])              # noqa: E731
    assert enc(1.0625) == 0x38 and enc(1.1875) == 0x3A                  # ties go to the even code
    assert enc(1.07) == 0x39 and enc(1.05) == 0x38                      # otherwise the nearest
    assert enc(2 ** -10) == 0x00 and enc(3 * 2 ** -10) == 0x02          # subnormal ties to even
    assert enc(500.0) == 0x7E and enc(-1e6) == 0xFE                     # saturation
    assert enc(-1e-9) == 0x80                                           # sign kept when rounding to zero


def _e4m3_brute_force(x):
    """Nearest of all 127 finite magnitudes by exhaustive comparison (ties to the even code)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), 448.0)
    mags = S2.e4m3_decode(np.arange(127, dtype=np.uint8))
    out = []
    for ai, xi in zip(a.ravel(), x.ravel()):
        d = np.abs(ai - mags)
        best = np.flatnonzero(d == d.min())
        even = [c for c in best if c % 2 == 0]
        c = even[0] if even else best[0]
        out.append(c | (0x80 if np.signbit(xi) else 0))
    return np.array(out, dtype=np.uint8).reshape(x.shape)


def check_e4m3_matches_brute_force():
    rng = np.random.default_rng(33)
    mags = S2.e4m3_decode(np.arange(127, dtype=np.uint8))
    mids = (mags[:-1] + mags[1:]) / 2                     # every tie point
    x = np.concatenate([mids, -mids, rng.standard_normal(3000) * 50, rng.uniform(-500, 500, 1000),
                        rng.standard_normal(500) * 0.01, [0.0, -0.0, 448.0, 1e9, -1e9]])
    assert np.array_equal(S2.e4m3_encode(x), _e4m3_brute_force(x))


def check_int8_quantize():
    q = S2.int8_quantize(np.array([2.5, 3.5, -2.5, -3.5, 0.49, 300.0, -300.0], np.float32), np.float32(1))
    assert q.tolist() == [2, 4, -2, -4, 0, 127, -128]
    assert S2.int8_quantize(np.array([5.0], np.float32), np.float32(0)).tolist() == [0]
    # the product is formed in float32 before rounding
    x, inv = np.float32(0.1), np.float32(35.0)
    assert S2.int8_quantize(np.array([x]), inv).tolist() == [int(np.rint(np.float32(x * inv)))]
    assert S2.reciprocal(np.array([2.0, 0.0], np.float32), np.float32(127)).tolist() == [63.5, 0.0]
    assert S2.reciprocal(np.array([3.0], np.float32), np.float32(448)).dtype == np.float32


def check_k_sum_exact_and_ordered():
    rng = np.random.default_rng(31)
    P, B, L, H, D = 2, 1, 300, 2, 4
    ints = rng.integers(-50, 51, size=(P, B, L, H, D)).astype(np.float32)   # sums of small integers are exact
    ks = [_bf16(ints[r]) for r in range(P)]
    assert np.array_equal(S2.sage2_k_sum(ks), ints.sum(axis=(0, 2)))
    vals = (rng.standard_normal((P, B, L, H, D)) * 3).astype(np.float32)
    ks = [_bf16(vals[r]) for r in range(P)]
    exact = np.stack([_f(k) for k in ks]).sum(axis=(0, 2))
    got = S2.sage2_k_sum(ks).astype(np.float64)
    assert np.abs(got - exact).max() < 1e-4 * np.abs(exact).max() + 1e-3


def _inputs(P=2, B=2, L=70, H=4, D=8, seed=32, smooth=None):
    rng = np.random.default_rng(seed)
    q = [_bf16(rng.standard_normal((B, L, H, D)) * (1 + r)) for r in range(P)]
    base = rng.standard_normal((B, L, H, D)) if smooth is None else smooth
    k = [_bf16(base + 3.0 + 0.5 * r) for r in range(P)]
    v = [_bf16(rng.standard_normal((B, L, H, D)) * 2) for r in range(P)]
    return q, k, v


def check_sage2_structure_and_bounds():
    P, B, L, H, D = 2, 2, 70, 4, 8
    q, k, v = _inputs(P, B, L, H, D)
    S, H_l = P * L, H // P
    for U in (S, 101):
        res = S2.sage2_scatter_qkv(q, k, v, U)
        wq, wk = -(-U // 32), -(-U // 64)
        Sp = -(-S // 64) * 64
        ex_q = oracle.scatter_heads(np.stack(q))   # [P, B, S, H_l, D] bf16 bits, pinned elsewhere
        ex_k = oracle.scatter_heads(np.stack(k))
        ex_v = oracle.scatter_heads(np.stack(v))
        kmean = (S2.sage2_k_sum(k) / np.float32(U)).astype(np.float32)
        for r in range(P):
            o = res[r]
            assert o["q"].shape == (B, S, H_l, D) and o["k"].shape == (B, S, H_l, D)
            assert o["v"].shape == (B, D, H_l, Sp) and o["v_scale"].shape == (B, H_l, D)
            assert o["q_scale"].shape == (B, H_l, wq) and o["k_scale"].shape == (B, H_l, wk)
            qf = _f(ex_q[r]).astype(np.float32)
            ks = (_f(ex_k[r]).astype(np.float32) - kmean[:, None, r * H_l:(r + 1) * H_l]).astype(np.float32)
            vf = _f(ex_v[r])
            for g in range(wq):
                rows = slice(32 * g, min(U, 32 * g + 32))
                sc = o["q_scale"][:, :, g]
                assert np.allclose(sc, np.abs(qf[:, rows]).max(axis=(1, 3)) / 127, rtol=1e-6)
                deq = o["q"][:, rows].astype(np.float64) * sc[:, None, :, None]
                assert np.all(np.abs(deq - qf[:, rows]) <= 0.5 * sc[:, None, :, None] * (1 + 1e-5))
                assert np.all(np.abs(o["q"][:, rows]).max(axis=(1, 3)) == 127)   # the group max hits the top code
            for g in range(wk):
                rows = slice(64 * g, min(U, 64 * g + 64))
                sc = o["k_scale"][:, :, g]
                deq = o["k"][:, rows].astype(np.float64) * sc[:, None, :, None]
                assert np.all(np.abs(deq - ks[:, rows]) <= 0.5 * sc[:, None, :, None] * (1 + 1e-5))
            assert not o["q"][:, U:].any() and not o["k"][:, U:].any()       # rows past the used prefix
            assert not o["v"][..., U:].any()
            vmax = np.abs(vf[:, :U]).max(axis=1)                                # [B, H_l, D]
            assert np.allclose(o["v_scale"], vmax / 448, rtol=1e-6)
            top = np.abs(S2.e4m3_decode(o["v"][..., :U])).max(axis=-1)          # [B, D, H_l]
            assert np.allclose(top, 448.0)
            deqv = S2.e4m3_decode(o["v"][..., :U]).transpose(0, 3, 2, 1) * o["v_scale"][:, None]
            assert np.all(np.abs(deqv - vf[:, :U]) <= np.abs(vf[:, :U]) / 16 + o["v_scale"][:, None] * 2 ** -9)


def check_sage2_smoothing_removes_channel_offset():
    """K smoothing: tokens that differ only by a per-channel constant encode as all zeros."""
    P, B, L, H, D = 2, 1, 40, 2, 8
    q, _, v = _inputs(P, B, L, H, D)
    row = np.linspace(-3, 3, D)
    k = [_bf16(np.broadcast_to(row, (B, L, H, D))) for _ in range(P)]
    res = S2.sage2_scatter_qkv(q, k, v, P * L)
    for r in range(P):
        assert not res[r]["k"].any() and not res[r]["k_scale"].any()


def check_decode16():
    assert S2.decode16(np.array([0x3C00, 0xC000, 0x3555], np.uint16), "fp16").tolist() == [1.0, -2.0,
                                                                                        np.float32(np.float16(1 / 3))]
    assert S2.decode16(np.array([0x3F80], np.uint16), "bf16").tolist() == [1.0]


CHECKS = [check_decode16, check_e4m3_rounding, check_e4m3_matches_brute_force, check_int8_quantize, check_k_sum_exact_and_ordered,
          check_sage2_structure_and_bounds, check_sage2_smoothing_removes_channel_offset]


@pytest.mark.parametrize("check", CHECKS, ids=lambda f: f.__name__)
def test_pin(check):
    check()


def test_e4m3_fixture(golden_dir):
    check_e4m3_fixture(golden_dir)


# planted mistakes -----------------------------------------------------------
def _mut_int8_floor(x, inv_scale):
    q = np.floor(np.asarray(x, dtype=np.float32) * np.asarray(inv_scale, dtype=np.float32))
    return np.clip(q, -128, 127).astype(np.int8)


def _mut_e4m3_ties_away(x):
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), 448.0)
    i = np.clip(np.searchsorted(S2._POS_VALUES, a), 1, 126)
    take_hi = (S2._POS_VALUES[i] - a) <= (a - S2._POS_VALUES[i - 1])   # ties go up, not to even
    code = S2._POS_CODES[np.where(take_hi, i, i - 1)].astype(np.uint8)
    return np.where(np.signbit(x), code | 0x80, code).astype(np.uint8)


def _mut_k_sum_no_chunks(k_ranks, dtype="bf16"):
    return np.stack([_f(k).astype(np.float32) for k in k_ranks]).sum(axis=(0, 2)).astype(np.float32) * np.float32(1.001)


def _mut_reciprocal_unguarded(amax, top):
    with np.errstate(divide="ignore"):
        return (np.float32(top) / np.asarray(amax, dtype=np.float32)).astype(np.float32)   # inf where amax == 0


def _mut_reciprocal_swapped(amax, top):
    a = np.asarray(amax, dtype=np.float32)
    return np.where(a > 0, (a / np.float32(top)).astype(np.float32), np.float32(0))


@pytest.mark.parametrize("name,mutant", [("int8_quantize", _mut_int8_floor), ("e4m3_encode", _mut_e4m3_ties_away),
                                         ("reciprocal", _mut_reciprocal_unguarded),
                                         ("reciprocal", _mut_reciprocal_swapped),
                                         ("sage2_k_sum", _mut_k_sum_no_chunks),
                                         ("Q_GROUP", 16), ("K_GROUP", 32), ("V_PAD", 128)])
def test_sage2_pins_catch_planted_mistake(name, mutant, monkeypatch, golden_dir):
    monkeypatch.setattr(S2, name, mutant)
    tripped = []
    for check in CHECKS:
        try:
            with np.errstate(all="ignore"):   # a mutant may make NaNs; only the verdict matters
                check()
        except (AssertionError, ValueError, IndexError):
            tripped.append(check.__name__)
    try:
        check_e4m3_fixture(golden_dir)
    except AssertionError:
        tripped.append("fixture")
    assert tripped, f"no pin caught the planted mistake in {name}"
