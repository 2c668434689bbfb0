"""Pins for the Sage2 oracle: the E4M3 and INT8 encoders against the formats' definitions,
the K mean against exact rational arithmetic, and the encoding against invariants that
any correct grouped quantiser satisfies.  Planted mistakes must trip a pin."""
import json
import os
from fractions import Fraction

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


def _f32_of_rational(q):
    """Nearest float32 to the rational q, ties to even, by integer arithmetic: scale q
    so that its float32 significand is an integer, round half to even, scale back."""
    q = Fraction(q)
    if q == 0:
        return np.float32(0.0)
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1                                            # now 2^e <= a < 2^(e+1)
    e = max(e, -126)                                      # subnormals share the smallest exponent
    m = round(a / Fraction(2) ** (e - 23))                # Fraction.__round__ ties to even
    v = float(Fraction(m) * Fraction(2) ** (e - 23))
    return np.float32(-v if q < 0 else v)


def check_k_mean_exact():
    """The K mean is the exact sum over the whole sequence divided by U, rounded once
    to fp32, in every case: small integers, random values against rational arithmetic,
    a column whose float32 sums (row by row, or in 256-row chunks) round differently,
    and a column too wide for float64 summation."""
    rng = np.random.default_rng(31)
    P, B, L, H, D = 2, 1, 300, 2, 4
    ints = rng.integers(-50, 51, size=(P, B, L, H, D)).astype(np.float32)
    ks = [_bf16(ints[r]) for r in range(P)]
    U = P * L
    want = np.vectorize(lambda v: _f32_of_rational(Fraction(int(v), U)))(ints.sum(axis=(0, 2)))
    assert np.array_equal(S2.sage2_k_mean(ks, U), want.astype(np.float32))
    # random bf16 values, U shorter than the sequence (rows past U zero)
    vals = (rng.standard_normal((P, B, L, H, D)) * 3 + 2).astype(np.float32)
    U = 517
    vals.reshape(P * L, H, D)[U:] = 0                    # B = 1: global row r*L + s, zero past U
    ks = [_bf16(vals[r]) for r in range(P)]
    dec = np.stack([_f(k) for k in ks])                  # [P, B, L, H, D] exact values
    got = S2.sage2_k_mean(ks, U)
    for b, h, d in np.ndindex(B, H, D):
        exact = sum((Fraction(float(v)) for v in dec[:, b, :, h, d].ravel()), Fraction(0)) / U
        assert got[b, h, d] == _f32_of_rational(exact), (b, h, d)
    # 2^24 followed by 299 ones: float32 sums lose the ones (row by row: 2^24; in
    # 256-row chunks: 2^24 + 44); the exact mean keeps them
    col = np.ones((1, 1, 300, 1, 1), np.float32)
    col[0, 0, 0] = 2.0 ** 24
    m = S2.sage2_k_mean([_bf16(col[0])], 300)
    assert m[0, 0, 0] == _f32_of_rational(Fraction(2 ** 24 + 299, 300))
    assert m[0, 0, 0] != np.float32(np.float32(2.0 ** 24) / np.float32(300))
    assert m[0, 0, 0] != np.float32(np.float32(2.0 ** 24 + 44) / np.float32(300))
    # 2^60 + 2^-60 - 2^60: float64 sums in row order give 0; the exact sum is 2^-60
    wide = np.zeros((1, 1, 3, 1, 1), np.float32)
    wide[0, 0, :, 0, 0] = [2.0 ** 60, 2.0 ** -60, -(2.0 ** 60)]
    m = S2.sage2_k_mean([_bf16(wide[0])], 3)
    assert m[0, 0, 0] == _f32_of_rational(Fraction(1, 3 * 2 ** 60)) and m[0, 0, 0] > 0


def check_round_to_f32():
    """round_to_f32 against the integer-arithmetic rounding above, at ties and between."""
    rng = np.random.default_rng(34)
    one = Fraction(1)
    cases = [one / 3, -one / 3, Fraction(2 ** 24 + 1), Fraction(2 ** 24 + 3), Fraction(1, 2 ** 149),
             Fraction(3, 2 ** 150), Fraction(10 ** 30, 7)]
    cases += [Fraction(int(n), int(dn)) for n, dn in zip(rng.integers(-10 ** 12, 10 ** 12, 300),
                                                        rng.integers(1, 10 ** 9, 300))]
    for q in cases:
        assert S2.round_to_f32(q) == _f32_of_rational(q), q
    assert S2.round_to_f32(Fraction(2 ** 24 + 1)) == np.float32(2 ** 24)       # tie to the even significand
    assert S2.round_to_f32(Fraction(2 ** 24 + 3)) == np.float32(2 ** 24 + 4)


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
        kmean = S2.sage2_k_mean(k, U)
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


CHECKS = [check_decode16, check_e4m3_rounding, check_e4m3_matches_brute_force, check_int8_quantize,
          check_k_mean_exact, check_round_to_f32, check_sage2_structure_and_bounds,
          check_sage2_smoothing_removes_channel_offset]


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


def _mut_k_mean_f32_rows(k_ranks, used_sequence, dtype="bf16"):
    """float32 sum row by row, then / U: a plausible kernel order, not the definition."""
    k = np.concatenate([S2.decode16(kr, dtype) for kr in k_ranks], axis=1)
    acc = np.zeros((k.shape[0], k.shape[2], k.shape[3]), np.float32)
    for s in range(k.shape[1]):
        acc = (acc + k[:, s]).astype(np.float32)
    return (acc / np.float32(used_sequence)).astype(np.float32)


def _mut_k_mean_f32_chunks(k_ranks, used_sequence, dtype="bf16"):
    """float32 sums of 256-row chunks, chunks in order, then / U."""
    k = np.concatenate([S2.decode16(kr, dtype) for kr in k_ranks], axis=1)
    total = np.zeros((k.shape[0], k.shape[2], k.shape[3]), np.float32)
    for c0 in range(0, k.shape[1], 256):
        acc = np.zeros_like(total)
        for s in range(c0, min(k.shape[1], c0 + 256)):
            acc = (acc + k[:, s]).astype(np.float32)
        total = (total + acc).astype(np.float32)
    return (total / np.float32(used_sequence)).astype(np.float32)


def _mut_k_mean_over_all_rows(k_ranks, used_sequence, dtype="bf16"):
    """divides by the whole sequence length instead of the used length U"""
    n = sum(kr.shape[1] for kr in k_ranks)
    return S2.__dict__["_orig_k_mean"](k_ranks, n, dtype)


def _mut_round_to_f32_truncate(q):
    """rounds toward zero instead of to nearest"""
    c = np.float32(float(q))
    return c if abs(Fraction(float(c))) <= abs(Fraction(q)) else np.nextafter(c, np.float32(0))


def _mut_reciprocal_unguarded(amax, top):
    with np.errstate(divide="ignore"):
        return (np.float32(top) / np.asarray(amax, dtype=np.float32)).astype(np.float32)   # inf where amax == 0


def _mut_reciprocal_swapped(amax, top):
    a = np.asarray(amax, dtype=np.float32)
    return np.where(a > 0, (a / np.float32(top)).astype(np.float32), np.float32(0))


@pytest.mark.parametrize("name,mutant", [("int8_quantize", _mut_int8_floor), ("e4m3_encode", _mut_e4m3_ties_away),
                                         ("reciprocal", _mut_reciprocal_unguarded),
                                         ("reciprocal", _mut_reciprocal_swapped),
                                         ("sage2_k_mean", _mut_k_mean_f32_rows),
                                         ("sage2_k_mean", _mut_k_mean_f32_chunks),
                                         ("sage2_k_mean", _mut_k_mean_over_all_rows),
                                         ("round_to_f32", _mut_round_to_f32_truncate),
                                         ("Q_GROUP", 16), ("K_GROUP", 32), ("V_PAD", 128)])
def test_sage2_pins_catch_planted_mistake(name, mutant, monkeypatch, golden_dir):
    monkeypatch.setitem(S2.__dict__, "_orig_k_mean", S2.sage2_k_mean)
    monkeypatch.setattr(S2, name, mutant)
    tripped = []
    for check in CHECKS:
        try:
            with np.errstate(all="ignore"):   # a mutant may make NaNs; only the outcome matters
                check()
        except (AssertionError, ValueError, IndexError):
            tripped.append(check.__name__)
    try:
        check_e4m3_fixture(golden_dir)
    except AssertionError:
        tripped.append("fixture")
    assert tripped, f"no pin caught the planted mistake in {name}"
