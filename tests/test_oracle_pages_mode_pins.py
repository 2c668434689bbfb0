"""Pins for the pages' test-reference form (oracle/pages_mode.py, a diagnostic): the
bf16 rounding against the format's definition, and the whole form against the pinned
float64 oracle within the error its extra roundings allow.  Planted mistakes trip a pin."""
from decimal import Decimal, localcontext
from fractions import Fraction

import numpy as np
import pytest

import oracle
import oracle.pages_mode as PM
from ulysses_qkv_proj_gb300 import workloads as WL


def check_round_bf16_exact_values():
    bits = np.arange(1 << 16, dtype=np.uint32)
    f = (bits << 16).view(np.float32)
    r = PM.round_bf16(f)
    nan = np.isnan(f)
    assert np.array_equal(r[~nan].view(np.uint32), f[~nan].view(np.uint32))   # every bf16 value is kept
    assert np.isnan(r[nan]).all()


def check_round_bf16_ties_and_nearest():
    lo = (np.arange(0x3F80, 0x4000, dtype=np.uint32) << 16).view(np.float32)  # bf16 values in [1, 2)
    mid = (lo.astype(np.float64) + 2.0 ** -8).astype(np.float32)             # exact midpoints
    r = PM.round_bf16(mid).view(np.uint32) >> 16
    assert np.all(r % 2 == 0)                                                # ties go to the even code
    assert PM.round_bf16(np.float32(1 + 2 ** -8)) == 1.0
    assert PM.round_bf16(np.float32(1 + 3 * 2 ** -8)) == np.float32(1 + 2 ** -6)
    assert PM.round_bf16(np.float32(-(1 + 2 ** -8))) == -1.0
    rng = np.random.default_rng(41)
    x = (rng.standard_normal(20000) * np.exp2(rng.integers(-20, 20, 20000))).astype(np.float32)
    down = (x.view(np.uint32) & 0xFFFF0000).view(np.float32).astype(np.float64)   # toward zero
    up = ((x.view(np.uint32) & 0xFFFF0000) + 0x10000).view(np.float32).astype(np.float64)
    got = PM.round_bf16(x).astype(np.float64)
    xd = x.astype(np.float64)
    assert np.all((got == down) | (got == up))                              # one of the two neighbours
    assert np.all(np.abs(got - xd) <= np.minimum(np.abs(xd - down), np.abs(xd - up)))  # the nearer one
    assert np.isinf(PM.round_bf16(np.float32(3.4e38)))                       # past the largest finite bf16
    assert np.isnan(PM.round_bf16(np.float32(np.nan)))


def _bound_check(wl, rope_style):
    """|pages form - float64 oracle| within the roundings the pages' form adds:
    n and n*w each rounded to bf16 (unit roundoff 2^-8 each: 8 significant
    bits), RoPE's two products in fp32, the output rounded once more
    (2^-8 |o|), fp32 projection noise."""
    inp = WL.make_fused_inputs(wl)
    T, K = wl.T, wl.hidden
    x = inp.x.reshape(T, K)
    pos = inp.positions.reshape(T)
    pm = PM.project_norm_rope_pages_mode(x, inp.w, inp.q_norm_w, inp.k_norm_w, inp.cos_sin, pos,
                                         wl.num_heads, rope_style).astype(np.float64)
    ref = oracle.project_norm_rope(x, inp.w, inp.q_norm_w, inp.k_norm_w, inp.cos_sin, pos, wl.num_heads,
                                   rope_style)
    y = oracle.split_qkv_heads(oracle.qkv_projection(x, inp.w), wl.num_heads)
    for g, wbits in ((0, inp.q_norm_w), (1, inp.k_norm_w)):
        n = np.abs(oracle.rms_norm(y[:, g], wbits))
        partner = np.empty_like(n)
        if rope_style == "interleaved":
            partner[..., 0::2], partner[..., 1::2] = n[..., 1::2], n[..., 0::2]
        else:
            h = n.shape[-1] // 2
            partner[..., :h], partner[..., h:] = n[..., h:], n[..., :h]
        bound = 2.0 ** -7 * (n + partner) * 1.001 + 2.0 ** -8 * np.abs(ref[:, g]) + 1e-5
        assert np.all(np.abs(pm[:, g] - ref[:, g]) <= bound), f"group {g}"
    assert np.all(np.abs(pm[:, 2] - ref[:, 2]) <= 2.0 ** -8 * np.abs(ref[:, 2]) + 1e-5)


def check_pages_form_within_rounding_of_oracle():
    for rope in ("interleaved", "rotate_half"):
        _bound_check(WL.FUSED_WORKLOADS["tiny_p2_s64_h4"], rope)


def check_pages_close_semantics():
    ref = np.array([0.0, 1.0, -3.0, 100.0])
    assert PM.pages_close(ref + np.array([0.0099, 0.0199, -0.0399, 1.0099]), ref).tolist() == [True] * 4
    assert PM.pages_close(ref + np.array([0.0101, 0.0201, 0.0401, 1.0101]), ref).tolist() == [False] * 4


def _rn(x, bits):
    """Round a rational to `bits` significant bits, to nearest, ties to even (normal range)."""
    if x == 0:
        return Fraction(0)
    sign = -1 if x < 0 else 1
    a = abs(Fraction(x))
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    scale = Fraction(2) ** (bits - 1 - e)
    m = a * scale
    fl = m.numerator // m.denominator
    rem = m - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return sign * Fraction(fl) / scale


def _sqrt_rn(x, bits):
    """Correctly rounded square root: 80 decimal digits, far more than a 24-bit rounding needs."""
    with localcontext() as ctx:
        ctx.prec = 80
        root = (Decimal(x.numerator) / Decimal(x.denominator)).sqrt()
    return _rn(Fraction(root), bits)


def check_cast_before_scale():
    """A head of one constant c = 2^-14 with weight 1.125 at position 0 (no rotation):
    the pages' reference casts the normalised value to bf16 before the scale.  The
    expected bf16 value is redone here in exact rationals (fp32 = 24 bits, bf16 = 8
    bits, each operation rounded once); the other cast placement gives another value."""
    c, w = Fraction(1, 2 ** 14), Fraction(9, 8)
    eps = Fraction(float(np.float32(PM.RMS_EPS)))
    r = _rn(1 / _sqrt_rn(_rn(c * c + eps, 24), 24), 24)       # mean of c^2 is exact
    n = _rn(c * r, 24)
    want = _rn(_rn(n, 8) * w, 8)
    other = _rn(_rn(n * w, 24), 8)
    assert want != other
    H, D = 1, oracle.HEAD_DIM
    x = np.zeros((1, H * D), np.uint16)
    x[0, 0] = 0x3F80                                           # one-hot row: y = W[0, :]
    wmat = np.zeros((H * D, 3 * H * D), np.uint16)
    wmat[0, :2 * D] = 0x3880                                   # q and k heads: c = 2^-14
    wmat[0, 2 * D:] = 0x3F80
    wn = np.full(D, 0x3F90, np.uint16)                         # 1.125
    cs = np.zeros((1, D), np.float32)
    cs[0, :D // 2] = 1.0                                       # position 0: cos 1, sin 0
    out = PM.project_norm_rope_pages_mode(x, wmat, wn, wn, cs, np.array([0]), H, "interleaved")
    assert np.all(out[0, :2].astype(np.float64) == float(want))


CHECKS = [check_round_bf16_exact_values, check_round_bf16_ties_and_nearest,
          check_pages_form_within_rounding_of_oracle, check_pages_close_semantics, check_cast_before_scale]


@pytest.mark.parametrize("check", CHECKS, ids=lambda f: f.__name__)
def test_pin(check):
    check()


# planted mistakes -----------------------------------------------------------
def _mut_round_truncate(a):
    a = np.asarray(a, dtype=np.float32)
    return (a.view(np.uint32) & 0xFFFF0000).view(np.float32)


def _mut_round_ties_up(a):
    a = np.asarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    return ((u + 0x8000) & 0xFFFF0000).astype(np.uint32).view(np.float32)


def _mut_rope_sign(n, cs, rope_style):
    half = oracle.HEAD_DIM // 2
    cos, sin = cs[:, None, :half], cs[:, None, half:]
    out = np.empty_like(n)
    a, b = n[..., 0::2], n[..., 1::2]
    out[..., 0::2] = a * cos + b * sin          # wrong sign
    out[..., 1::2] = b * cos - a * sin
    return out


def _mut_rms_sum(yg):                          # sum instead of mean over the head
    ms = np.sum(yg * yg, axis=-1, keepdims=True, dtype=np.float32)
    return (np.float32(1) / np.sqrt(ms + np.float32(PM.RMS_EPS))).astype(np.float32)


def _mut_rope_pairing(n, cs, rope_style):      # always rotate-half
    half = oracle.HEAD_DIM // 2
    cos, sin = cs[:, None, :half], cs[:, None, half:]
    out = np.empty_like(n)
    a, b = n[..., :half], n[..., half:]
    out[..., :half] = a * cos - b * sin
    out[..., half:] = b * cos + a * sin
    return out


def _mut_cast_after_scale(yg, w):               # one rounding after the weight product
    return PM.round_bf16(yg * PM._rms_scale(yg) * w)


@pytest.mark.parametrize("name,mutant", [("round_bf16", _mut_round_truncate), ("round_bf16", _mut_round_ties_up),
                                         ("_rope_f32", _mut_rope_sign), ("_rope_f32", _mut_rope_pairing),
                                         ("_rms_scale", _mut_rms_sum), ("_normalise", _mut_cast_after_scale)])
def test_pages_mode_pins_catch_planted_mistake(name, mutant, monkeypatch):
    monkeypatch.setattr(PM, name, mutant)
    tripped = []
    for check in CHECKS:
        try:
            with np.errstate(all="ignore"):
                check()
        except (AssertionError, ValueError):
            tripped.append(check.__name__)
    assert tripped, f"no pin caught the planted mistake in {name}"
