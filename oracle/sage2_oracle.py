"""Plain CPU oracle for the Sage2 low-precision QKV exchange (test infrastructure only).

Source: flashinfer.comm API reference v0.7.4, "Prepared Low-Precision QKV
Exchange" and UlyssesCommunicator.prepare_qkv / scatter_qkv, with the
"Low-Precision Implementation Primitives" list: grouped INT8 Q/K and
channel-scaled FP8 E4M3 V; FP32 statistics (a local K sum and V absolute
maximum over the sequence, gathered across ranks); Q amax per global group of
32 tokens, K amax of (K - global mean) per global group of 64 tokens; q, k INT8
[B, S, H/P, D]; v FP8 E4M3 [B, D, H/P, S_pad]; Q/K scales FP32
[B, H/P, width] with widths from the used sequence U; V scales FP32
[B, H/P, D].

Readings where the pages are silent (listed with reasons in the design notes):
  * stored scale = amax / 127 (INT8) or amax / 448 (E4M3 maximum), FP32
    division; the codes use the reciprocal once per group or channel:
    inv = 127 / amax (448 / amax), 0 when amax == 0, and code =
    round-half-even(x * inv) in FP32 (INT8 saturating to [-128, 127]; E4M3
    nearest, ties to even, saturating at +-448).
  * K mean = (sum of K over the whole exchanged sequence) / U, taken exactly and
    rounded once to FP32: the pages fix FP32 statistics but no summation order,
    so the oracle uses the one result every order approximates.
  * Rows at or beyond U get code 0 and take no part in any amax; S_pad = S
    rounded up to a multiple of 64, padded with code 0.
  * Group g of Q covers global rows [32 g, 32 g + 32); of K, [64 g, 64 g + 64).
"""
from __future__ import annotations

from fractions import Fraction
from typing import Dict, List

import numpy as np

from .qnre_oracle import all_to_all, bf16_to_f64

Q_GROUP = 32
K_GROUP = 64
V_PAD = 64
INT8_DIV = np.float32(127.0)
E4M3_MAX = np.float32(448.0)

__all__ = ["decode16", "e4m3_decode", "e4m3_encode", "int8_quantize", "reciprocal", "round_to_f32",
           "sage2_k_mean", "sage2_scatter_qkv", "Q_GROUP", "K_GROUP", "V_PAD"]


# ---------------------------------------------------------------------------
# FP8 E4M3 (sign, 4 exponent bits with bias 7, 3 mantissa bits, no infinity,
# S.1111.111 is NaN, largest finite 448)
# ---------------------------------------------------------------------------
def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return sign * val


_POS_CODES = np.arange(0x7F, dtype=np.uint8)          # 0x00 .. 0x7E: every finite non-negative value
_POS_VALUES = e4m3_decode(_POS_CODES)


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """Nearest E4M3 value (ties to the even code), saturating at +-448; NaN -> 0x7F.

    The 127 finite magnitudes rise with their codes, so the nearest one is one of
    the two neighbours found by a sorted search."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), 448.0)
    i = np.clip(np.searchsorted(_POS_VALUES, a), 1, len(_POS_VALUES) - 1)
    d_lo = a - _POS_VALUES[i - 1]
    d_hi = _POS_VALUES[i] - a
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & ((_POS_CODES[i] & 1) == 0))
    code = _POS_CODES[np.where(take_hi, i, i - 1)].astype(np.uint8)
    code = np.where(np.signbit(x), code | 0x80, code)  # the sign survives rounding to zero
    code = np.where(np.isnan(x), 0x7F, code)
    return code.astype(np.uint8)


def int8_quantize(x: np.ndarray, inv_scale: np.ndarray) -> np.ndarray:
    """round-half-even(x * inv_scale) in FP32, saturated to [-128, 127]."""
    x = np.asarray(x, dtype=np.float32)
    inv = np.asarray(inv_scale, dtype=np.float32)
    q = np.rint((x * inv).astype(np.float32))
    return np.clip(q, -128, 127).astype(np.int8)


def reciprocal(amax: np.ndarray, top: np.float32) -> np.ndarray:
    """top / amax in FP32, 0 where amax == 0 (every code of that group or channel is 0)."""
    a = np.asarray(amax, dtype=np.float32)
    with np.errstate(divide="ignore"):
        inv = (np.float32(top) / a).astype(np.float32)
    return np.where(a > 0, inv, np.float32(0)).astype(np.float32)


# ---------------------------------------------------------------------------
# Statistics
# ---------------------------------------------------------------------------
def decode16(bits: np.ndarray, dtype: str = "bf16") -> np.ndarray:
    """bf16 or fp16 bit patterns (uint16) -> float32 (both convert exactly)."""
    if dtype == "bf16":
        return bf16_to_f64(bits).astype(np.float32)
    if dtype == "fp16":
        return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float32)
    raise ValueError(f"unsupported input dtype {dtype!r}")


def round_to_f32(q: Fraction) -> np.float32:
    """The float32 nearest to the rational q (ties to the even significand): the best
    of the float32 neighbours of q's float64 approximation, compared exactly."""
    c = np.float32(float(q))
    best = None
    for cand in (np.nextafter(c, np.float32(-np.inf)), c, np.nextafter(c, np.float32(np.inf))):
        key = (abs(Fraction(float(cand)) - q), int(np.float32(cand).view(np.uint32)) & 1)
        if best is None or key < best[0]:
            best = (key, np.float32(cand))
    return best[1]


def _exact_row_sums(x: np.ndarray, significant_bits: int) -> np.ndarray:
    """Exact sum over axis 1 of x [B, S, H, D] (float64 decodes of 16-bit floats with
    `significant_bits` bits each), as an object array of Fractions [B, H, D].

    Where every partial sum of a column is a multiple of its smallest bit weight
    below 2^53 of them, float64 addition in any order is exact; other columns are
    summed as Fractions."""
    n = x.shape[1]
    nz = x != 0
    _, e = np.frexp(x)                                   # |x| < 2^e, lowest bit 2^(e - significant_bits)
    e_top = np.where(nz, e, -(1 << 20)).max(axis=1)
    e_low = np.where(nz, e - significant_bits, 1 << 20).min(axis=1)
    fits = ~nz.any(axis=1) | (np.log2(max(n, 1)) + 1 + e_top - e_low <= 53)
    approx = x.sum(axis=1)
    out = np.empty(approx.shape, dtype=object)
    for idx in np.ndindex(approx.shape):
        if fits[idx]:
            out[idx] = Fraction(float(approx[idx]))
        else:
            b, h, d = idx
            out[idx] = sum((Fraction(float(v)) for v in x[b, :, h, d]), Fraction(0))
    return out


def sage2_k_mean(k_ranks: List[np.ndarray], used_sequence: int, dtype: str = "bf16") -> np.ndarray:
    """K mean per (batch, head, channel) over the global sequence: the exact sum of
    every rank's K rows divided by the used length U, rounded once to FP32.
    k_ranks[r] is rank r's [B, L, H, D]; returns [B, H, D] float32.  Rows at or past
    U are zero on input ("Prepared Low-Precision QKV Exchange": zero-padded tail), so
    summing every row sums the used prefix."""
    k = np.concatenate([decode16(kr, dtype).astype(np.float64) for kr in k_ranks], axis=1)   # [B, S, H, D]
    total = _exact_row_sums(k, 8 if dtype == "bf16" else 11)
    U = int(used_sequence)
    out = np.empty(total.shape, np.float32)
    for idx in np.ndindex(total.shape):
        out[idx] = round_to_f32(total[idx] / U)
    return out


def sage2_scatter_qkv(q_ranks: List[np.ndarray], k_ranks: List[np.ndarray], v_ranks: List[np.ndarray],
                      used_sequence: int, dtype: str = "bf16",
                      with_k_scaled: bool = False) -> List[Dict[str, np.ndarray]]:
    """Sage2 encoding after the head exchange, for every virtual rank.

    q/k/v_ranks[r]: bf16 (or fp16) bits [B, L, H, D] of source rank r.  Returns, for each
    destination rank r2 (heads [r2*H/P, (r2+1)*H/P)), a dict with
    q, k: int8 [B, S, H/P, D]; v: E4M3 codes [B, D, H/P, S_pad];
    q_scale [B, H/P, ceil(U/32)], k_scale [B, H/P, ceil(U/64)], v_scale [B, H/P, D] (float32).
    with_k_scaled adds "k_scaled": the fp32 values (K - mean) * 127 / amax that the K
    codes round, [B, S, H/P, D] (0 past U).
    """
    P = len(q_ranks)
    B, L, H, D = q_ranks[0].shape
    if H % P:
        raise ValueError("H must be divisible by P")
    S = P * L
    U = int(used_sequence)
    if not 0 < U <= S:
        raise ValueError("used_sequence must lie in (0, P*L]")
    H_l = H // P
    S_pad = -(-S // V_PAD) * V_PAD
    wq, wk = -(-U // Q_GROUP), -(-U // K_GROUP)

    # the exchange: rank r2 receives heads of its band for the whole sequence, in source-rank order
    def exchange(xs):
        sent = [[x[:, :, r2 * H_l:(r2 + 1) * H_l] for r2 in range(P)] for x in xs]
        return [np.concatenate(rows, axis=1) for rows in all_to_all(sent)]   # [B, S, H_l, D] each

    qg, kg, vg = exchange(q_ranks), exchange(k_ranks), exchange(v_ranks)
    k_mean_all = sage2_k_mean(k_ranks, U, dtype)         # [B, H, D]
    out = []
    live = np.arange(S) < U
    for r2 in range(P):
        qf = decode16(qg[r2], dtype)
        kf = decode16(kg[r2], dtype)
        vf = decode16(vg[r2], dtype)
        k_mean = k_mean_all[:, r2 * H_l:(r2 + 1) * H_l]                     # [B, H_l, D]
        ks = (kf - k_mean[:, None]).astype(np.float32)
        q_scale = np.zeros((B, H_l, wq), np.float32)
        k_scale = np.zeros((B, H_l, wk), np.float32)
        q8 = np.zeros((B, S, H_l, D), np.int8)
        k8 = np.zeros((B, S, H_l, D), np.int8)
        k_scaled = np.zeros((B, S, H_l, D), np.float32)
        for g in range(wq):
            rows = slice(g * Q_GROUP, min(U, (g + 1) * Q_GROUP))
            amax = np.abs(qf[:, rows]).max(axis=(1, 3))                       # [B, H_l]
            q_scale[:, :, g] = (amax / INT8_DIV).astype(np.float32)
            q8[:, rows] = int8_quantize(qf[:, rows], reciprocal(amax, INT8_DIV)[:, None, :, None])
        for g in range(wk):
            rows = slice(g * K_GROUP, min(U, (g + 1) * K_GROUP))
            amax = np.abs(ks[:, rows]).max(axis=(1, 3))
            k_scale[:, :, g] = (amax / INT8_DIV).astype(np.float32)
            inv = reciprocal(amax, INT8_DIV)[:, None, :, None]
            k8[:, rows] = int8_quantize(ks[:, rows], inv)
            k_scaled[:, rows] = (ks[:, rows] * inv).astype(np.float32)
        vamax = np.where(live[None, :, None, None], np.abs(vf), 0).max(axis=1)   # [B, H_l, D]
        v_scale = (vamax / E4M3_MAX).astype(np.float32)
        vq = (vf * reciprocal(vamax, E4M3_MAX)[:, None]).astype(np.float32)
        v8 = np.where(live[None, :, None, None], e4m3_encode(vq), 0).astype(np.uint8)  # [B, S, H_l, D]
        v_out = np.zeros((B, D, H_l, S_pad), np.uint8)
        v_out[..., :S] = v8.transpose(0, 3, 2, 1)
        res = {"q": q8, "k": k8, "v": v_out, "q_scale": q_scale, "k_scale": k_scale, "v_scale": v_scale}
        if with_k_scaled:
            res["k_scaled"] = k_scaled
        out.append(res)
    return out
