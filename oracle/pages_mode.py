"""The pages' own test-reference form of the fused op (diagnostic; test infrastructure only).

Source: "QKV projection + RMSNorm + RoPE overlapped with the Ulysses head exchange"
(flashinfer PR #6332 commit text), "Tests": every path is checked against an fp32
step-by-step reference -- projection, RMSNorm with the bf16 cast before the bf16
scale, interleaved RoPE, bf16 output -- with atol = rtol = 1e-2.

Readings taken where that sentence leaves a step open:
  * projection: fp32 products and sums of the bf16 inputs (a library fp32 matmul),
    not rounded before the norm;
  * RMSNorm: r = 1 / sqrt(mean(y^2) + 1e-6) in fp32, n = bf16(y * r), then the
    weight product bf16(n * w) (a bf16 x bf16 product is exact in fp32 and is
    rounded once, as a bf16 tensor product is);
  * RoPE in fp32 on those bf16 values with the fp32 cos/sin row, either pairing;
  * every output value, v included, rounded to bf16.

This module is a diagnostic beside the float64 oracle, which stays the parity
reference.  Pins: the bf16 rounding against the format's definition (ties to
even, nearest neighbour, NaN and overflow), the whole form against the pinned
float64 oracle within the rounding it adds, and the cast before the scale on an
input where the two cast placements give different bf16 results, against the
steps redone in exact rational arithmetic.
"""
from __future__ import annotations

from typing import Dict, Optional

import numpy as np

from .qnre_oracle import HEAD_DIM, RMS_EPS, bf16_to_f64, place_bands, split_qkv_heads

__all__ = ["round_bf16", "project_norm_rope_pages_mode", "qnre_forward_pages_mode", "pages_close"]

PAGES_ATOL = 1e-2
PAGES_RTOL = 1e-2


def round_bf16(a: np.ndarray) -> np.ndarray:
    """float32 -> float32 holding the nearest bf16 value (ties to the even code); NaN stays NaN."""
    a = np.asarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) & 0xFFFF0000).astype(np.uint32).view(np.float32)
    return np.where(np.isnan(a), np.float32(np.nan), r).astype(np.float32)


def _rms_scale(yg: np.ndarray) -> np.ndarray:
    """1 / sqrt(mean over the head of y^2 + eps), in fp32."""
    ms = np.mean(yg * yg, axis=-1, keepdims=True, dtype=np.float32)
    return (np.float32(1) / np.sqrt(ms + np.float32(RMS_EPS))).astype(np.float32)


def _normalise(yg: np.ndarray, w: np.ndarray) -> np.ndarray:
    """RMSNorm as the pages' reference takes it: the normalised value cast to bf16,
    then the bf16 weight product, rounded to bf16 again."""
    return round_bf16(round_bf16(yg * _rms_scale(yg)) * w)


def _rope_f32(n: np.ndarray, cs: np.ndarray, rope_style: str) -> np.ndarray:
    half = HEAD_DIM // 2
    cos = cs[:, None, :half]
    sin = cs[:, None, half:]
    out = np.empty_like(n)
    if rope_style == "rotate_half":
        a, b = n[..., :half], n[..., half:]
        out[..., :half] = a * cos - b * sin
        out[..., half:] = b * cos + a * sin
    elif rope_style == "interleaved":
        a, b = n[..., 0::2], n[..., 1::2]
        out[..., 0::2] = a * cos - b * sin
        out[..., 1::2] = b * cos + a * sin
    else:
        raise ValueError(f"unknown rope_style {rope_style!r}")
    return out


def project_norm_rope_pages_mode(x_bits: np.ndarray, w_bits: np.ndarray, q_norm_w: np.ndarray,
                                 k_norm_w: np.ndarray, cos_sin: np.ndarray, pos: np.ndarray,
                                 num_heads: int, rope_style: str = "interleaved") -> np.ndarray:
    """O[t, g, h, d] (float32 holding bf16 values) for the token rows x_bits [T, hidden]."""
    x = bf16_to_f64(x_bits).astype(np.float32)
    w = bf16_to_f64(w_bits).astype(np.float32)
    y = split_qkv_heads(x @ w, num_heads).astype(np.float32)            # [T, 3, H, D] fp32
    pos = np.asarray(pos, dtype=np.int64)
    if np.any((pos < 0) | (pos >= cos_sin.shape[0])):
        raise ValueError("a position lies outside the cos/sin table")
    cs = np.asarray(cos_sin, dtype=np.float32)[pos]
    out = np.empty_like(y)
    for g, wbits in ((0, q_norm_w), (1, k_norm_w)):
        n = _normalise(y[:, g], bf16_to_f64(wbits).astype(np.float32))
        out[:, g] = round_bf16(_rope_f32(n, cs, rope_style))
    out[:, 2] = round_bf16(y[:, 2])
    return out


def qnre_forward_pages_mode(x_bits: np.ndarray, w_bits: np.ndarray, q_norm_w: np.ndarray,
                            k_norm_w: np.ndarray, cos_sin: np.ndarray, positions: Optional[np.ndarray],
                            P: int, num_heads: int, layout: str = "bshd",
                            rope_style: str = "interleaved") -> Dict[str, np.ndarray]:
    """The whole fused op in the pages' reference form, placed like the oracle's (float64 arrays)."""
    _, B, S, K = x_bits.shape
    T = P * B * S
    pos = np.arange(T) if positions is None else np.asarray(positions).reshape(T)
    O = project_norm_rope_pages_mode(x_bits.reshape(T, K), w_bits, q_norm_w, k_norm_w, cos_sin, pos,
                                     num_heads, rope_style)
    return place_bands(O.astype(np.float64), P, B, S, num_heads, layout)


def pages_close(got: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """The pages' acceptance test per element: |got - ref| <= atol + rtol |ref|."""
    return np.abs(got - ref) <= PAGES_ATOL + PAGES_RTOL * np.abs(ref)
