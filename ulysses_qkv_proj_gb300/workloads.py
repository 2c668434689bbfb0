"""Seeded synthetic workloads for the Ulysses QKV front end and the head-chunk kernels.

This module only draws inputs. It holds none of the method's arithmetic: no
projection, normalisation, rotation or placement happens here. The tests, the
benchmark and the smoke check draw their inputs from it, and both the CUDA path
and the CPU oracle consume the same arrays.

Shapes follow the pages' workloads:
  * the fused projection grid of "QKV projection + RMSNorm + RoPE overlapped with
    the Ulysses head exchange" (flashinfer PR #6332, Description and Speedup
    sections): hidden = heads x 128, bf16 operands, B = 1 or 2;
  * the MiniMax-H3-like head-chunk shape [1, 37760, 56, 128] with the uneven
    schedule [7, 14, 7] of "allocation-stable, head-chunked Ulysses
    communication primitives" (flashinfer PR #5027, performance table).

Every array is drawn from numpy's PCG64 generator with a fixed seed per tensor
(x=1, W=2, q-norm weight=3, k-norm weight=4, head-chunk q/k/v buffer=5, merge
input=6).  bf16 tensors are returned as uint16 bit patterns, rounded to nearest
even from float32 draws.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Dict, Tuple

import numpy as np

HEAD_DIM = 128
ROPE_THETA = 1.0e4

SEED_X = 1
SEED_W = 2
SEED_QW = 3
SEED_KW = 4
SEED_QKV_BUFFER = 5
SEED_RECEIVED = 6


@dataclass(frozen=True)
class FusedWorkload:
    """One shape of the fused QKV projection + norm + RoPE + band scatter.

    P virtual ranks each hold a [B, S, hidden] activation shard; the whole
    problem on one GPU is T = P*B*S tokens.
    """

    name: str
    P: int
    B: int
    S: int
    num_heads: int
    layout: str = "bshd"          # "bshd" or "fused"
    rope_style: str = "rotate_half"  # "rotate_half" or "interleaved"

    @property
    def hidden(self) -> int:
        return self.num_heads * HEAD_DIM

    @property
    def H_local(self) -> int:
        return self.num_heads // self.P

    @property
    def S_global(self) -> int:
        return self.P * self.S

    @property
    def T(self) -> int:
        return self.P * self.B * self.S

    @property
    def N(self) -> int:
        return 3 * self.num_heads * HEAD_DIM

    @property
    def n_pos(self) -> int:
        return self.S_global

    def flops(self) -> float:
        return 2.0 * self.T * self.hidden * self.N


@dataclass(frozen=True)
class HeadChunkWorkload:
    """Head-chunk pack/merge shape: P virtual ranks, each a [B, S, H, D] shard."""

    name: str
    P: int
    B: int
    S_global: int
    num_heads: int
    schedule: Tuple[Tuple[int, int], ...]
    D: int = HEAD_DIM

    @property
    def S(self) -> int:
        return self.S_global // self.P

    @property
    def H_local(self) -> int:
        return self.num_heads // self.P


# The shapes. Names say what they are.
FUSED_WORKLOADS: Dict[str, FusedWorkload] = {
    "tiny_p2_s64_h4": FusedWorkload("tiny_p2_s64_h4", P=2, B=1, S=64, num_heads=4),
    "h4096_p4_s4096": FusedWorkload("h4096_p4_s4096", P=4, B=1, S=1024, num_heads=32),
    "h7168_p4_s37888_fused": FusedWorkload(
        "h7168_p4_s37888_fused", P=4, B=1, S=9472, num_heads=56, layout="fused"),
    "h8192_p8_b2_s16384": FusedWorkload("h8192_p8_b2_s16384", P=8, B=2, S=2048, num_heads=64),
}

HEADCHUNK_WORKLOADS: Dict[str, HeadChunkWorkload] = {
    "headchunk_p2_s37760_h56": HeadChunkWorkload(
        "headchunk_p2_s37760_h56", P=2, B=1, S_global=37760, num_heads=56,
        schedule=((0, 7), (7, 14), (21, 7))),
    # the same heads over a 16k-token global sequence (q/k/v 0.7 GB): small enough
    # for a per-kernel profile, still several times the L2
    "headchunk_p2_s16384_h56": HeadChunkWorkload(
        "headchunk_p2_s16384_h56", P=2, B=1, S_global=16384, num_heads=56,
        schedule=((0, 7), (7, 14), (21, 7))),
}

# The benchmarked step runs the fused op on the largest fused shape, and the
# head-chunk pack and merge over the same Q/K/V geometry with an uneven schedule
# over H_local = 8.  Beside it the benchmark times the fused op alone on the
# 4096-token shape and the pack/merge alone on the pages' head-chunk shape.
BENCH_FUSED = "h8192_p8_b2_s16384"
BENCH_FUSED_SMALL = "h4096_p4_s4096"
BENCH_HEADCHUNK = "headchunk_p2_s37760_h56"
BENCH_SCHEDULE: Tuple[Tuple[int, int], ...] = ((0, 2), (2, 4), (6, 2))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    bias = ((u >> 16) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> 16).astype(np.uint16)


def _normal_bf16(seed: int, shape, std: float = 1.0, mean: float = 0.0) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(seed))
    a = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    if mean != 0.0:
        a += np.float32(mean)
    return f32_to_bf16_bits(a)


def rope_table(n_pos: int, theta: float = ROPE_THETA, head_dim: int = HEAD_DIM) -> np.ndarray:
    """fp32 cos/sin table [n_pos, head_dim]: row p = [cos(p*f_0..f_63) | sin(p*f_0..f_63)].

    f_i = theta^(-2i/head_dim), evaluated in float64 then rounded to float32.
    The table is an input of the fused op (a per-token fp32 cos/sin table in
    PR #6332, Description, "Architectures").
    """
    half = head_dim // 2
    i = np.arange(half, dtype=np.float64)
    inv_freq = theta ** (-2.0 * i / head_dim)
    p = np.arange(n_pos, dtype=np.float64)[:, None]
    ang = p * inv_freq[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


def global_positions(P: int, B: int, S: int) -> np.ndarray:
    """int32 [P, B, S]: position of token (r, b, s) = r*S + s, its index in the
    global sequence of its batch row (restarts for every b)."""
    r = np.arange(P, dtype=np.int64)[:, None, None]
    s = np.arange(S, dtype=np.int64)[None, None, :]
    pos = r * S + s + np.zeros((1, B, 1), dtype=np.int64)
    return pos.astype(np.int32)


@dataclass
class FusedInputs:
    x: np.ndarray          # uint16 [P, B, S, hidden]
    w: np.ndarray          # uint16 [hidden, 3*H*128]
    q_norm_w: np.ndarray   # uint16 [128]
    k_norm_w: np.ndarray   # uint16 [128]
    cos_sin: np.ndarray    # float32 [n_pos, 128]
    positions: np.ndarray  # int32 [P, B, S]


def make_fused_inputs(wl: FusedWorkload, with_x: bool = True, with_w: bool = True) -> FusedInputs:
    """Draw x ~ N(0,1), W ~ N(0, (1/sqrt(hidden))^2), norm weights ~ 1 + 0.1 N(0,1)."""
    K = wl.hidden
    x = _normal_bf16(SEED_X, (wl.P, wl.B, wl.S, K)) if with_x else None
    w = _normal_bf16(SEED_W, (K, wl.N), std=1.0 / np.sqrt(K)) if with_w else None
    qw = _normal_bf16(SEED_QW, (HEAD_DIM,), std=0.1, mean=1.0)
    kw = _normal_bf16(SEED_KW, (HEAD_DIM,), std=0.1, mean=1.0)
    return FusedInputs(x=x, w=w, q_norm_w=qw, k_norm_w=kw,
                       cos_sin=rope_table(wl.n_pos),
                       positions=global_positions(wl.P, wl.B, wl.S))


def make_exact_fused_inputs(wl: FusedWorkload, wmax: int = 64) -> FusedInputs:
    """Integer-coded inputs whose projection is exact in fp32 and in bf16.

    x[t] has a 1 at column t % K and another +1 at column K-1 - (t // K) % K, W
    holds integers in [-wmax, wmax].  Every projected value is the sum of two
    W entries (|y| <= 2*wmax <= 128), so it is exactly representable in bf16,
    and distinct tokens get distinct rows with high probability: any misplaced
    token shows up as a bit difference.
    """
    K = wl.hidden
    T = wl.T
    x = np.zeros((T, K), dtype=np.uint16)
    t = np.arange(T)
    one = np.uint16(0x3F80)
    two = np.uint16(0x4000)
    c1 = t % K
    c2 = K - 1 - (t // K) % K
    x[t, c1] = one
    same = c1 == c2
    x[t[~same], c2[~same]] = one
    x[t[same], c1[same]] = two
    rng = np.random.Generator(np.random.PCG64(SEED_W))
    wi = rng.integers(-wmax, wmax + 1, size=(K, wl.N)).astype(np.float32)
    base = make_fused_inputs(wl, with_x=False, with_w=False)
    base.x = x.reshape(wl.P, wl.B, wl.S, K)
    base.w = f32_to_bf16_bits(wi)
    return base


def make_headchunk_buffer(B: int, S_global: int, H: int, D: int = HEAD_DIM,
                          seed: int = SEED_QKV_BUFFER) -> np.ndarray:
    """bf16 N(0,1) buffer [B, S_global, 3, H, D]; q/k/v are its [..., c, :, :] slices."""
    return _normal_bf16(seed, (B, S_global, 3, H, D))


def make_received(B: int, S: int, heads: int, D: int = HEAD_DIM,
                  seed: int = SEED_RECEIVED) -> np.ndarray:
    """bf16 N(0,1) gathered output band [B, S, heads, D] (merge input)."""
    return _normal_bf16(seed, (B, S, heads, D))
