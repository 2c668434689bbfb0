"""Plain float64 CPU oracle (test infrastructure only; see the package docstring).

Sources, by page and section:

[FUSED]  flashinfer.comm API reference (v0.7.4), "Fused QKV Projection + Norm +
         RoPE + Head Exchange" (class QkvNormRopeExchangeOverlap): bf16 QKV
         projection, per-head RMSNorm of Q and K with one [D] scale each, RoPE
         from a per-token [rows, D] cos/sin table, head exchange; layouts
         "bshd" = (q, k, v) each [B, S_global, H_local, D] and "fused" =
         [B, S_global, H_local, 3*D]; each rank receives head band
         [rank*H_local, (rank+1)*H_local) of the whole sequence.
[MATH]   "QKV projection + RMSNorm + RoPE overlapped with the Ulysses head
         exchange" (flashinfer PR #6332 commit text, quoted on the docs PR
         #4240 page), "Assumptions", "Operator math": fp32 RMSNorm with
         eps = 1e-6 and a shared [head_dim] weight per Q / K, RoPE applied in
         fp32 from a per-token cos/sin table, order projection -> QK-norm ->
         RoPE; Ulysses all-to-all (every rank holds a token shard and the full
         QKV weight).
[GROUPS] same API page, Notes on the 256-column pair tile: the projection's
         columns are grouped Q | K | V, each group H*D columns wide.
[ULY]    same API reference, "Ulysses Context-Parallel All-to-All":
         scatter_heads [B, S_local, H, D] -> [B, S_global, H_local, D], rank r
         keeps heads [r*H_local, (r+1)*H_local) of the full sequence;
         S_global = S_local * world_size; world_size == 1 is the identity.
[PACK]   same API reference, "Head-Chunk Layout and Transport Primitives",
         pack_ulysses_qkv_head_chunk.
[MERGE]  same section, merge_ulysses_output_head_chunk.
[XCHG]   same API reference, UlyssesCommunicator.scatter_qkv_head_chunk (pack +
         one all-to-all; its result is [B, S_global, head_count, 3*D]) and
         gather_output_head_chunk (x [B, S_global, head_count, D]; the NCCL
         path packs the sequence split into staging, exchanges, and merges the
         received band into out [B, S_global/world_size, world_size*local_heads,
         D]); exchange_chunks: chunk r goes to peer r and lands in slot `rank`
         there ("Ulysses Context-Parallel All-to-All").

Readings taken where the pages leave a step open (each is listed with its
reason in the design notes):
  * RoPE pairing: the pages describe interleaved (pairwise) RoPE; rotate-half
    (pairs (i, i+64)) is the default here and both are provided.
  * cos/sin row layout: row p = [cos_0 .. cos_63 | sin_0 .. sin_63] (fp32).
  * A token's cos/sin row is positions[token]; with no positions it is the
    token's index in the [P, B, S] token order.  A position outside the table
    has no rotation: that token's q and k rows are NaN.
  * Intermediate rounding: none. The oracle keeps float64 from the bf16 inputs
    to the final value.
  * x is [P, B, S, hidden]: virtual rank r_s's [B, S, hidden] shard first.
"""
from __future__ import annotations

from typing import Dict, Optional, Sequence, Tuple

import numpy as np

HEAD_DIM = 128
RMS_EPS = 1.0e-6

__all__ = [
    "HEAD_DIM", "RMS_EPS", "bf16_to_f64", "qkv_projection", "split_qkv_heads",
    "rms_norm", "rope_rotate_half", "rope_interleaved", "apply_rope",
    "project_norm_rope", "token_coords", "band_destination", "place_bands",
    "qnre_forward", "pack_head_chunk", "merge_output_head_chunk",
    "scatter_heads", "gather_heads", "all_to_all", "pack_output_sequence_chunk",
    "gather_output_head_chunk", "scatter_qkv_head_chunk", "bf16_ulp", "fused_tolerance",
]


# ---------------------------------------------------------------------------
# bf16 decoding (data format, not part of the method)
# ---------------------------------------------------------------------------
def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64. A bf16 is the top half of a float32."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# Step 1: projection  Y = x W   [MATH], [FUSED]
# ---------------------------------------------------------------------------
def qkv_projection(x_bits: np.ndarray, w_bits: np.ndarray) -> np.ndarray:
    """Y[t, c] = sum_k x[t, k] * W[k, c] in float64.

    x: bf16 [T, hidden]; W: bf16 [hidden, 3*H*D].  Every bf16 product is exact
    in float64, so Y differs from the exact sum only by float64 rounding.
    """
    x = bf16_to_f64(x_bits)
    w = bf16_to_f64(w_bits)
    if x.ndim != 2 or w.ndim != 2 or x.shape[1] != w.shape[0]:
        raise ValueError(f"projection shapes {x.shape} x {w.shape}")
    return x @ w


def split_qkv_heads(y: np.ndarray, num_heads: int, head_dim: int = HEAD_DIM) -> np.ndarray:
    """[T, 3*H*D] -> [T, 3, H, D]: column c = g*H*D + h*D + d  [GROUPS]."""
    T = y.shape[0]
    if y.shape[1] != 3 * num_heads * head_dim:
        raise ValueError("projection width is not 3*H*D")
    return y.reshape(T, 3, num_heads, head_dim)


# ---------------------------------------------------------------------------
# Step 2: per-head RMSNorm of q and k   [MATH] "Operator math"
# ---------------------------------------------------------------------------
def rms_norm(y: np.ndarray, weight_bits: np.ndarray, eps: float = RMS_EPS) -> np.ndarray:
    """n_d = y_d / sqrt(mean_d(y^2) + eps) * w_d over the last (head) axis."""
    w = bf16_to_f64(weight_bits)
    ms = np.mean(y * y, axis=-1, keepdims=True)
    return y / np.sqrt(ms + eps) * w


# ---------------------------------------------------------------------------
# Step 3: RoPE from the cos/sin table   [MATH], [FUSED]
# ---------------------------------------------------------------------------
def rope_rotate_half(n: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    """Rotate pairs (i, i + D/2) by the angle whose cosine/sine are cos_i, sin_i.

    o_i       = n_i cos_i - n_{i+D/2} sin_i
    o_{i+D/2} = n_{i+D/2} cos_i + n_i sin_i
    """
    half = n.shape[-1] // 2
    a = n[..., :half]
    b = n[..., half:]
    return np.concatenate([a * cos - b * sin, b * cos + a * sin], axis=-1)


def rope_interleaved(n: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    """Rotate pairs (2i, 2i+1): o_2i = n_2i cos_i - n_2i+1 sin_i, o_2i+1 = n_2i+1 cos_i + n_2i sin_i."""
    a = n[..., 0::2]
    b = n[..., 1::2]
    out = np.empty_like(n)
    out[..., 0::2] = a * cos - b * sin
    out[..., 1::2] = b * cos + a * sin
    return out


def apply_rope(n: np.ndarray, cos_sin_rows: np.ndarray, rope_style: str) -> np.ndarray:
    """n: [T, heads, D]; cos_sin_rows: [T, D] float (row = [cos | sin])."""
    half = n.shape[-1] // 2
    cs = np.asarray(cos_sin_rows, dtype=np.float64)
    cos = cs[:, None, :half]
    sin = cs[:, None, half:]
    if rope_style == "rotate_half":
        return rope_rotate_half(n, cos, sin)
    if rope_style == "interleaved":
        return rope_interleaved(n, cos, sin)
    raise ValueError(f"unknown rope_style {rope_style!r}")


# ---------------------------------------------------------------------------
# Steps 1-3 for a set of tokens
# ---------------------------------------------------------------------------
def project_norm_rope(x_bits: np.ndarray, w_bits: np.ndarray, q_norm_w: np.ndarray,
                      k_norm_w: np.ndarray, cos_sin: np.ndarray, pos: np.ndarray,
                      num_heads: int, rope_style: str = "rotate_half",
                      epilogue: bool = True) -> np.ndarray:
    """Per-token result O[t, g, h, d] (float64) for the token rows of x_bits [T, hidden].

    pos[t] is the cos/sin row of token t.  g = 0, 1, 2 is q, k, v: q and k are
    normalised then rotated; v is the projection unchanged.  With
    epilogue=False the result is the bare projection (all three groups).
    """
    y = split_qkv_heads(qkv_projection(x_bits, w_bits), num_heads)
    if not epilogue:
        return y
    pos = np.asarray(pos, dtype=np.int64)
    n_pos = cos_sin.shape[0]
    ok = (pos >= 0) & (pos < n_pos)
    rows = np.where(ok, pos, 0)
    cs = np.asarray(cos_sin, dtype=np.float64)[rows]
    out = np.empty_like(y)
    for g, wbits in ((0, q_norm_w), (1, k_norm_w)):
        out[:, g] = apply_rope(rms_norm(y[:, g], wbits), cs, rope_style)
        out[~ok, g] = np.nan
    out[:, 2] = y[:, 2]
    return out


# ---------------------------------------------------------------------------
# Step 4: head-band placement   [ULY], [FUSED]
# ---------------------------------------------------------------------------
def token_coords(t: int, P: int, B: int, S: int) -> Tuple[int, int, int]:
    """Token t of the [P, B, S] order -> (source rank r_s, batch b, local position s)."""
    if not 0 <= t < P * B * S:
        raise IndexError(t)
    return t // (B * S), (t // S) % B, t % S


def band_destination(r_s: int, b: int, s: int, h: int, P: int, B: int, S: int,
                     num_heads: int) -> Tuple[int, int, int, int]:
    """Where head h of token (r_s, b, s) lands: (dest rank r, batch b, global row, local head).

    Rank r receives heads [r*H_local, (r+1)*H_local) of every token; the token of
    source rank r_s at local position s sits at global row r_s*S + s.
    """
    H_local = num_heads // P
    return h // H_local, b, r_s * S + s, h % H_local


def place_bands(O: np.ndarray, P: int, B: int, S: int, num_heads: int,
                layout: str) -> Dict[str, np.ndarray]:
    """Scatter per-token results O [P*B*S, 3, H, D] into every rank's band.

    bshd : {"q","k","v"}: [P, B, S_global, H_local, D]
    fused: {"fused"}:     [P, B, S_global, H_local, 3*D], q|k|v in the last axis.
    The result has O's dtype.  Unwritten elements stay NaN (float) or all-ones
    (integer bit patterns), so a hole in the map is visible.
    """
    if num_heads % P:
        raise ValueError("num_heads must be divisible by P")
    H_local = num_heads // P
    S_g = P * S
    D = O.shape[-1]
    fill = np.nan if np.issubdtype(O.dtype, np.floating) else np.iinfo(O.dtype).max
    if layout == "bshd":
        out = {g: np.full((P, B, S_g, H_local, D), fill, dtype=O.dtype) for g in "qkv"}
    elif layout == "fused":
        out = {"fused": np.full((P, B, S_g, H_local, 3 * D), fill, dtype=O.dtype)}
    else:
        raise ValueError(f"unknown layout {layout!r}")
    for r_s in range(P):
        for b in range(B):
            t0 = (r_s * B + b) * S
            rows = slice(r_s * S, r_s * S + S)
            for r in range(P):
                heads = slice(r * H_local, (r + 1) * H_local)
                for gi, g in enumerate("qkv"):
                    src = O[t0:t0 + S, gi, heads, :]
                    if layout == "bshd":
                        out[g][r, b, rows, :, :] = src
                    else:
                        out["fused"][r, b, rows, :, gi * D:(gi + 1) * D] = src
    return out


def qnre_forward(x_bits: np.ndarray, w_bits: np.ndarray, q_norm_w: np.ndarray,
                 k_norm_w: np.ndarray, cos_sin: np.ndarray,
                 positions: Optional[np.ndarray], P: int, num_heads: int,
                 layout: str = "bshd", rope_style: str = "rotate_half",
                 epilogue: bool = True) -> Dict[str, np.ndarray]:
    """The whole fused op: x [P, B, S, hidden] -> every rank's head band (float64)."""
    if x_bits.ndim != 4 or x_bits.shape[0] != P:
        raise ValueError("x must be [P, B, S, hidden]")
    _, B, S, K = x_bits.shape
    if K != num_heads * HEAD_DIM:
        raise ValueError("hidden must equal num_heads * 128")
    T = P * B * S
    pos = np.arange(T) if positions is None else np.asarray(positions).reshape(T)
    O = project_norm_rope(x_bits.reshape(T, K), w_bits, q_norm_w, k_norm_w, cos_sin, pos,
                          num_heads, rope_style, epilogue)
    return place_bands(O, P, B, S, num_heads, layout)


# ---------------------------------------------------------------------------
# Head-chunk pack and merge   [PACK], [MERGE]
# ---------------------------------------------------------------------------
def pack_head_chunk(q: np.ndarray, k: np.ndarray, v: np.ndarray, world_size: int,
                    head_offset: int, head_count: int) -> np.ndarray:
    """[B, S, H, D] x 3 -> contiguous [B, S, world_size*head_count, 3*D].

    Slot r*head_count + j holds local head head_offset + j of destination rank
    r's head slice, i.e. global head r*(H/world_size) + head_offset + j, with
    q | k | v along the last axis.
    """
    if not (q.shape == k.shape == v.shape) or q.ndim != 4:
        raise ValueError("q, k, v must share one [B, S, H, D] shape")
    B, S, H, D = q.shape
    if world_size < 1 or H % world_size:
        raise ValueError("H must be divisible by world_size")
    H_local = H // world_size
    if head_offset < 0 or head_count < 1 or head_offset + head_count > H_local:
        raise ValueError("band outside the local heads")
    out = np.empty((B, S, world_size * head_count, 3 * D), dtype=q.dtype)
    for r in range(world_size):
        for j in range(head_count):
            h = r * H_local + head_offset + j
            for c, X in enumerate((q, k, v)):
                out[:, :, r * head_count + j, c * D:(c + 1) * D] = X[:, :, h, :]
    return out


def merge_output_head_chunk(received: np.ndarray, world_size: int, local_heads: int,
                            head_offset: int, out: np.ndarray) -> np.ndarray:
    """Return a copy of out [B, S, world_size*local_heads, D] with the band merged.

    Head r*local_heads + head_offset + j of the result is received head
    r*head_count + j; every other element keeps its value.
    """
    B, S, WC, D = received.shape
    if world_size < 1 or WC % world_size:
        raise ValueError("received heads must be a multiple of world_size")
    head_count = WC // world_size
    if head_offset < 0 or head_offset + head_count > local_heads:
        raise ValueError("band outside the local heads")
    if out.shape != (B, S, world_size * local_heads, D):
        raise ValueError("out must be [B, S, world_size*local_heads, D]")
    res = out.copy()
    for r in range(world_size):
        for j in range(head_count):
            res[:, :, r * local_heads + head_offset + j, :] = received[:, :, r * head_count + j, :]
    return res


# ---------------------------------------------------------------------------
# Ordinary (whole-band) layout transforms over P virtual ranks   [ULY]
# ---------------------------------------------------------------------------
def scatter_heads(x: np.ndarray) -> np.ndarray:
    """[P, B, S, H, D] (rank r_s's shard first) -> [P, B, P*S, H/P, D].

    Result rank r, row r_s*S + s, local head hl = x[r_s, b, s, r*H_local + hl].
    """
    P, B, S, H, D = x.shape
    if H % P:
        raise ValueError("H must be divisible by P")
    H_local = H // P
    out = np.empty((P, B, P * S, H_local, D), dtype=x.dtype)
    for r in range(P):
        for r_s in range(P):
            out[r, :, r_s * S:(r_s + 1) * S] = x[r_s, :, :, r * H_local:(r + 1) * H_local]
    return out


def gather_heads(y: np.ndarray) -> np.ndarray:
    """Inverse of scatter_heads: [P, B, S_global, H_local, D] -> [P, B, S_global/P, H, D]."""
    P, B, S_g, H_local, D = y.shape
    if S_g % P:
        raise ValueError("S_global must be divisible by P")
    S = S_g // P
    out = np.empty((P, B, S, P * H_local, D), dtype=y.dtype)
    for r_s in range(P):
        for r in range(P):
            out[r_s, :, :, r * H_local:(r + 1) * H_local] = y[r, :, r_s * S:(r_s + 1) * S]
    return out


# ---------------------------------------------------------------------------
# The exchange and the head-chunk compositions over P virtual ranks   [XCHG]
# ---------------------------------------------------------------------------
def all_to_all(sent):
    """sent[r][r2] is the chunk rank r sends to rank r2; returns received with
    received[r2][r] = sent[r][r2] (chunk from rank r lands in slot r on rank r2)."""
    P = len(sent)
    return [[sent[r][r2] for r in range(P)] for r2 in range(P)]


def pack_output_sequence_chunk(x: np.ndarray, world_size: int) -> np.ndarray:
    """Sequence split of an output band for the output exchange:
    x [B, S_global, head_count, D] -> [world_size, B, S_global/world_size, head_count, D],
    chunk r = sequence rows [r*S_local, (r+1)*S_local) (the rows rank r owns)."""
    B, S_g, cnt, D = x.shape
    if world_size < 1 or S_g % world_size:
        raise ValueError("S_global must be divisible by world_size")
    S = S_g // world_size
    out = np.empty((world_size, B, S, cnt, D), dtype=x.dtype)
    for r in range(world_size):
        out[r] = x[:, r * S:(r + 1) * S]
    return out


def gather_output_head_chunk(x_ranks: Sequence[np.ndarray], local_heads: int, head_offset: int,
                             out_ranks: Sequence[np.ndarray]):
    """One output band on every virtual rank: x_ranks[r] [B, S_global, head_count, D]
    -> copies of out_ranks[r2] [B, S_local, P*local_heads, D] with the band merged.

    Written as the pages' three steps: sequence-split pack on every rank, the
    all-to-all, and merge of the received band on every rank."""
    P = len(x_ranks)
    staged = [pack_output_sequence_chunk(x, P) for x in x_ranks]
    received = all_to_all([[staged[r][r2] for r2 in range(P)] for r in range(P)])
    res = []
    for r2 in range(P):
        band = np.stack(received[r2], axis=0)            # [P(src), B, S, cnt, D]
        P_, B, S, cnt, D = band.shape
        rec = band.transpose(1, 2, 0, 3, 4).reshape(B, S, P * cnt, D)  # slot = src*cnt + j
        res.append(merge_output_head_chunk(rec, P, local_heads, head_offset, out_ranks[r2]))
    return res


def scatter_qkv_head_chunk(q_ranks, k_ranks, v_ranks, head_offset: int, head_count: int):
    """One input band on every virtual rank: q/k/v_ranks[r] [B, S_local, H, D]
    -> per rank r2 the exchanged payload [B, S_global, head_count, 3*D].

    The pages' steps: pack on every rank, then the all-to-all of the packed
    payload's destination slots (slots [r2*head_count, (r2+1)*head_count) go to
    rank r2, which stacks them in source-rank order along the sequence)."""
    P = len(q_ranks)
    packed = [pack_head_chunk(q_ranks[r], k_ranks[r], v_ranks[r], P, head_offset, head_count)
              for r in range(P)]
    sent = [[packed[r][:, :, r2 * head_count:(r2 + 1) * head_count, :] for r2 in range(P)]
            for r in range(P)]
    received = all_to_all(sent)
    return [np.concatenate(received[r2], axis=1) for r2 in range(P)]


# ---------------------------------------------------------------------------
# Comparison rule for the fused values
# ---------------------------------------------------------------------------
def bf16_ulp(ref: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |ref|: 2^(floor(log2|ref|) - 7); the smallest normal's spacing at 0."""
    a = np.abs(np.asarray(ref, dtype=np.float64))
    tiny = 2.0 ** -126
    e = np.floor(np.log2(np.maximum(a, tiny)))
    return np.exp2(e - 7.0)


def fused_tolerance(ref: np.ndarray, ulps: float = 2.0, floor: float = 2e-2) -> np.ndarray:
    """Allowed |gpu - ref| per element: max(ulps * ulp_bf16(ref), floor)."""
    return np.maximum(ulps * bf16_ulp(ref), floor)
