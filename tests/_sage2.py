"""Comparison of the GPU Sage2 encoding with the CPU oracle, shared by the GPU tests.

Q and V codes and the Q and V scales do not depend on any summation order: both
sides take the same fp32 steps, so they must agree bit for bit.  The K codes and
scales depend on the K mean, which the oracle takes exactly (the exact sum over the
sequence, divided by U, rounded once) and the kernel sums in fp32 in an order of its
own.  Any fp32 summation order of S terms is within gamma_S * sum|k| of the exact sum
(gamma_S = S u / (1 - S u), u = 2^-24), so the two means differ by at most
delta = gamma_S * sum|k| / U + 2 u |mean| (both roundings of the quotient).  The K
scales must then agree within delta / 127 + 4 u scale, a K code may differ by at most
one and only where the oracle's unrounded value (K - mean) * 127 / amax lies within
2 delta 127 / amax + 4 u |value| of a rounding tie, and such codes must be rare.
"""
import numpy as np

import oracle

U_F32 = 2.0 ** -24
EXACT_KEYS = ("q", "v", "q_scale", "v_scale")
MAX_K_CODE_FLIPS = 1e-3   # share of K codes allowed to differ by one (near rounding ties)


def sage2_oracle(buf, U, dtype):
    """Oracle outputs for every rank, with the unrounded K values and each rank's
    per-channel bound `delta` [B, H_l, D] on the difference of the two K means."""
    P = buf.shape[0]
    ref = oracle.sage2_scatter_qkv([buf[r][:, :, 0] for r in range(P)], [buf[r][:, :, 1] for r in range(P)],
                                   [buf[r][:, :, 2] for r in range(P)], U, dtype, with_k_scaled=True)
    B, L, H = buf.shape[1], buf.shape[2], buf.shape[4]
    S, H_l = P * L, H // P
    k = np.stack([oracle.decode16(buf[r][:, :, 1], dtype).astype(np.float64) for r in range(P)])  # [P,B,L,H,D]
    abs_sum = np.abs(k).sum(axis=(0, 2))                                                        # [B, H, D]
    mean = np.abs(k.sum(axis=(0, 2))) / U
    gamma = S * U_F32 / (1 - S * U_F32)
    delta = 1.01 * gamma * abs_sum / U + 2.01 * U_F32 * mean
    for r in range(P):
        ref[r]["delta"] = delta[:, r * H_l:(r + 1) * H_l]
    return ref


def _take(a, key, heads):
    if heads is None:
        return a
    return np.take(a, heads, axis=1 if key.endswith("scale") or key == "delta" else 2)


def assert_sage2_matches(out, ref, P, heads=None):
    """Q/V codes and scales bit for bit; K scales and codes within the bounds of the
    module docstring; optionally over local heads `heads` of each rank only."""
    flips, total = 0, 0
    for r in range(P):
        for key in EXACT_KEYS:
            got = _take(out[key][r].cpu().numpy(), key, heads)
            want = ref[r][key]
            view = np.uint32 if got.dtype == np.float32 else np.uint8
            assert got.shape == want.shape, (r, key)
            assert np.array_equal(got.view(view), want.view(view)), \
                f"rank {r} {key}: {(got.view(view) != want.view(view)).sum()} of {got.size} differ"
        delta = ref[r]["delta"]                                                  # [B, H_l', D]
        ks_got = _take(out["k_scale"][r].cpu().numpy(), "k_scale", heads).astype(np.float64)
        ks_want = ref[r]["k_scale"].astype(np.float64)                           # [B, H_l', groups]
        d_head = delta.max(axis=2)[:, :, None]                                   # amax runs over all channels
        assert ks_got.shape == ks_want.shape
        bad = np.abs(ks_got - ks_want) > d_head / 127 + 4 * U_F32 * ks_want + 1e-38
        assert not bad.any(), f"rank {r} k_scale: {bad.sum()} of {bad.size} beyond the mean's bound"
        k_got = _take(out["k"][r].cpu().numpy(), "k", heads).astype(np.int64)    # [B, S, H_l', D]
        k_want = ref[r]["k"].astype(np.int64)
        diff = np.abs(k_got - k_want)
        assert diff.max(initial=0) <= 1, f"rank {r} k: a code differs by {diff.max()}"
        if diff.any():
            p = ref[r]["k_scaled"].astype(np.float64)
            inv = np.where(ks_want > 0, 1.0 / np.maximum(ks_want, 1e-38), 0.0)  # 127 / amax per group
            S = p.shape[1]
            inv_rows = np.zeros(inv.shape[:2] + (S,))
            g_rows = np.repeat(inv, oracle.K_GROUP, axis=2)[:, :, :S]             # row s is in group s // 64
            inv_rows[:, :, :g_rows.shape[2]] = g_rows
            inv_rows = inv_rows.transpose(0, 2, 1)[..., None]                     # [B, S, H_l', 1]
            tau = 2.02 * delta[:, None] * inv_rows + 4 * U_F32 * np.abs(p) + 1e-6
            tie_dist = np.abs(np.abs(p - np.floor(p)) - 0.5)
            far = (diff > 0) & (tie_dist > tau)
            assert not far.any(), f"rank {r} k: {far.sum()} codes differ away from a rounding tie"
        flips += int((diff > 0).sum())
        total += diff.size
    assert flips <= max(4, MAX_K_CODE_FLIPS * total), f"{flips} of {total} K codes differ by one"
    return flips
