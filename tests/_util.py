"""Shared test helpers: numpy <-> torch bf16 moves and the fused comparison."""
import numpy as np

import oracle


def to_dev_bf16(a, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)


def to_host_bits(t):
    """Device bf16/fp16 tensor -> numpy uint16 bit patterns (any strides)."""
    import torch
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def to_host_f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_fused_close(got, ref, what=""):
    """|got - ref| <= max(2 bf16 ulp(ref), 2e-2) elementwise; NaN must match NaN."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    nan_ref = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan_ref), f"{what}: NaN pattern differs"
    g, r = got[~nan_ref], ref[~nan_ref]
    err = np.abs(g - r)
    tol = oracle.fused_tolerance(r)
    bad = err > tol
    if bad.any():
        i = np.argmax(err - tol)
        raise AssertionError(f"{what}: {bad.sum()} / {bad.size} elements out of tolerance; "
                             f"worst got={g[i]!r} ref={r[i]!r} err={err[i]:.3g} tol={tol[i]:.3g}")
    return float(err.max()) if err.size else 0.0


def dest_index(tokens, P, B, S, H):
    """Destination (rank, batch, row, local head) arrays [n, H] for token ids, by the oracle's map."""
    n = len(tokens)
    idx = np.zeros((4, n, H), dtype=np.int64)
    for i, t in enumerate(tokens):
        r_s, b, s = oracle.token_coords(int(t), P, B, S)
        for h in range(H):
            idx[:, i, h] = oracle.band_destination(r_s, b, s, h, P, B, S, H)
    return idx


def sample_tokens(T, S, n=512, seed=0):
    """Stratified token sample of a [P, B, S]-ordered problem of T tokens: always the
    first and last token of every (rank, batch) segment of S tokens and of every
    256-row pair tile and 128-row CTA half, then random tokens until there are at
    least n.  The mandatory picks are never dropped, so the sample may exceed n."""
    rng = np.random.default_rng(seed)
    picks = set()
    for t0 in range(0, T, S):
        picks.update({t0, min(T - 1, t0 + S - 1)})
    for t0 in range(0, T, 128):
        picks.update({t0, min(T - 1, t0 + 127)})
    rest = n - len(picks)
    if rest > 0:
        pool = np.setdiff1d(np.arange(T), np.fromiter(picks, dtype=np.int64))
        picks.update(rng.choice(pool, size=min(rest, len(pool)), replace=False).tolist())
    return np.array(sorted(picks))
