"""Seeded random shapes for every layout entry point, bit-exact against the oracle.

Each case draws a world size, local head count, head dim, batch, ragged sequence
length, element type and an uneven schedule that may leave heads out, and takes
q/k/v as strided views of a padded [B, S, 3, H + pad, D] buffer.  The single-chunk
and schedule forms of pack and merge, scatter/gather heads, the sequence pack and
both composed exchanges are compared with the oracle bit for bit; every merge
starts from a filled output so untouched elements are checked too."""
import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from ulysses_qkv_proj_gb300 import binding as qb  # noqa: E402

N_CASES = 64


def _case(seed):
    rng = np.random.default_rng(1000 + seed)
    W = int(rng.choice([1, 2, 3, 4, 8]))
    L = int(rng.integers(1, 9))
    D = int(rng.choice([64, 128]))
    B = int(rng.integers(1, 4))
    S = int(rng.integers(1, 260))
    wide = bool(rng.integers(0, 2))             # 4-byte elements
    pad = int(rng.integers(0, 3))               # extra heads in the buffer: head stride > D
    # an uneven schedule over [0, L): contiguous chunks, some dropped (at most 8)
    cuts = sorted(set(rng.integers(1, L, size=int(rng.integers(0, L))).tolist())) if L > 1 else []
    edges = [0] + cuts + [L]
    chunks = [(a, b - a) for a, b in zip(edges[:-1], edges[1:])][:8]
    keep = [c for c in chunks if rng.random() < 0.8] or chunks[:1]
    S = max(1, min(S, 8_000_000 // (W * B * W * L * D)))   # at most ~8 M elements per rank set
    return rng, W, L, D, B, S, wide, pad, keep


def _bits(rng, shape, wide):
    if wide:
        return rng.integers(0, 1 << 32, size=shape, dtype=np.uint64).astype(np.uint32)
    return rng.integers(0, 1 << 16, size=shape).astype(np.uint16)


def _dev(a):
    if a.dtype == np.uint32:
        return torch.from_numpy(a.view(np.int32)).view(torch.float32).cuda()
    return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()


def _host(t):
    t = t.contiguous().cpu()
    if t.element_size() == 4:
        return t.view(torch.int32).numpy().view(np.uint32)
    return t.view(torch.int16).numpy().view(np.uint16)


def _empty(shape, wide):
    return torch.empty(shape, dtype=torch.float32 if wide else torch.bfloat16, device="cuda")


@pytest.mark.parametrize("seed", range(N_CASES))
def test_head_chunk_pack_merge(seed):
    rng, W, L, D, B, S, wide, pad, sched = _case(seed)
    H = W * L
    buf = _bits(rng, (B, S, 3, H + pad, D), wide)
    tb = _dev(buf)
    q, k, v = (tb[:, :, c, :H] for c in range(3))
    hq, hk, hv = (buf[:, :, c, :H] for c in range(3))
    want = [oracle.pack_head_chunk(hq, hk, hv, W, off, cnt) for off, cnt in sched]
    # one launch per chunk
    outs = [_empty((B, S, W * cnt, 3 * D), wide) for _, cnt in sched]
    for (off, cnt), o in zip(sched, outs):
        qb.ulysses_pack_head_chunk(q, k, v, W, off, cnt, o)
    # one launch for the schedule
    outs_s = [_empty((B, S, W * cnt, 3 * D), wide) for _, cnt in sched]
    qb.ulysses_pack_head_chunk_schedule(q, k, v, W, sched, outs_s)
    torch.cuda.synchronize()
    for i in range(len(sched)):
        assert np.array_equal(_host(outs[i]), want[i]), f"pack chunk {i}"
        assert np.array_equal(_host(outs_s[i]), want[i]), f"pack schedule chunk {i}"
    # merge each chunk's v slice (a strided received view) into a filled output
    fill = _bits(rng, (B, S, H, D), wide)
    m1, m2 = _dev(fill), _dev(fill)
    ref = fill
    for (off, cnt), o, w in zip(sched, outs, want):
        qb.ulysses_merge_output_head_chunk(o[..., 2 * D:], W, L, off, m1)
        ref = oracle.merge_output_head_chunk(w[..., 2 * D:], W, L, off, ref)
    qb.ulysses_merge_output_head_chunk_schedule([o[..., 2 * D:] for o in outs], W, L, [off for off, _ in sched], m2)
    # the same merges from contiguous received bands (heads back to back)
    m3, m4 = _dev(fill), _dev(fill)
    recv = [o[..., 2 * D:].contiguous() for o in outs]
    for (off, _), r in zip(sched, recv):
        qb.ulysses_merge_output_head_chunk(r, W, L, off, m3)
    qb.ulysses_merge_output_head_chunk_schedule(recv, W, L, [off for off, _ in sched], m4)
    torch.cuda.synchronize()
    for m in (m1, m2, m3, m4):
        assert np.array_equal(_host(m), ref)


@pytest.mark.parametrize("seed", range(N_CASES))
def test_ordinary_and_composed_exchanges(seed):
    rng, P, L, D, B, S, wide, _, sched = _case(seed)
    H = P * L
    x = _bits(rng, (P, B, S, H, D), wide)
    tx = _dev(x)
    y = _empty((P, B, P * S, L, D), wide)
    qb.ulysses_scatter_heads(tx, y)
    g = _empty((P, B, S, H, D), wide)
    qb.ulysses_gather_heads(y, g)
    torch.cuda.synchronize()
    want_y = oracle.scatter_heads(x)
    assert np.array_equal(_host(y), want_y)
    assert np.array_equal(_host(g), oracle.gather_heads(want_y))
    assert np.array_equal(_host(g), x)
    # composed exchanges of each chunk: q/k/v of every rank as views [P*B, S, H, D]
    buf = _bits(rng, (P * B, S, 3, H, D), wide)
    tb = _dev(buf)
    ranks = buf.reshape(P, B, S, 3, H, D)
    fill = _bits(rng, (P, B, S, H, D), wide)
    got_out = _dev(fill)
    ref_out = [fill[r] for r in range(P)]
    for off, cnt in sched:
        pay = _empty((P, B, P * S, cnt, 3 * D), wide)
        qb.ulysses_scatter_qkv_head_chunk(tb[:, :, 0], tb[:, :, 1], tb[:, :, 2], P, off, cnt, pay)
        want = oracle.scatter_qkv_head_chunk([ranks[r, :, :, 0] for r in range(P)],
                                             [ranks[r, :, :, 1] for r in range(P)],
                                             [ranks[r, :, :, 2] for r in range(P)], off, cnt)
        torch.cuda.synchronize()
        assert np.array_equal(_host(pay), np.stack(want, axis=0)), f"scatter_qkv chunk {off}"
        band = pay[..., :D].contiguous()                       # the q band of every rank
        qb.ulysses_gather_output_head_chunk(band, L, off, got_out)
        ref_out = oracle.gather_output_head_chunk([np.stack(want, 0)[r][..., :D] for r in range(P)], L, off, ref_out)
        seqp = _empty((P, B, S, cnt, D), wide)
        qb.ulysses_pack_output_sequence_chunk(band[0], P, seqp)
        torch.cuda.synchronize()
        assert np.array_equal(_host(seqp), oracle.pack_output_sequence_chunk(_host(band[0]), P))
    assert np.array_equal(_host(got_out), np.stack(ref_out, axis=0))
