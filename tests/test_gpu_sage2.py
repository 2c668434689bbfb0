"""GPU parity of the Sage2 quantise-and-exchange with the CPU oracle ("Prepared
Low-Precision QKV Exchange").

Q and V codes and the Q and V scales do not depend on any summation order: both
sides take the same fp32 steps, so they must agree bit for bit.  The K codes and
scales depend on the K mean, which the oracle takes exactly (the exact sum over the
sequence, divided by U, rounded once) and the kernel sums in fp32 in an order of its
own.  Any fp32 summation order of S terms is within gamma_S * sum|k| of the exact sum
(gamma_S = S u / (1 - S u), u = 2^-24), so the two means differ by at most
delta = gamma_S * sum|k| / U + 2 u |mean| (both roundings of the quotient).  The K
scales must then agree within delta / 127 + 4 u scale, a K code may differ by at most
one and only where the oracle's unrounded value (K - mean) * 127 / amax lies within
2 delta 127 / amax + 4 u |value| of a rounding tie, and such codes must be rare."""
import numpy as np
import pytest

import oracle
from ulysses_qkv_proj_gb300 import workloads as WL

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from ulysses_qkv_proj_gb300 import binding as qb  # noqa: E402

TD = {"bf16": torch.bfloat16, "fp16": torch.float16}
KEYS = ("q", "k", "v", "q_scale", "k_scale", "v_scale")


def _bits(a, dtype):
    a = np.asarray(a, np.float32)
    if dtype == "bf16":
        return WL.f32_to_bf16_bits(a)
    return a.astype(np.float16).view(np.uint16)


def _case(P, B, L, H, D, U, dtype, seed):
    """[P, B, L, 3, H, D] bits: q, k, v of source rank r are buf[r][:, :, c]."""
    rng = np.random.default_rng(seed)
    live = (np.arange(P * L) < U).reshape(P, 1, L, 1, 1, 1)

    def gen(scale, shift=0.0):
        a = (rng.standard_normal((P, B, L, 3, H, D)) * scale + shift).astype(np.float32)
        return _bits(np.where(live, a, 0), dtype)   # rows past the used prefix are zero
    buf = gen(1.5, 0.0)
    buf[:, :, :, 1] = gen(1.0, 2.0)[:, :, :, 1]   # K with a per-channel offset (smoothing matters)
    return buf


def _run(buf, P, U, dtype):
    Pb, B, L, _, H, D = buf.shape
    t = torch.from_numpy(np.ascontiguousarray(buf).view(np.int16)).view(TD[dtype]).cuda().reshape(P * B, L, 3, H, D)
    out = qb.sage2_outputs(P, B, L, H, D, U)
    for key in KEYS:
        out[key].view(torch.uint8).fill_(0x55)   # stale contents must be overwritten
    qb.ulysses_sage2_scatter_qkv(t[:, :, 0], t[:, :, 1], t[:, :, 2], P, U, out)
    torch.cuda.synchronize()
    return out


U_F32 = 2.0 ** -24
EXACT_KEYS = ("q", "v", "q_scale", "v_scale")
MAX_K_CODE_FLIPS = 1e-3   # share of K codes allowed to differ by one (near rounding ties)


def _oracle(buf, U, dtype):
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


def _assert_matches_oracle(out, ref, P, heads=None):
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


def _assert_equal(out, ref, P, heads=None):
    return _assert_matches_oracle(out, ref, P, heads)


@pytest.mark.parametrize("P,B,L,H,D,U,dtype", [
    (2, 1, 96, 4, 128, 192, "bf16"),
    (2, 2, 70, 4, 128, 101, "bf16"),     # ragged: groups and chunks straddle ranks, U inside a group
    (4, 1, 300, 8, 64, 1100, "fp16"),    # D = 64, several 256-row chunks per rank
    (2, 1, 150, 4, 128, 277, "fp16"),    # fp16 at D = 128
    (2, 2, 51, 6, 64, 77, "bf16"),       # bf16 at D = 64, a rank boundary inside a thread's rows
    (1, 1, 40, 2, 128, 40, "bf16"),      # one rank
    (3, 1, 21, 3, 128, 1, "bf16"),       # a single used row
])
def test_sage2_matches_oracle(P, B, L, H, D, U, dtype):
    buf = _case(P, B, L, H, D, U, dtype, seed=P * 1000 + L)
    _assert_equal(_run(buf, P, U, dtype), _oracle(buf, U, dtype), P)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_sage2_degenerate_groups(dtype):
    """All-zero Q head (scale 0, codes 0), V channels of zeros and of negative zeros,
    K constant over the sequence for one head (K - mean is tiny or zero)."""
    P, B, L, H, D, U = 2, 1, 80, 4, 128, 150
    buf = _case(P, B, L, H, D, U, dtype, seed=11)
    buf[:, :, :, 0, 1] = 0                                   # Q head 1: zeros
    buf[:, :, :, 2, 2, :5] = 0                               # V head 2 channels 0..4: +0
    buf[:, :, :, 2, 3, 7] = 0x8000                           # V head 3 channel 7: -0
    buf[:, :, :, 1, 0] = _bits(np.linspace(-2, 3, D), dtype)  # K head 0: one row repeated
    live = (np.arange(P * L) < U).reshape(P, 1, L, 1)
    buf[:, :, :, 1, 0] = np.where(live, buf[:, :, :, 1, 0], 0)
    out = _run(buf, P, U, dtype)
    ref = _oracle(buf, U, dtype)
    _assert_equal(out, ref, P)
    assert not out["q_scale"][0, :, 1].any()                 # rank 0 holds head 1
    assert (out["v"][1, :, 7, 1, :U] == 0x80).all()          # rank 1 holds head 3: -0 keeps its sign


def test_sage2_independent_views():
    """q, k, v from different buffers with different strides give the same codes."""
    P, B, L, H, D, U = 2, 1, 80, 4, 128, 160
    buf = _case(P, B, L, H, D, U, "bf16", seed=7)
    base = torch.from_numpy(buf.view(np.int16)).view(torch.bfloat16).cuda().reshape(P * B, L, 3, H, D)
    q = base[:, :, 0].contiguous()                                   # dense [P*B, L, H, D]
    kbig = torch.zeros((P * B, L, H + 2, D), dtype=torch.bfloat16, device="cuda")
    kbig[:, :, 1:H + 1] = base[:, :, 1]
    k = kbig[:, :, 1:H + 1]                                          # batch / row strides differ
    v = base[:, :, 2]                                                # strided view of the fused buffer
    out = qb.sage2_outputs(P, B, L, H, D, U)
    qb.ulysses_sage2_scatter_qkv(q, k, v, P, U, out)
    torch.cuda.synchronize()
    _assert_equal(out, _oracle(buf, U, "bf16"), P)


def test_sage2_repeat_calls_identical():
    """Two calls on the same inputs (the workspace reused) give the same bits."""
    P, B, L, H, D, U = 2, 1, 300, 4, 128, 600
    buf = _case(P, B, L, H, D, U, "bf16", seed=9)
    a = _run(buf, P, U, "bf16")
    b = _run(buf, P, U, "bf16")
    for key in KEYS:
        assert torch.equal(a[key].view(torch.uint8), b[key].view(torch.uint8)), key


def test_sage2_rejects():
    P, B, L, H, D = 2, 1, 32, 4, 128
    x = torch.zeros((P * B, L, H, D), dtype=torch.bfloat16, device="cuda")
    out = qb.sage2_outputs(P, B, L, H, D, P * L)
    with pytest.raises(qb.QnreError) as e:
        qb.ulysses_sage2_scatter_qkv(x, x, x, P, P * L + 1, out)
    assert e.value.status == 1
    with pytest.raises(qb.QnreError) as e:
        qb.ulysses_sage2_scatter_qkv(x.float(), x.float(), x.float(), P, P * L, out)
    assert e.value.status == 2
    small = dict(out)
    small["workspace"] = out["workspace"][:-16]
    with pytest.raises(qb.QnreError) as e:
        qb.ulysses_sage2_scatter_qkv(x, x, x, P, P * L, small)
    assert e.value.status == 5
    x64 = torch.zeros((P * B, L, H, 96), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(qb.QnreError) as e:
        qb.ulysses_sage2_scatter_qkv(x64, x64, x64, P, P * L, out)
    assert e.value.status == 2


@pytest.mark.slow
def test_sage2_pages_shape_full_size():
    """[1, 37760, 56, 128] over 2 virtual ranks, as the bench times it.  Each output
    depends only on its own (batch, head), so the oracle runs on two heads of each
    rank's band and those heads are compared bit for bit."""
    wl = WL.HEADCHUNK_WORKLOADS["headchunk_p2_s37760_h56"]
    P, L, H, D, H_l = wl.P, wl.S, wl.num_heads, wl.D, wl.H_local
    U = P * L - 123                                                # a ragged used prefix
    buf = WL.make_headchunk_buffer(1, wl.S_global, H, D).reshape(P, 1, L, 3, H, D)
    live = (np.arange(P * L) < U).reshape(P, 1, L, 1, 1, 1)
    buf = np.where(live, buf, np.uint16(0))
    out = _run(buf, P, U, "bf16")
    pick = [0, H_l - 1]                                            # first and last head of each band
    heads = [r * H_l + j for r in range(P) for j in pick]
    ref = _oracle(np.ascontiguousarray(buf[..., heads, :]), U, "bf16")
    _assert_equal(out, ref, P, heads=pick)
