"""GPU parity of the Sage2 quantise-and-exchange with the CPU oracle ("Prepared
Low-Precision QKV Exchange"): Q/V codes and scales bit for bit, K codes and scales
within the bound of the kernel's fp32 K mean against the oracle's exact one
(tests/_sage2.py states it)."""
import numpy as np
import pytest

from ulysses_qkv_proj_gb300 import workloads as WL
from _sage2 import assert_sage2_matches, sage2_oracle

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


def _oracle(buf, U, dtype):
    return sage2_oracle(buf, U, dtype)


def _assert_equal(out, ref, P, heads=None):
    return assert_sage2_matches(out, ref, P, heads)


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
    # every head, by properties that hold at any size: each group's (Q: 32 rows, K: 64
    # rows below U) largest code is 127 and each V channel reaches 448 (code 0x7E),
    # every scale is positive, and codes past U are zero
    for r in range(P):
        q, k = out["q"][r].int(), out["k"][r].int()                  # [1, S, H_l, D]
        assert not q[:, U:].any() and not k[:, U:].any()
        for codes, grp in ((q, 32), (k, 64)):
            full = (U // grp) * grp
            top = codes[:, :full].abs().reshape(1, U // grp, grp, H_l, D).amax(dim=(2, 4))
            assert bool((top == 127).all()), "a group's largest code is not 127"
        vcodes = out["v"][r][..., :U].int()                           # [1, D, H_l, U]
        assert bool(((vcodes & 0x7F).amax(dim=-1) == 0x7E).all()), "a V channel does not reach 448"
        assert not out["v"][r][..., U:].int().any()
        for key in ("q_scale", "k_scale", "v_scale"):
            assert bool((out[key][r] > 0).all()), key
    pick = [0, H_l - 1]                                            # first and last head of each band
    heads = [r * H_l + j for r in range(P) for j in pick]
    ref = _oracle(np.ascontiguousarray(buf[..., heads, :]), U, "bf16")
    _assert_equal(out, ref, P, heads=pick)


@pytest.mark.parametrize("seed", range(16))
def test_sage2_random_shapes(seed):
    """Seeded random (P, B, L, H, D, used prefix, dtype) against the oracle."""
    rng = np.random.default_rng(700 + seed)
    P = int(rng.choice([1, 2, 3, 4, 8]))
    B = int(rng.integers(1, 3))
    L = int(rng.integers(1, 400))
    H = P * int(rng.integers(1, 4))
    D = int(rng.choice([64, 128]))
    U = int(rng.integers(1, P * L + 1))
    dtype = str(rng.choice(["bf16", "fp16"]))
    buf = _case(P, B, L, H, D, U, dtype, seed=seed)
    _assert_equal(_run(buf, P, U, dtype), _oracle(buf, U, dtype), P)
